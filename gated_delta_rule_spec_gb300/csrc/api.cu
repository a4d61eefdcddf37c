// api.cu -- the extern "C" entry points of libgdnspec (declared and documented
// in include/gdn_spec.h): host-side validation, kernel selection and
// stream-ordered launches.  Nothing here allocates, frees or synchronises,
// except gdn_spec_read_status.
#include <atomic>
#include <cstdint>
#include <cstring>

#include "common.cuh"

namespace gdnspec {

namespace {
std::atomic<uint32_t> g_data_wait_limit{kWaitLimitDefault};
}  // namespace

uint32_t data_wait_limit() { return g_data_wait_limit.load(std::memory_order_relaxed); }

cudaError_t launch_verify_generic(const LayerArgs &P, const CursorArgs &C, bool kda, bool bf16,
                                  const int32_t *slot_idx, int B, const void *q, const void *k,
                                  const void *v, const void *a, const void *b,
                                  const float *A_log, const float *dt_bias, void *out,
                                  cudaStream_t stream);
size_t verify_generic_smem_bytes(int K, int L, int T, bool kda);
bool verify_tc_supported(const LayerArgs &P, bool kda, bool bf16);
bool verify_kda_tc_supported(const LayerArgs &P, bool kda, bool bf16);
cudaError_t launch_verify_kda_tc(const LayerArgs &P, const CursorArgs &C, const int32_t *slot_idx, int B,
                                 const void *q, const void *k, const void *v, const void *a, const void *b,
                                 const float *A_log, const float *dt_bias, void *out, cudaStream_t stream);
cudaError_t launch_verify_tc(const LayerArgs &P, const CursorArgs &C, const int32_t *slot_idx,
                             int B, const void *q, const void *k, const void *v, const void *a,
                             const void *b, const float *A_log, const float *dt_bias, void *out,
                             cudaStream_t stream);
cudaError_t launch_fold(const LayerArgs &P, const FoldLayers &FL, int n_layers, bool kda,
                        bool bf16, const CursorArgs &C, const int32_t *slot_idx, int B,
                        cudaStream_t stream);
size_t fold_smem_bytes(int K, int L, bool kda, bool bf16);
cudaError_t launch_commit(const CursorArgs &C, int T, int L, const int32_t *slot_idx, int B,
                          const int32_t *accept_len, cudaStream_t stream);
cudaError_t launch_fold_cursors(const CursorArgs &C, int L, const int32_t *slot_idx, int B,
                                cudaStream_t stream);
cudaError_t launch_reset(const CursorArgs &C, const int32_t *slot_idx, int B, cudaStream_t stream);
cudaError_t launch_prefill(const LayerArgs &P, const CursorArgs &C, bool kda, bool bf16,
                           const int32_t *slot_idx, int B, int N, const void *q, const void *k,
                           const void *v, const void *a, const void *b, const float *A_log,
                           const float *dt_bias, void *out, int from_zero, cudaStream_t stream);
size_t prefill_smem_bytes(int K, bool kda, bool bf16);
bool prefill_tc_supported(const LayerArgs &P, bool kda, bool bf16);
bool verify_d_supported(const LayerArgs &P, bool kda, bool bf16);
cudaError_t launch_verify_d(const LayerArgs &P, const CursorArgs &C, float *dring,
                            const int32_t *slot_idx, int B, const void *q, const void *k,
                            const void *v, const void *a, const void *b, const float *A_log,
                            const float *dt_bias, void *out, cudaStream_t stream);
cudaError_t launch_snapshot_verify(const LayerArgs &P, const CursorArgs &C, bool kda, bool bf16,
                                   const int32_t *slot_idx, int B, const void *q, const void *k,
                                   const void *v, const void *a, const void *b, const float *A_log,
                                   const float *dt_bias, void *out, float *snap, cudaStream_t stream);
cudaError_t launch_snapshot_commit(const LayerArgs &P, const CursorArgs &C, const int32_t *slot_idx,
                                   int B, const int32_t *accept_len, const float *snap,
                                   cudaStream_t stream);
}  // namespace gdnspec

using namespace gdnspec;

namespace {

constexpr size_t kMaxSmem = 227 * 1024;

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

int check_cursors(const gdn_spec_cursors *c) {
    if (!c || !c->write_pos || !c->cache_base || !c->is_flush || !c->status) return GDN_SPEC_EINVAL;
    if (c->num_slots <= 0) return GDN_SPEC_EINVAL;
    return GDN_SPEC_OK;
}

int check_layer(const gdn_spec_layer *L) {
    if (!L) return GDN_SPEC_EINVAL;
    if (L->gate_kind != GDN_SPEC_GATE_SCALAR && L->gate_kind != GDN_SPEC_GATE_PER_KEY)
        return GDN_SPEC_EDTYPE;
    if (L->io_dtype != GDN_SPEC_DTYPE_BF16 && L->io_dtype != GDN_SPEC_DTYPE_FP32)
        return GDN_SPEC_EDTYPE;
    if (L->H <= 0 || L->HV <= 0 || L->K <= 0 || L->V <= 0 || L->T <= 0 || L->num_slots <= 0)
        return GDN_SPEC_EINVAL;
    if (L->HV % L->H != 0) return GDN_SPEC_EINVAL;
    if (!pow2(L->L) || L->L < 2 * L->T) return GDN_SPEC_EINVAL;
    if (L->K % 8 != 0 || L->V % 8 != 0) return GDN_SPEC_EALIGN;
    if (!L->checkpoint || !L->rawv || !L->rawk || !L->ring_g || !L->ring_beta) return GDN_SPEC_EINVAL;
    if (!aligned16(L->checkpoint) || !aligned16(L->rawv) || !aligned16(L->rawk) ||
        !aligned16(L->ring_g) || !aligned16(L->ring_beta))
        return GDN_SPEC_EALIGN;
    if ((L->K != 32 && L->K != 64 && L->K != 128) || L->T > 16) return GDN_SPEC_EUNSUPPORTED;
    if (L->L > (L->gate_kind == GDN_SPEC_GATE_PER_KEY ? 64 : 128)) return GDN_SPEC_EUNSUPPORTED;
    return GDN_SPEC_OK;
}

LayerArgs layer_args(const gdn_spec_layer *L) {
    LayerArgs P;
    P.H = L->H;
    P.HV = L->HV;
    P.G = L->HV / L->H;
    P.K = L->K;
    P.V = L->V;
    P.T = L->T;
    P.L = L->L;
    P.num_slots = L->num_slots;
    P.scale = L->scale;
    P.l2_eps = L->l2_eps;
    P.checkpoint = L->checkpoint;
    P.rawv = L->rawv;
    P.rawk = L->rawk;
    P.ring_g = L->ring_g;
    P.ring_beta = L->ring_beta;
    return P;
}

CursorArgs cursor_args(const gdn_spec_cursors *c) {
    CursorArgs C;
    C.num_slots = c->num_slots;
    C.write_pos = c->write_pos;
    C.cache_base = c->cache_base;
    C.is_flush = c->is_flush;
    C.status = c->status;
    return C;
}

int cuda_rc(cudaError_t e) { return e == cudaSuccess ? GDN_SPEC_OK : GDN_SPEC_ECUDA; }

}  // namespace

extern "C" {

int gdn_spec_abi_version(void) { return GDN_SPEC_ABI_VERSION; }

const char *gdn_spec_strerror(int code) {
    switch (code) {
        case GDN_SPEC_OK: return "ok";
        case GDN_SPEC_EINVAL: return "invalid argument (null pointer, size, L, T or head counts)";
        case GDN_SPEC_EDTYPE: return "unknown io_dtype or gate_kind";
        case GDN_SPEC_EALIGN: return "pointer not 16-byte aligned or K/V not a multiple of 8";
        case GDN_SPEC_ECUDA: return "CUDA launch or call failed";
        case GDN_SPEC_EUNSUPPORTED: return "shape not supported by the kernels";
        default: return "unknown error code";
    }
}

const char *gdn_spec_verify_path(const gdn_spec_layer *layer) {
    if (check_layer(layer) != GDN_SPEC_OK) return nullptr;
    const LayerArgs P = layer_args(layer);
    const bool kda = layer->gate_kind == GDN_SPEC_GATE_PER_KEY;
    const bool bf16 = layer->io_dtype == GDN_SPEC_DTYPE_BF16;
    if (verify_tc_supported(P, kda, bf16)) return "tc";
    return verify_kda_tc_supported(P, kda, bf16) ? "tc_kda" : "generic";
}

const char *gdn_spec_prefill_path(const gdn_spec_layer *layer) {
    if (check_layer(layer) != GDN_SPEC_OK) return nullptr;
    const LayerArgs P = layer_args(layer);
    const bool kda = layer->gate_kind == GDN_SPEC_GATE_PER_KEY;
    const bool bf16 = layer->io_dtype == GDN_SPEC_DTYPE_BF16;
    return prefill_tc_supported(P, kda, bf16) ? "chunk" : "sequential";
}

int gdn_spec_verify(const gdn_spec_layer *layer, const gdn_spec_cursors *cursors,
                    const int32_t *slot_idx, int32_t B, const void *q, const void *k,
                    const void *v, const void *a, const void *b, const float *A_log,
                    const float *dt_bias, void *out, void *stream) {
    int rc = check_layer(layer);
    if (rc) return rc;
    if ((rc = check_cursors(cursors))) return rc;
    if (cursors->num_slots != layer->num_slots) return GDN_SPEC_EINVAL;
    if (B < 0) return GDN_SPEC_EINVAL;
    if (B == 0) return GDN_SPEC_OK;
    if (!slot_idx || !q || !k || !v || !a || !b || !A_log || !dt_bias || !out) return GDN_SPEC_EINVAL;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return GDN_SPEC_EALIGN;
    const LayerArgs P = layer_args(layer);
    const CursorArgs C = cursor_args(cursors);
    const bool kda = layer->gate_kind == GDN_SPEC_GATE_PER_KEY;
    const bool bf16 = layer->io_dtype == GDN_SPEC_DTYPE_BF16;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (verify_tc_supported(P, kda, bf16))
        return cuda_rc(launch_verify_tc(P, C, slot_idx, B, q, k, v, a, b, A_log, dt_bias, out, st));
    if (verify_kda_tc_supported(P, kda, bf16))
        return cuda_rc(launch_verify_kda_tc(P, C, slot_idx, B, q, k, v, a, b, A_log, dt_bias, out, st));
    if (verify_generic_smem_bytes(P.K, P.L, P.T, kda) > kMaxSmem) return GDN_SPEC_EUNSUPPORTED;
    return cuda_rc(launch_verify_generic(P, C, kda, bf16, slot_idx, B, q, k, v, a, b, A_log,
                                         dt_bias, out, st));
}

int gdn_spec_verify_d(const gdn_spec_layer *layer, float *dring, const gdn_spec_cursors *cursors,
                      const int32_t *slot_idx, int32_t B, const void *q, const void *k,
                      const void *v, const void *a, const void *b, const float *A_log,
                      const float *dt_bias, void *out, void *stream) {
    int rc = check_layer(layer);
    if (rc) return rc;
    if ((rc = check_cursors(cursors))) return rc;
    if (cursors->num_slots != layer->num_slots) return GDN_SPEC_EINVAL;
    if (B < 0) return GDN_SPEC_EINVAL;
    if (B == 0) return GDN_SPEC_OK;
    if (!dring || !slot_idx || !q || !k || !v || !a || !b || !A_log || !dt_bias || !out)
        return GDN_SPEC_EINVAL;
    if (!aligned16(dring) || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
        return GDN_SPEC_EALIGN;
    const LayerArgs P = layer_args(layer);
    const bool kda = layer->gate_kind == GDN_SPEC_GATE_PER_KEY;
    const bool bf16 = layer->io_dtype == GDN_SPEC_DTYPE_BF16;
    if (!verify_d_supported(P, kda, bf16)) return GDN_SPEC_EUNSUPPORTED;
    return cuda_rc(launch_verify_d(P, cursor_args(cursors), dring, slot_idx, B, q, k, v, a, b, A_log,
                                   dt_bias, out, static_cast<cudaStream_t>(stream)));
}

int gdn_spec_commit(const gdn_spec_cursors *cursors, int32_t T, int32_t L,
                    const int32_t *slot_idx, int32_t B, const int32_t *accept_len, void *stream) {
    int rc = check_cursors(cursors);
    if (rc) return rc;
    if (T <= 0 || !pow2(L) || L < 2 * T || B < 0) return GDN_SPEC_EINVAL;
    if (B == 0) return GDN_SPEC_OK;
    if (!slot_idx || !accept_len) return GDN_SPEC_EINVAL;
    return cuda_rc(launch_commit(cursor_args(cursors), T, L, slot_idx, B, accept_len,
                                 static_cast<cudaStream_t>(stream)));
}

int gdn_spec_fold(const gdn_spec_layer *layers, int32_t n_layers, const gdn_spec_cursors *cursors,
                  const int32_t *slot_idx, int32_t B, void *stream) {
    int rc = check_cursors(cursors);
    if (rc) return rc;
    if (!layers || n_layers <= 0 || B < 0) return GDN_SPEC_EINVAL;
    for (int i = 0; i < n_layers; ++i) {
        if ((rc = check_layer(&layers[i]))) return rc;
        const gdn_spec_layer &a = layers[0], &b = layers[i];
        if (a.H != b.H || a.HV != b.HV || a.K != b.K || a.V != b.V || a.T != b.T || a.L != b.L ||
            a.num_slots != b.num_slots || a.gate_kind != b.gate_kind || a.io_dtype != b.io_dtype ||
            a.l2_eps != b.l2_eps)
            return GDN_SPEC_EINVAL;
    }
    if (cursors->num_slots != layers[0].num_slots) return GDN_SPEC_EINVAL;
    if (B == 0) return GDN_SPEC_OK;
    if (!slot_idx) return GDN_SPEC_EINVAL;
    const bool kda = layers[0].gate_kind == GDN_SPEC_GATE_PER_KEY;
    const bool bf16 = layers[0].io_dtype == GDN_SPEC_DTYPE_BF16;
    if (fold_smem_bytes(layers[0].K, layers[0].L, kda, bf16) > kMaxSmem) return GDN_SPEC_EUNSUPPORTED;
    const LayerArgs P = layer_args(&layers[0]);
    const CursorArgs C = cursor_args(cursors);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    for (int first = 0; first < n_layers; first += kFoldMaxLayers) {
        const int cnt = n_layers - first < kFoldMaxLayers ? n_layers - first : kFoldMaxLayers;
        FoldLayers FL;
        std::memset(&FL, 0, sizeof FL);
        for (int i = 0; i < cnt; ++i) {
            FL.checkpoint[i] = layers[first + i].checkpoint;
            FL.rawv[i] = layers[first + i].rawv;
            FL.rawk[i] = layers[first + i].rawk;
            FL.ring_g[i] = layers[first + i].ring_g;
            FL.ring_beta[i] = layers[first + i].ring_beta;
        }
        if ((rc = cuda_rc(launch_fold(P, FL, cnt, kda, bf16, C, slot_idx, B, st)))) return rc;
    }
    return cuda_rc(launch_fold_cursors(C, P.L, slot_idx, B, st));
}

int gdn_spec_prefill(const gdn_spec_layer *layer, const gdn_spec_cursors *cursors,
                     const int32_t *slot_idx, int32_t B, int32_t N, const void *q, const void *k,
                     const void *v, const void *a, const void *b, const float *A_log,
                     const float *dt_bias, void *out, int32_t from_zero, void *stream) {
    int rc = check_layer(layer);
    if (rc) return rc;
    if ((rc = check_cursors(cursors))) return rc;
    if (cursors->num_slots != layer->num_slots) return GDN_SPEC_EINVAL;
    if (B < 0 || N < 0) return GDN_SPEC_EINVAL;
    if (B == 0) return GDN_SPEC_OK;
    if (!slot_idx) return GDN_SPEC_EINVAL;
    if (N > 0 && (!q || !k || !v || !a || !b || !A_log || !dt_bias || !out)) return GDN_SPEC_EINVAL;
    if (N > 0 && (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)))
        return GDN_SPEC_EALIGN;
    const bool kda = layer->gate_kind == GDN_SPEC_GATE_PER_KEY;
    const bool bf16 = layer->io_dtype == GDN_SPEC_DTYPE_BF16;
    if (prefill_smem_bytes(layer->K, kda, bf16) > kMaxSmem) return GDN_SPEC_EUNSUPPORTED;
    return cuda_rc(launch_prefill(layer_args(layer), cursor_args(cursors), kda, bf16, slot_idx, B, N,
                                  q, k, v, a, b, A_log, dt_bias, out, from_zero ? 1 : 0,
                                  static_cast<cudaStream_t>(stream)));
}

int gdn_spec_snapshot_verify(const gdn_spec_layer *layer, const gdn_spec_cursors *cursors,
                             const int32_t *slot_idx, int32_t B, const void *q, const void *k,
                             const void *v, const void *a, const void *b, const float *A_log,
                             const float *dt_bias, void *out, float *snap, void *stream) {
    int rc = check_layer(layer);
    if (rc) return rc;
    if ((rc = check_cursors(cursors))) return rc;
    if (cursors->num_slots != layer->num_slots) return GDN_SPEC_EINVAL;
    if (B < 0) return GDN_SPEC_EINVAL;
    if (B == 0) return GDN_SPEC_OK;
    if (!slot_idx || !q || !k || !v || !a || !b || !A_log || !dt_bias || !out || !snap)
        return GDN_SPEC_EINVAL;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(snap))
        return GDN_SPEC_EALIGN;
    const bool kda = layer->gate_kind == GDN_SPEC_GATE_PER_KEY;
    const bool bf16 = layer->io_dtype == GDN_SPEC_DTYPE_BF16;
    if (prefill_smem_bytes(layer->K, kda, bf16) > kMaxSmem) return GDN_SPEC_EUNSUPPORTED;
    return cuda_rc(launch_snapshot_verify(layer_args(layer), cursor_args(cursors), kda, bf16, slot_idx, B,
                                          q, k, v, a, b, A_log, dt_bias, out, snap,
                                          static_cast<cudaStream_t>(stream)));
}

int gdn_spec_snapshot_commit(const gdn_spec_layer *layer, const gdn_spec_cursors *cursors,
                             const int32_t *slot_idx, int32_t B, const int32_t *accept_len,
                             const float *snap, void *stream) {
    int rc = check_layer(layer);
    if (rc) return rc;
    if ((rc = check_cursors(cursors))) return rc;
    if (cursors->num_slots != layer->num_slots) return GDN_SPEC_EINVAL;
    if (B < 0) return GDN_SPEC_EINVAL;
    if (B == 0) return GDN_SPEC_OK;
    if (!slot_idx || !accept_len || !snap) return GDN_SPEC_EINVAL;
    if (!aligned16(snap)) return GDN_SPEC_EALIGN;
    return cuda_rc(launch_snapshot_commit(layer_args(layer), cursor_args(cursors), slot_idx, B,
                                          accept_len, snap, static_cast<cudaStream_t>(stream)));
}

int gdn_spec_reset(const gdn_spec_cursors *cursors, const int32_t *slot_idx, int32_t B,
                   void *stream) {
    int rc = check_cursors(cursors);
    if (rc) return rc;
    if (B < 0) return GDN_SPEC_EINVAL;
    if (B == 0) return GDN_SPEC_OK;
    if (!slot_idx) return GDN_SPEC_EINVAL;
    return cuda_rc(launch_reset(cursor_args(cursors), slot_idx, B, static_cast<cudaStream_t>(stream)));
}

uint32_t gdn_spec_set_wait_limit(uint32_t polls) {
    return g_data_wait_limit.exchange(polls == 0xFFFFFFFFu ? kWaitLimitDefault : polls);
}

int gdn_spec_read_status(const gdn_spec_cursors *cursors, uint32_t *host_out, int32_t clear,
                         void *stream) {
    int rc = check_cursors(cursors);
    if (rc) return rc;
    if (!host_out) return GDN_SPEC_EINVAL;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(host_out, cursors->status, sizeof(uint32_t),
                                    cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess && clear) e = cudaMemsetAsync(cursors->status, 0, sizeof(uint32_t), st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    return cuda_rc(e);
}

}  // extern "C"
