// verify_tc.cu -- verify kernel for the Qwen3-Next-shaped GDN layer on
// sm_103a: TMA + tcgen05 (5th-generation tensor cores, TMEM accumulators).
//
// Shapes: bf16 I/O, scalar (GDN) gate, K = 128, V a multiple of 128, ring
// L <= 64, window T <= 8.  One CTA of 128 threads per (V-block of 128 rows,
// batch row, v-head); no layer axis (layers are chain-dependent inside the
// forward; blog post on sglang PR #28695, §1.2).
//
// The math is the chunked UT transform applied from the output side (see
// verify_generic.cu for the derivation):
//   Gram       G = X X^T over the n = W + T keys (rows 0..n-1 of X) and the
//              T window queries (rows 64..64+T-1 of X), K = 128 contraction
//              -> tcgen05.mma kind::tf32, fp32 accumulator in TMEM.
//   per row i  A[i, r] = beta_i Gamma(i, r) G[i, r], F[i, s] = Gamma(W+s, i) G[i, 64+s]
//              (decays as running products of alpha; one thread per token)
//   M          M (I + A) = F^T, backward substitution (one warp per window token)
//   q_eff_s    eG_{W+s} q^_s - sum_j M[s, j] beta_j eG_j k^_j       (K-vector)
//   P          P = S0 q_eff^T: the checkpoint tile times T columns
//              -> tcgen05.mma kind::tf32 with S0 staged by TMA.
//   o_s        scale * (P[:, s] + sum_j M[s, j] beta_j v_j)
// The Gram and the checkpoint product are the two dense contractions of the
// path; everything else is O(n) per thread or O(n^2) per CTA on CUDA cores.
//
// Data movement: the checkpoint tile (128 x 128 fp32 = 64 KiB) is the bulk of
// the bytes.  Its L2 prefetch is issued as soon as the cursors are known; the
// keys, gates and ring history are read while it is in flight; the TMA tile
// load into shared memory is issued after the key buffers are dead, so the
// checkpoint tile reuses their space and the CTA needs ~77 KiB of shared
// memory (two CTAs per SM).  The ring history of v is prefetched to L2 too and
// read by each thread for its own row.
//
// Side channel (sglang PR #36821 ring-write placement): the window's raw k
// (one writer per k-head), raw v (each V-block its rows) and the fp32 g and
// beta computed here (V-block 0) go to ring positions (base + W + s) & (L-1),
// which no CTA reads in this launch.
#include <cuda.h>

#include "common.cuh"
#include "ptx_sm100.cuh"

namespace gdnspec {
namespace tc {

constexpr int kThreads = 128;
constexpr int kK = 128;
constexpr int kBV = 128;           // rows of the checkpoint tile per CTA
constexpr int kLMax = 64;          // ring length limit (keys fit rows 0..63)
constexpr int kTMax = 8;           // window limit (queries in rows 64..71)
constexpr int kQRow = 64;          // first query row of X
constexpr int kXRows = 80;         // Gram N (keys + queries, padded to 16)
constexpr int kXAtom = kXRows * 128;   // bytes of one 32-float K slice of X
constexpr int kS0Atom = kBV * 128;     // bytes of one 32-float K slice of S0
constexpr int kQAtom = 16 * 128;       // bytes of one K slice of q_eff (N = 16)
constexpr int kALd = kLMax + 1;        // row stride (floats) of A
constexpr int kFLd = kLMax;            // row stride (floats) of F and c

// shared-memory map (bytes from a 1024-aligned base); R0 is reused: first the
// key phase (X, A, F, gates), then the checkpoint tile
constexpr int kOffX = 0;
constexpr int kOffA = kOffX + 4 * kXAtom;                    // 40960
constexpr int kOffF = kOffA + kLMax * kALd * 4;              // 57600
constexpr int kOffAlpha = kOffF + kTMax * kFLd * 4;          // 59648
constexpr int kOffBeta = kOffAlpha + kLMax * 4;
constexpr int kOffEG = kOffBeta + kLMax * 4;
constexpr int kEndKeyPhase = kOffEG + kLMax * 4;             // 60416
constexpr int kOffS0 = 0;
constexpr int kR0Bytes = 4 * kS0Atom;                        // 65536
constexpr int kOffQ = kR0Bytes;                              // q_eff operand
constexpr int kOffC = kOffQ + 4 * kQAtom;                    // 73728: c = M beta
constexpr int kOffBar = kOffC + kTMax * kFLd * 4;            // 75776
constexpr int kOffMisc = kOffBar + 32;
constexpr int kSmemBytes = kOffMisc + 64 + 1024;             // + alignment slack
static_assert(kEndKeyPhase <= kR0Bytes, "key phase must fit under the checkpoint tile");
// the Gram's A operand reads 128 rows of each X slice; slice 3 runs 48 rows
// past X into the A matrix, which is inside shared memory
static_assert(3 * kXAtom + 128 * 128 <= kR0Bytes, "Gram operand overrun leaves R0");

constexpr uint32_t kTmemCols = 128;
constexpr uint32_t kGramCol = 0;
constexpr uint32_t kPCol = 96;

// byte offset of element (row, k) in a K-major SW128 tile of 128-byte rows
__device__ __forceinline__ uint32_t sw128(int atom_bytes, int row, int k) {
    const int atom = k >> 5, byte = (k & 31) * 4, chunk = byte >> 4;
    return atom * atom_bytes + row * 128 + (((chunk ^ (row & 7)) << 4) | (byte & 15));
}

__global__ void __launch_bounds__(kThreads, 2)
verify_tc_kernel(const __grid_constant__ CUtensorMap tmap_s0, LayerArgs P, CursorArgs C,
                 const int32_t *__restrict__ slot_idx, const __nv_bfloat16 *__restrict__ q,
                 const __nv_bfloat16 *__restrict__ k, const __nv_bfloat16 *__restrict__ v,
                 const __nv_bfloat16 *__restrict__ a, const __nv_bfloat16 *__restrict__ bgate,
                 const float *__restrict__ A_log, const float *__restrict__ dt_bias,
                 __nv_bfloat16 *__restrict__ out) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = ptx::smem_addr(smem_raw);
    const uint32_t pad = (1024u - (raw_s & 1023u)) & 1023u;
    uint8_t *sm = smem_raw + pad;
    const uint32_t sm_s = raw_s + pad;
    float *A = reinterpret_cast<float *>(sm + kOffA);
    float *F = reinterpret_cast<float *>(sm + kOffF);
    float *alpha = reinterpret_cast<float *>(sm + kOffAlpha);
    float *betaS = reinterpret_cast<float *>(sm + kOffBeta);
    float *eG = reinterpret_cast<float *>(sm + kOffEG);
    float *cm = reinterpret_cast<float *>(sm + kOffC);
    int *misc = reinterpret_cast<int *>(sm + kOffMisc);  // slot, base, W, ok, tmem, err
    const uint32_t bar_gram = sm_s + kOffBar, bar_s0 = sm_s + kOffBar + 8,
                   bar_p = sm_s + kOffBar + 16;

    const int hv = blockIdx.x, bb = blockIdx.y, vb = blockIdx.z;
    const int T = P.T, L = P.L, HV = P.HV, H = P.H, V = P.V;
    const int h = hv / P.G;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int v0 = vb * kBV;

    if (tid == 0) {
        int slot = slot_idx[bb], base = 0, W = 0;
        uint32_t st = 0;
        const bool ok = row_cursor_ok(C, slot, T, L, &base, &W, &st);
        if (st && vb == 0 && hv == 0) atomicOr(C.status, st);
        misc[0] = slot;
        misc[1] = base;
        misc[2] = W;
        misc[3] = ok ? 1 : 0;
        misc[5] = 0;
        ptx::mbar_init(bar_gram, 1);
        ptx::mbar_init(bar_s0, 1);
        ptx::mbar_init(bar_p, 1);
        ptx::mbar_init_fence();
        ptx::prefetch_tmap(&tmap_s0);
        if (ok) {  // checkpoint tile and v history into L2 now; used at the end
            const float *s0 = P.checkpoint + (((size_t)slot * HV + hv) * V + v0) * kK;
            ptx::prefetch_l2(s0, kBV * kK * 4);
            const __nv_bfloat16 *rv = reinterpret_cast<const __nv_bfloat16 *>(P.rawv) +
                                      ((size_t)slot * HV + hv) * L * V;
            const int first = (L - base) < W ? (L - base) : W;   // records before the wrap
            if (first > 0) ptx::prefetch_l2(rv + (size_t)base * V, first * V * 2);
            if (W > first) ptx::prefetch_l2(rv, (W - first) * V * 2);
        }
    }
    if (warp == 0) ptx::tmem_alloc(sm_s + kOffMisc + 16, kTmemCols);
    // zero the q_eff operand (rows T..15 stay zero)
    for (int i = tid; i < 4 * kQAtom / 16; i += kThreads)
        reinterpret_cast<float4 *>(sm + kOffQ)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    const uint32_t tmem = static_cast<uint32_t>(misc[4]);
    const int slot = misc[0], base = misc[1], W = misc[2];
    const bool ok = misc[3] != 0;
    const int n = W + T;
    const int vrow = v0 + tid;

    if (ok) {
        const size_t sh_hv = (size_t)slot * HV + hv, sh_h = (size_t)slot * H + h;
        const __nv_bfloat16 *rawk = reinterpret_cast<const __nv_bfloat16 *>(P.rawk);
        __nv_bfloat16 *rawk_w = reinterpret_cast<__nv_bfloat16 *>(P.rawk);
        const __nv_bfloat16 *rawv = reinterpret_cast<const __nv_bfloat16 *>(P.rawv);
        __nv_bfloat16 *rawv_w = reinterpret_cast<__nv_bfloat16 *>(P.rawv);
        const bool k_writer = (hv % P.G == 0) && vb == 0;

        // ---- 1. keys (rows 0..n-1) and queries (rows 64..64+T-1): load, L2-normalise,
        //         store fp32 into X in the SW128 K-major layout.  Lane l holds k = 4l..4l+3.
        {
            constexpr int kRowsPerWarp = (kLMax + kTMax) / 4;  // 18
            uint2 raw[kRowsPerWarp];
#pragma unroll
            for (int i = 0; i < kRowsPerWarp; ++i) {
                const int t = warp + 4 * i;  // token index: keys 0..n-1, then queries
                raw[i] = make_uint2(0u, 0u);
                if (t < n + T) {
                    const __nv_bfloat16 *src;
                    if (t < W)
                        src = rawk + (sh_h * L + ring_pos(base, t, L)) * kK;
                    else if (t < n)
                        src = k + (((size_t)bb * T + (t - W)) * H + h) * kK;
                    else
                        src = q + (((size_t)bb * T + (t - n)) * H + h) * kK;
                    raw[i] = reinterpret_cast<const uint2 *>(src)[lane];
                }
            }
#pragma unroll
            for (int i = 0; i < kRowsPerWarp; ++i) {
                const int t = warp + 4 * i;
                if (t < n + T) {
                    const __nv_bfloat162 lo = *reinterpret_cast<const __nv_bfloat162 *>(&raw[i].x);
                    const __nv_bfloat162 hi = *reinterpret_cast<const __nv_bfloat162 *>(&raw[i].y);
                    const float2 f0 = __bfloat1622float2(lo), f1 = __bfloat1622float2(hi);
                    float ss = f0.x * f0.x + f0.y * f0.y + f1.x * f1.x + f1.y * f1.y;
                    ss = warp_sum(ss);
                    const float r = 1.0f / sqrtf(ss + P.l2_eps);
                    const int row = t < n ? t : kQRow + (t - n);
                    *reinterpret_cast<float4 *>(sm + kOffX + sw128(kXAtom, row, 4 * lane)) =
                        make_float4(f0.x * r, f0.y * r, f1.x * r, f1.y * r);
                    if (t >= W && t < n && k_writer)  // side channel: raw key, bitwise
                        reinterpret_cast<uint2 *>(rawk_w + (sh_h * L + ring_pos(base, t, L)) * kK)[lane] =
                            raw[i];
                }
            }
        }
        // ---- 2. gates: history from the ring, window computed (and written to the ring)
        if (tid < n) {
            const int j = tid, p = ring_pos(base, j, L);
            float g, be;
            if (j < W) {
                g = P.ring_g[sh_hv * L + p];
                be = P.ring_beta[sh_hv * L + p];
            } else {
                const size_t tok = (size_t)bb * T + (j - W);
                g = gate_g(A_log[hv], __bfloat162float(a[tok * HV + hv]), dt_bias[hv]);
                be = gate_beta(__bfloat162float(bgate[tok * HV + hv]));
                if (vb == 0) {
                    P.ring_g[sh_hv * L + p] = g;
                    P.ring_beta[sh_hv * L + p] = be;
                }
            }
            alpha[j] = expf(g);
            betaS[j] = be;
        }
        // window values of this thread's row: kept for the output, copied to the ring
        float vwin[kTMax];
#pragma unroll
        for (int s = 0; s < kTMax; ++s) {
            vwin[s] = 0.0f;
            if (s < T && vrow < V) {
                const __nv_bfloat16 x = v[(((size_t)bb * T + s) * HV + hv) * V + vrow];
                rawv_w[(sh_hv * L + ring_pos(base, W + s, L)) * V + vrow] = x;
                vwin[s] = __bfloat162float(x);
            }
        }
        ptx::fence_proxy_async_smem();
        __syncthreads();

        // ---- 3. Gram on the tensor core: D[i, j] = <X_i, X_j>, M = 128, N = 80
        if (tid == 0) {
            ptx::tc_fence_after_sync();
            constexpr uint32_t idesc = ptx::idesc_tf32(128, kXRows);
#pragma unroll
            for (int kb = 0; kb < 4; ++kb)
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    const uint64_t d = ptx::smem_desc_sw128(sm_s + kOffX + kb * kXAtom + ks * 32);
                    ptx::mma_tf32(tmem + kGramCol, d, d, idesc, (kb | ks) != 0);
                }
            ptx::mma_commit(bar_gram);
        }
        bool waited = ptx::mbar_wait(bar_gram, 0);
        ptx::tc_fence_after_sync();
        float g[kXRows];
        {
            const uint32_t tbase = tmem + ((uint32_t)(warp * 32) << 16) + kGramCol;
#pragma unroll
            for (int c = 0; c < kXRows / 16; ++c) {
                float r[16];
                ptx::tmem_ld16(tbase + 16 * c, r);
#pragma unroll
                for (int x = 0; x < 16; ++x) g[16 * c + x] = r[x];
            }
            ptx::tmem_ld_wait();
        }
        if (!waited && tid == 0) misc[5] = 1;

        // ---- 4. per token i (thread i): row i of A, row i of F, eG_i
        const int i = tid;
        if (i < n) {
            const float bi = betaS[i];
            float c = 1.0f;
#pragma unroll
            for (int r = kLMax - 1; r >= 0; --r) {
                if (r < i) {
                    c *= alpha[r + 1];                       // Gamma(i, r)
                    A[i * kALd + r] = bi * c * g[r];
                }
            }
            float cf = 1.0f;
            for (int t = i + 1; t < W; ++t) cf *= alpha[t];  // Gamma(W-1, i)
#pragma unroll
            for (int s = 0; s < kTMax; ++s) {
                if (s < T) {
                    const int t = W + s;
                    if (t > i) cf *= alpha[t];
                    F[s * kFLd + i] = t >= i ? cf * g[kQRow + s] : 0.0f;
                }
            }
            float e = 1.0f;
            for (int t = 0; t <= i; ++t) e *= alpha[t];
            eG[i] = e;
        }
        __syncthreads();

        // ---- 5. M (I + A) = F^T by backward substitution; c[s, j] = M[s, j] beta_j
        for (int s = warp; s < T; s += kThreads / 32) {
            float f0 = lane < n ? F[s * kFLd + lane] : 0.0f;
            float f1 = lane + 32 < n ? F[s * kFLd + lane + 32] : 0.0f;
            for (int j = W + s; j >= 0; --j) {
                const float m = __shfl_sync(0xffffffffu, j < 32 ? f0 : f1, j & 31);
                if (lane == 0) cm[s * kFLd + j] = m * betaS[j];
                if (lane < j) f0 -= A[j * kALd + lane] * m;
                if (lane + 32 < j) f1 -= A[j * kALd + lane + 32] * m;
            }
            for (int j = W + s + 1 + lane; j < kLMax; j += 32) cm[s * kFLd + j] = 0.0f;
        }
        __syncthreads();

        // ---- 6. q_eff (thread = key channel): eG_{W+s} q^_s - sum_j c[s, j] eG_j k^_j
        {
            const int kk = tid;
            float acc[kTMax];
#pragma unroll
            for (int s = 0; s < kTMax; ++s) acc[s] = 0.0f;
            for (int j = 0; j < n; ++j) {
                const float x = eG[j] * *reinterpret_cast<const float *>(sm + kOffX + sw128(kXAtom, j, kk));
#pragma unroll
                for (int s = 0; s < kTMax; ++s)
                    if (s < T) acc[s] -= cm[s * kFLd + j] * x;
            }
#pragma unroll
            for (int s = 0; s < kTMax; ++s) {
                if (s < T) {
                    acc[s] += eG[W + s] *
                              *reinterpret_cast<const float *>(sm + kOffX + sw128(kXAtom, kQRow + s, kk));
                    *reinterpret_cast<float *>(sm + kOffQ + sw128(kQAtom, s, kk)) = acc[s];
                }
            }
        }
        ptx::fence_proxy_async_smem();
        __syncthreads();

        // ---- 7. checkpoint tile by TMA (over the dead key buffers), then P = S0 q_eff^T
        if (tid == 0) {
            ptx::fence_proxy_async_smem();
            ptx::mbar_expect_tx(bar_s0, kR0Bytes);
            const int32_t y = (int32_t)((sh_hv * V) + v0);
#pragma unroll
            for (int kb = 0; kb < 4; ++kb)
                ptx::tma_load_2d(sm_s + kOffS0 + kb * kS0Atom, &tmap_s0, bar_s0, kb * 32, y);
        }
        // the v history of this thread's row (L2-resident by now), folded with c
        float vt[kTMax];
#pragma unroll
        for (int s = 0; s < kTMax; ++s) vt[s] = 0.0f;
        if (vrow < V) {
            for (int j0 = 0; j0 < W; j0 += 8) {
                float x[8];
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    x[u] = j0 + u < W ? __bfloat162float(rawv[(sh_hv * L + ring_pos(base, j0 + u, L)) * V + vrow])
                                      : 0.0f;
#pragma unroll
                for (int u = 0; u < 8; ++u)
#pragma unroll
                    for (int s = 0; s < kTMax; ++s)
                        if (s < T && j0 + u < W) vt[s] += cm[s * kFLd + j0 + u] * x[u];
            }
#pragma unroll
            for (int s2 = 0; s2 < kTMax; ++s2)
#pragma unroll
                for (int s = 0; s < kTMax; ++s)
                    if (s < T && s2 < T) vt[s] += cm[s * kFLd + W + s2] * vwin[s2];
        }
        waited = ptx::mbar_wait(bar_s0, 0);
        if (tid == 0) {
            if (!waited) {
                misc[5] = 1;
            } else {
                ptx::tc_fence_after_sync();
                constexpr uint32_t idesc = ptx::idesc_tf32(128, 16);
#pragma unroll
                for (int kb = 0; kb < 4; ++kb)
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        ptx::mma_tf32(tmem + kPCol,
                                      ptx::smem_desc_sw128(sm_s + kOffS0 + kb * kS0Atom + ks * 32),
                                      ptx::smem_desc_sw128(sm_s + kOffQ + kb * kQAtom + ks * 32),
                                      idesc, (kb | ks) != 0);
            }
            ptx::mma_commit(bar_p);
        }
        waited = ptx::mbar_wait(bar_p, 0) && waited;
        ptx::tc_fence_after_sync();
        float pr[16];
        ptx::tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + kPCol, pr);
        ptx::tmem_ld_wait();
        if (!waited) misc[5] = 1;
        if (vrow < V) {
#pragma unroll
            for (int s = 0; s < kTMax; ++s)
                if (s < T)
                    out[(((size_t)bb * T + s) * HV + hv) * V + vrow] =
                        __float2bfloat16_rn(P.scale * (pr[s] + vt[s]));
        }
    } else if (vrow < V) {
        for (int s = 0; s < T; ++s)
            out[(((size_t)bb * T + s) * HV + hv) * V + vrow] = __float2bfloat16_rn(0.0f);
    }

    // ---- teardown: every TMEM read is complete; free the columns
    ptx::tc_fence_before_sync();
    __syncthreads();
    if (tid == 0 && misc[5]) atomicOr(C.status, GDN_SPEC_ST_TIMEOUT);
    if (warp == 0) {
        ptx::tc_fence_after_sync();
        ptx::tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace tc

bool verify_tc_supported(const LayerArgs &P, bool kda, bool bf16) {
    return bf16 && !kda && P.K == tc::kK && P.V % tc::kBV == 0 && P.L <= tc::kLMax &&
           P.T <= tc::kTMax;
}

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

}  // namespace

cudaError_t launch_verify_tc(const LayerArgs &P, const CursorArgs &C, const int32_t *slot_idx,
                             int B, const void *q, const void *k, const void *v, const void *a,
                             const void *b, const float *A_log, const float *dt_bias, void *out,
                             cudaStream_t stream) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    // the checkpoint as a 2-D tensor [num_slots * HV * V rows, K fp32], boxes of
    // 32 x 128 (one 128-byte swizzle span by the CTA's 128 rows)
    CUtensorMap tmap;
    const cuuint64_t gdim[2] = {(cuuint64_t)P.K, (cuuint64_t)P.num_slots * P.HV * P.V};
    const cuuint64_t gstride[1] = {(cuuint64_t)P.K * sizeof(float)};
    const cuuint32_t box[2] = {32, (cuuint32_t)tc::kBV};
    const cuuint32_t estride[2] = {1, 1};
    CUresult r = enc(&tmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, P.checkpoint, gdim, gstride, box,
                     estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(tc::verify_tc_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         tc::kSmemBytes);
    if (e != cudaSuccess) return e;
    dim3 grid(P.HV, B, P.V / tc::kBV);
    tc::verify_tc_kernel<<<grid, tc::kThreads, tc::kSmemBytes, stream>>>(
        tmap, P, C, slot_idx, static_cast<const __nv_bfloat16 *>(q),
        static_cast<const __nv_bfloat16 *>(k), static_cast<const __nv_bfloat16 *>(v),
        static_cast<const __nv_bfloat16 *>(a), static_cast<const __nv_bfloat16 *>(b), A_log, dt_bias,
        static_cast<__nv_bfloat16 *>(out));
    return cudaGetLastError();
}

}  // namespace gdnspec
