// verify_d.cu -- comparison variant of verify for a ring that also caches
// each token's corrected delta d_t = beta_t (v_t - S_t^- k^_t) (S_t^- the state
// after token t's decay), the first design of the blog post on sglang PR
// #28695 (§12.1, appendix A.1), later replaced there by the raw-record ring.
// With the history's d cached, a verify needs no history solve: only the
// window's T x T system remains, and with T = 1 (plain decode) no system at
// all (the blog's Part A decode, §12.2, §12.9).  The fold still replays the
// raw records, so no rounding of the cached d ever reaches the checkpoint.
//
// Per window position s (token t = W + s), with eG_t the decay from the
// checkpoint through t and Gamma(t, r) the decay over (r, t]:
//   S_t^- k^_t = eG_t S0 k^_t + Hk[s] + sum_{W <= r < t} Gamma(t, r) <k^_r, k^_t> d_r
//   Hk[s]      = sum_{r < W} Gamma(t, r) <k^_r, k^_t> d_r          (history, through d)
//   d_t        = beta_t (v_t - eG_t S0 k^_t - Hk[s]) - sum_{W <= r < t} A[s][r - W] d_r
//   o_t        = scale (eG_t S0 q^_t + Hq[s] + sum_{W <= r <= t} Gamma(t, r) <k^_r, q^_t> d_r)
//   Hq[s]      = sum_{r < W} Gamma(t, r) <k^_r, q^_t> d_r
// Dense contractions on the tensor cores: the raw Gram of all n + T rows
// against the T window keys and T queries (kind::f16, M = 128, N = 16), and
// the checkpoint tile against the 2T scaled window keys and queries
// (kind::tf32, M = 128, N = 16, the tile staged by TMA).  Per state row, the
// history terms Hk, Hq (2T dot products of length W with the d history staged
// in shared memory), the window system and the outputs run on CUDA cores.
//
// Side channels (as gdn_spec_verify): the window's raw records go into the
// ring, and the window's d into the d ring at the same positions.
#include <cuda.h>

#include <mutex>

#include "common.cuh"
#include "ptx_sm100.cuh"

namespace gdnspec {
namespace dtc {

constexpr int kThreads = 128;
constexpr int kK = 128;
constexpr int kBV = 128;           // rows of the checkpoint tile per CTA
constexpr int kLMax = 64;          // ring length limit
constexpr int kTMax = 8;           // window limit
constexpr int kQRow = 64;          // first query row of X
constexpr int kXRows = 80;
constexpr int kXAtom = kXRows * 128;   // one 64-element (bf16) K slice of X
constexpr int kYAtom = 16 * 128;       // one 64-element (bf16) K slice of Y (window keys, queries)
constexpr int kS0Atom = kBV * 128;     // one 32-float K slice of the checkpoint tile
constexpr int kQAtom = 16 * 128;       // one 32-float K slice of the scaled window operand
constexpr int kR0Bytes = 4 * kS0Atom;  // key phase, then the checkpoint tile

// R0 (key phase): X (all key rows, then the queries at row 64), Y (window keys
// in rows 0..T-1, queries in rows 8..8+T-1), the d history, the history
// coefficients, gate tables and norms
constexpr int kOffX = 0;
constexpr int kOffY = kOffX + 2 * kXAtom;                  // 20480
constexpr int kOffDh = kOffY + 2 * kYAtom;                 // [W][kBV] fp32
constexpr int kOffCK = kOffDh + kLMax * kBV * 4;           // [64][kTMax]
constexpr int kOffCQ = kOffCK + kLMax * kTMax * 4;         // [64][kTMax]
constexpr int kOffAlpha = kOffCQ + kLMax * kTMax * 4;
constexpr int kOffBeta = kOffAlpha + kLMax * 4;
constexpr int kOffEG = kOffBeta + kLMax * 4;
constexpr int kOffSuf = kOffEG + kLMax * 4;                // [kLMax + 4]
constexpr int kOffWP = kOffSuf + (kLMax + 4) * 4;          // [kTMax]
constexpr int kOffRn = kOffWP + kTMax * 4;                 // [kXRows]
constexpr int kEndKey = kOffRn + kXRows * 4;
static_assert(kEndKey <= kR0Bytes, "key phase must fit under the checkpoint tile");
static_assert(kXAtom + 128 * 128 <= kR0Bytes, "Gram operand overrun leaves R0");
// after R0: the scaled window operand, the window system, barriers, words
constexpr int kOffQ = kR0Bytes;
constexpr int kOffWin = kOffQ + 4 * kQAtom;                // A[8][8], F[8][8], beta[8]
constexpr int kOffBar = kOffWin + (2 * kTMax * kTMax + kTMax) * 4;
constexpr int kOffMisc = kOffBar + 32;
constexpr int kSmemUsed = kOffMisc + 32;
constexpr int kSmemBytes = kSmemUsed + 1024;
static_assert(3 * (kSmemBytes + 1024) <= 228 * 1024, "three CTAs per SM");

constexpr uint32_t kTmemCols = 32;   // Gram columns 0..15, product columns 16..31
constexpr int kCtasPerSm = 3;
constexpr uint32_t kPCol = 16;

__device__ __forceinline__ uint32_t sw128f(int atom_bytes, int row, int k) {   // fp32 element
    const int atom = k >> 5, byte = (k & 31) * 4, chunk = byte >> 4;
    return atom * atom_bytes + row * 128 + (((chunk ^ (row & 7)) << 4) | (byte & 15));
}
__device__ __forceinline__ uint32_t sw128h(int atom_bytes, int row, int k) {   // bf16 element
    const int atom = k >> 6, e = k & 63;
    return atom * atom_bytes + row * 128 + ((((e >> 3) ^ (row & 7)) << 4) | ((e & 7) * 2));
}

__device__ __forceinline__ float warp_prefix_prod(float x, int lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x *= y;
    }
    return x;
}

__device__ __forceinline__ float bf16w(uint32_t w) { return __uint_as_float(w << 16); }

__device__ __forceinline__ void unit_coords(int u, int HV, int VB, int &bb, int &hv, int &vb) {
    hv = u % HV;
    const int rest = u / HV;
    vb = rest % VB;
    bb = rest / VB;
}

// slot and cursors of unit u into dst[0..3] (slot, base, W, ok); status bits
// as row_cursor_ok sets them
__device__ __forceinline__ void fetch_unit(const LayerArgs &P, const CursorArgs &C,
                                           const int32_t *slot_idx, int u, int nunits, int VB,
                                           int *dst) {
    if (u >= nunits) {
        dst[0] = -1; dst[1] = 0; dst[2] = 0; dst[3] = 0;
        return;
    }
    int bb, hv, vb;
    unit_coords(u, P.HV, VB, bb, hv, vb);
    const int slot = slot_idx[bb];
    uint32_t st = 0;
    int base = 0, wp = 0;
    const bool ok = row_cursor_ok(C, slot, P.T, P.L, &base, &wp, &st);
    if (st && vb == 0 && hv == 0) atomicOr(C.status, st);
    dst[0] = slot; dst[1] = ok ? base : 0; dst[2] = ok ? wp : 0; dst[3] = ok ? 1 : 0;
}

template <int TM>
struct Loads {
    uint4 raw[8];
    uint32_t g_in, b_in;
    float alog, dtb;
    uint32_t vwin[TM];
};

template <int TM>
__device__ __forceinline__ void issue_loads(const LayerArgs &P, int slot, int base, int W, bool ok,
                                            int bb, int hv, int vb, int tid,
                                            const __nv_bfloat16 *__restrict__ q,
                                            const __nv_bfloat16 *__restrict__ k,
                                            const __nv_bfloat16 *__restrict__ v,
                                            const __nv_bfloat16 *__restrict__ a,
                                            const __nv_bfloat16 *__restrict__ bgate,
                                            const float *__restrict__ A_log,
                                            const float *__restrict__ dt_bias, Loads<TM> &R) {
    const int T = P.T, L = P.L, HV = P.HV, H = P.H, V = P.V;
    const int h = hv / P.G, n = W + T;
    const size_t sh_h = (size_t)slot * H + h, sh_hv = (size_t)slot * HV + hv;
    const __nv_bfloat16 *rawk = reinterpret_cast<const __nv_bfloat16 *>(P.rawk);
    const int t = tid >> 1, half = tid & 1;
    const bool has_row = ok && t < n + T;
    const __nv_bfloat16 *src = q;
    if (t < W)
        src = rawk + (sh_h * L + ring_pos(base, t, L)) * kK;
    else if (t < n)
        src = k + (((size_t)bb * T + (t - W)) * H + h) * kK;
    else if (has_row)
        src = q + (((size_t)bb * T + (t - n)) * H + h) * kK;
#pragma unroll
    for (int c = 0; c < 8; ++c) R.raw[c] = make_uint4(0u, 0u, 0u, 0u);
    if (has_row) {
        const uint4 *s4 = reinterpret_cast<const uint4 *>(src) + 8 * half;
#pragma unroll
        for (int c = 0; c < 8; ++c) R.raw[c] = s4[c];
    }
    R.g_in = R.b_in = 0u;
    R.alog = R.dtb = 0.0f;
    if (ok && tid < W) {
        const int pj = ring_pos(base, tid, L);
        R.g_in = reinterpret_cast<const uint32_t *>(P.ring_g)[sh_hv * L + pj];
        R.b_in = reinterpret_cast<const uint32_t *>(P.ring_beta)[sh_hv * L + pj];
    } else if (ok && tid < n) {
        const size_t tk = (size_t)bb * T + (tid - W);
        R.g_in = reinterpret_cast<const unsigned short *>(a)[tk * HV + hv];
        R.b_in = reinterpret_cast<const unsigned short *>(bgate)[tk * HV + hv];
        R.alog = A_log[hv];
        R.dtb = dt_bias[hv];
    }
    const int vrow = vb * kBV + tid;
#pragma unroll
    for (int s = 0; s < TM; ++s) R.vwin[s] = 0u;
    if (ok && vrow < V) {
#pragma unroll
        for (int s = 0; s < TM; ++s)
            if (s < T)
                R.vwin[s] = reinterpret_cast<const unsigned short *>(v)[(((size_t)bb * T + s) * HV + hv) * V + vrow];
    }
}

// One unit = (batch row, v-head, block of 128 state rows); persistent CTAs.
template <int TM>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
verify_d_kernel(const __grid_constant__ CUtensorMap tmap_s0, LayerArgs P, CursorArgs C,
                float *__restrict__ dring, const int32_t *__restrict__ slot_idx, int nunits,
                const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k,
                const __nv_bfloat16 *__restrict__ v, const __nv_bfloat16 *__restrict__ a,
                const __nv_bfloat16 *__restrict__ bgate, const float *__restrict__ A_log,
                const float *__restrict__ dt_bias, __nv_bfloat16 *__restrict__ out,
                uint32_t tile_wait_limit) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = ptx::smem_addr(smem_raw);
    const uint32_t pad = (1024u - (raw_s & 1023u)) & 1023u;
    uint8_t *sm = smem_raw + pad;
    const uint32_t sm_s = raw_s + pad;
    float *const dh = reinterpret_cast<float *>(sm + kOffDh);
    float *const cK = reinterpret_cast<float *>(sm + kOffCK);
    float *const cQ = reinterpret_cast<float *>(sm + kOffCQ);
    float *const alpha = reinterpret_cast<float *>(sm + kOffAlpha);
    float *const betaS = reinterpret_cast<float *>(sm + kOffBeta);
    float *const eG = reinterpret_cast<float *>(sm + kOffEG);
    float *const suf = reinterpret_cast<float *>(sm + kOffSuf);
    float *const wprod = reinterpret_cast<float *>(sm + kOffWP);
    float *const rn = reinterpret_cast<float *>(sm + kOffRn);
    float *const Aw = reinterpret_cast<float *>(sm + kOffWin);             // [kTMax][kTMax]
    float *const Fw = Aw + kTMax * kTMax;                                   // [kTMax][kTMax]
    float *const bw = Fw + kTMax * kTMax;                                   // [kTMax]
    int *misc = reinterpret_cast<int *>(sm + kOffMisc);   // [0..3] next unit, [4] tmem, [5] err
    const uint32_t bar_gram = sm_s + kOffBar, bar_dh = sm_s + kOffBar + 8,
                   bar_s0 = sm_s + kOffBar + 16, bar_p = sm_s + kOffBar + 24;

    const int T = P.T, L = P.L, HV = P.HV, H = P.H, V = P.V;
    const int VB = V / kBV;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const __nv_bfloat16 *rawk = reinterpret_cast<const __nv_bfloat16 *>(P.rawk);
    __nv_bfloat16 *rawk_w = reinterpret_cast<__nv_bfloat16 *>(P.rawk);
    __nv_bfloat16 *rawv_w = reinterpret_cast<__nv_bfloat16 *>(P.rawv);

    if (tid == 0) {
        misc[5] = 0;
        ptx::mbar_init(bar_gram, 1);
        ptx::mbar_init(bar_dh, 1);
        ptx::mbar_init(bar_s0, 1);
        ptx::mbar_init(bar_p, 1);
        ptx::mbar_init_fence();
        ptx::prefetch_tmap(&tmap_s0);
        fetch_unit(P, C, slot_idx, blockIdx.x, nunits, VB, misc);
    }
    if (warp == 0) ptx::tmem_alloc(sm_s + kOffMisc + 16, kTmemCols);
    for (int i = tid; i < 4 * kQAtom / 16; i += kThreads)
        reinterpret_cast<float4 *>(sm + kOffQ)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    const uint32_t tmem = static_cast<uint32_t>(misc[4]);
    uint32_t ph_gram = 0, ph_dh = 0, ph_s0 = 0, ph_p = 0;

    int slot = misc[0], base = misc[1], W = misc[2];
    bool ok = misc[3] != 0;
    Loads<TM> R;
    int u = blockIdx.x;
    if (u < nunits) {
        int bb0, hv0, vb0;
        unit_coords(u, HV, VB, bb0, hv0, vb0);
        issue_loads<TM>(P, slot, base, W, ok, bb0, hv0, vb0, tid, q, k, v, a, bgate, A_log, dt_bias, R);
    }

    for (; u < nunits; u += gridDim.x) {
        int bb, hv, vb;
        unit_coords(u, HV, VB, bb, hv, vb);
        const int un = u + gridDim.x;
        const int h = hv / P.G;
        const int v0 = vb * kBV, vrow = v0 + tid;
        const int n = W + T;
        const size_t sh_hv = (size_t)slot * HV + hv, sh_h = (size_t)slot * H + h;
        const bool k_writer = (hv % P.G == 0) && vb == 0;
        uint32_t lost = 0;
        float Hk[TM], Hq[TM];
#pragma unroll
        for (int s = 0; s < TM; ++s) Hk[s] = Hq[s] = 0.0f;

        if (ok) {
            // the d history of this CTA's rows into shared memory (bulk copies;
            // the tile of the previous unit is consumed: its MMA completed)
            if (warp == 0 && W > 0) {
                ptx::fence_proxy_async_smem();
                if (lane == 0) ptx::mbar_expect_tx(bar_dh, (uint32_t)W * kBV * 4);
                __syncwarp();
                if (V == kBV) {
                    if (lane == 0) {
                        const int n1 = (L - base) < W ? (L - base) : W;
                        ptx::bulk_copy_g2s(sm_s + kOffDh, dring + (sh_hv * L + base) * V, n1 * kBV * 4, bar_dh);
                        if (W > n1)
                            ptx::bulk_copy_g2s(sm_s + kOffDh + n1 * kBV * 4, dring + sh_hv * L * V,
                                               (W - n1) * kBV * 4, bar_dh);
                    }
                } else {
                    for (int jj = lane; jj < W; jj += 32)
                        ptx::bulk_copy_g2s(sm_s + kOffDh + jj * kBV * 4,
                                           dring + (sh_hv * L + ring_pos(base, jj, L)) * V + v0, kBV * 4,
                                           bar_dh);
                }
            }
            // ---- 1. raw key rows into X (and the window keys and queries into
            //         Y), their norms; gates; the ring side channel
            const int half = tid & 1;
            for (int pass = 0; pass < 2; ++pass) {
                if (pass == 1 && n + T <= 64) break;
                const int t = (tid >> 1) + 64 * pass;
                const bool has_row = t < n + T;
                if (pass == 1) {
                    const __nv_bfloat16 *src = q;
                    if (t < W)
                        src = rawk + (sh_h * L + ring_pos(base, t, L)) * kK;
                    else if (t < n)
                        src = k + (((size_t)bb * T + (t - W)) * H + h) * kK;
                    else if (has_row)
                        src = q + (((size_t)bb * T + (t - n)) * H + h) * kK;
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        R.raw[c] = has_row ? reinterpret_cast<const uint4 *>(src)[8 * half + c]
                                           : make_uint4(0u, 0u, 0u, 0u);
                }
                float ss[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint32_t w4[4] = {R.raw[c].x, R.raw[c].y, R.raw[c].z, R.raw[c].w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w4[e]));
                        ss[e] = fmaf(f.x, f.x, ss[e]);
                        ss[e] = fmaf(f.y, f.y, ss[e]);
                    }
                }
                float sq = (ss[0] + ss[1]) + (ss[2] + ss[3]);
                sq += __shfl_xor_sync(0xffffffffu, sq, 1);
                if (has_row) {
                    const int row = t < n ? t : kQRow + (t - n);
                    if (half == 0) rn[row] = 1.0f / sqrtf(sq + P.l2_eps);
                    uint8_t *xr = sm + kOffX + half * kXAtom + row * 128;
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        *reinterpret_cast<uint4 *>(xr + ((c ^ (row & 7)) << 4)) = R.raw[c];
                    if (t >= W) {   // a window key (Y row s) or a query (Y row 8 + s)
                        const int yrow = t < n ? t - W : 8 + (t - n);
                        uint8_t *yr = sm + kOffY + half * kYAtom + yrow * 128;
#pragma unroll
                        for (int c = 0; c < 8; ++c)
                            *reinterpret_cast<uint4 *>(yr + ((c ^ (yrow & 7)) << 4)) = R.raw[c];
                    }
                    if (t >= W && t < n && k_writer) {
                        uint4 *dst = reinterpret_cast<uint4 *>(rawk_w + (sh_h * L + ring_pos(base, t, L)) * kK);
#pragma unroll
                        for (int c = 0; c < 8; ++c) dst[8 * half + c] = R.raw[c];
                    }
                }
            }
            if (tid < n) {
                const int pj = ring_pos(base, tid, L);
                float g = __uint_as_float(R.g_in), be = __uint_as_float(R.b_in);
                if (tid >= W) {
                    g = gate_g(R.alog, bf16w(R.g_in), R.dtb);
                    be = gate_beta(bf16w(R.b_in));
                    if (vb == 0) {
                        P.ring_g[sh_hv * L + pj] = g;
                        P.ring_beta[sh_hv * L + pj] = be;
                    }
                }
                alpha[tid] = expf(g);
                betaS[tid] = be;
            }
#pragma unroll
            for (int s = 0; s < TM; ++s)
                if (s < T && vrow < V) rawv_w[(sh_hv * L + ring_pos(base, W + s, L)) * V + vrow] =
                        __ushort_as_bfloat16((unsigned short)R.vwin[s]);
            ptx::fence_proxy_async_smem();
            __syncthreads();

            // ---- 2. raw Gram of every row against the window keys and queries
            //         (D[r][s] = <x_r, k_s>, D[r][8 + s] = <x_r, q_s>); decays meanwhile
            if (tid == 0) {
                ptx::tc_fence_after_sync();
                constexpr uint32_t idesc = ptx::idesc_bf16(128, 16);
#pragma unroll
                for (int kb = 0; kb < 2; ++kb)
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        ptx::mma_bf16(tmem, ptx::smem_desc_sw128(sm_s + kOffX + kb * kXAtom + ks * 32),
                                      ptx::smem_desc_sw128(sm_s + kOffY + kb * kYAtom + ks * 32), idesc,
                                      (kb | ks) != 0);
                ptx::mma_commit(bar_gram);
            }
            if (warp == 1) {   // eG_j = prod_{t <= j} alpha_t
                const float a0 = 2 * lane < n ? alpha[2 * lane] : 1.0f;
                const float a1 = 2 * lane + 1 < n ? alpha[2 * lane + 1] : 1.0f;
                const float incl = warp_prefix_prod(a0 * a1, lane);
                float excl = __shfl_up_sync(0xffffffffu, incl, 1);
                if (lane == 0) excl = 1.0f;
                eG[2 * lane] = excl * a0;
                eG[2 * lane + 1] = incl;
            } else if (warp == 2) {   // suf[t] = prod_{u=t}^{W-1} alpha_u (suf[W] = 1)
                const int u0 = 2 * lane, u1 = 2 * lane + 1;
                const float a0 = u0 < W ? alpha[W - 1 - u0] : 1.0f;
                const float a1 = u1 < W ? alpha[W - 1 - u1] : 1.0f;
                const float incl = warp_prefix_prod(a0 * a1, lane);
                float excl = __shfl_up_sync(0xffffffffu, incl, 1);
                if (lane == 0) excl = 1.0f;
                if (u0 < W) suf[W - 1 - u0] = excl * a0;
                if (u1 < W) suf[W - 1 - u1] = incl;
                if (lane == 0) suf[W] = 1.0f;
            } else if (warp == 3 && lane == 0) {   // wprod[s] = prod_{t=W}^{W+s} alpha_t
                float c = 1.0f;
#pragma unroll
                for (int s = 0; s < TM; ++s)
                    if (s < T) {
                        c *= alpha[W + s];
                        wprod[s] = c;
                    }
            }
            __syncthreads();
            if (!ptx::mbar_wait(bar_gram, ph_gram)) lost |= 1u;
            ph_gram ^= 1u;
            ptx::tc_fence_after_sync();

            // ---- 3. coefficients: history rows (Gamma(W+s, r) G^), the window
            //         system; the scaled window operand of the checkpoint product
            if (warp * 32 < n) {
                const uint32_t taddr = tmem + ((uint32_t)(warp * 32) << 16);
                float gr[16];
                ptx::tmem_ld16(taddr, gr);
                ptx::tmem_ld_wait();
                const int r = tid;
                if (r < W) {
                    const float base_f = suf[r + 1] * rn[r];
#pragma unroll
                    for (int s = 0; s < TM; ++s) {
                        float ck = 0.0f, cq = 0.0f;
                        if (s < T) {
                            const float f = base_f * wprod[s];
                            ck = f * rn[W + s] * gr[s];
                            cq = f * rn[kQRow + s] * gr[8 + s];
                        }
                        cK[r * kTMax + s] = ck;
                        cQ[r * kTMax + s] = cq;
                    }
                } else if (r < n) {   // window key s' = r - W: column s' of A, row s' of F
                    const int sp = r - W;
                    float gam = 1.0f;   // Gamma(W+s, W+s'), s >= s'
#pragma unroll
                    for (int s = 0; s < TM; ++s) {
                        if (s < T && s >= sp) {
                            if (s > sp) gam *= alpha[W + s];
                            if (s > sp) Aw[s * kTMax + sp] = betaS[W + s] * gam * rn[r] * rn[W + s] * gr[s];
                            Fw[sp * kTMax + s] = gam * rn[r] * rn[kQRow + s] * gr[8 + s];
                        }
                    }
                    bw[sp] = betaS[r];
                }
            }
            {   // thread = key channel: rows s and 8 + s of the operand
                const int kk = tid;
#pragma unroll
                for (int s = 0; s < TM; ++s)
                    if (s < T) {
                        const float e = eG[W + s];
                        const float xk = bf16w(*reinterpret_cast<const unsigned short *>(sm + kOffY + sw128h(kYAtom, s, kk)));
                        const float xq = bf16w(*reinterpret_cast<const unsigned short *>(sm + kOffY + sw128h(kYAtom, 8 + s, kk)));
                        *reinterpret_cast<float *>(sm + kOffQ + sw128f(kQAtom, s, kk)) = e * rn[W + s] * xk;
                        *reinterpret_cast<float *>(sm + kOffQ + sw128f(kQAtom, 8 + s, kk)) = e * rn[kQRow + s] * xq;
                    }
            }
            ptx::fence_proxy_async_smem();
            __syncthreads();

            // ---- 4. the history through d: Hk[s], Hq[s] of this thread's state row
            if (W > 0) {
                if (!ptx::mbar_wait(bar_dh, ph_dh)) lost |= 2u;
                ph_dh ^= 1u;
            }
            if (!(lost & 2u)) {
                float2 hk[TM / 2 > 0 ? TM / 2 : 1], hq[TM / 2 > 0 ? TM / 2 : 1];
#pragma unroll
                for (int s2 = 0; s2 < (TM + 1) / 2; ++s2) hk[s2] = hq[s2] = make_float2(0.f, 0.f);
#pragma unroll 4
                for (int r = 0; r < W; ++r) {
                    const float x = dh[r * kBV + tid];
                    const float2 x2 = make_float2(x, x);
#pragma unroll
                    for (int s = 0; s < TM; s += 2) {
                        const float2 ck = *reinterpret_cast<const float2 *>(cK + r * kTMax + s);
                        const float2 cq = *reinterpret_cast<const float2 *>(cQ + r * kTMax + s);
                        hk[s / 2] = __ffma2_rn(ck, x2, hk[s / 2]);
                        hq[s / 2] = __ffma2_rn(cq, x2, hq[s / 2]);
                    }
                }
#pragma unroll
                for (int s = 0; s < TM; ++s) {
                    Hk[s] = (s & 1) ? hk[s / 2].y : hk[s / 2].x;
                    Hq[s] = (s & 1) ? hq[s / 2].y : hq[s / 2].x;
                }
            }
            // the tile's TMA load follows the barrier below: order this
            // thread's generic shared-memory reads before it
            ptx::fence_proxy_async_smem();
            if (tid == 32) fetch_unit(P, C, slot_idx, un, nunits, VB, misc);
        } else {
            if (tid == 0) fetch_unit(P, C, slot_idx, un, nunits, VB, misc);
            if (vrow < V)
                for (int s = 0; s < T; ++s)
                    out[(((size_t)bb * T + s) * HV + hv) * V + vrow] = __float2bfloat16_rn(0.0f);
        }
        int stop = __syncthreads_or(lost != 0);   // R0 free; the next unit's cursors visible

        // ---- 5. checkpoint tile by TMA; P = S0 [eG k^ ; eG q^]^T; the window
        //         system and the outputs per state row; d into the d ring
        const bool tiles = ok && !stop;
        if (tiles && tid == 0) {
            ptx::mbar_expect_tx(bar_s0, kR0Bytes);
            const int32_t y = (int32_t)(sh_hv * V + v0);
#pragma unroll
            for (int kb = 0; kb < 4; ++kb) ptx::tma_load_2d(sm_s + kb * kS0Atom, &tmap_s0, bar_s0, kb * 32, y);
        }
        // this unit's window values, before the next unit's loads replace them
        uint32_t vcur[TM];
#pragma unroll
        for (int s = 0; s < TM; ++s) vcur[s] = R.vwin[s];
        const int nslot = misc[0], nbase = misc[1], nW = misc[2];
        const bool nok = misc[3] != 0;
        if (un < nunits) {
            int bbn, hvn, vbn;
            unit_coords(un, HV, VB, bbn, hvn, vbn);
            issue_loads<TM>(P, nslot, nbase, nW, nok, bbn, hvn, vbn, tid, q, k, v, a, bgate, A_log, dt_bias, R);
        }
        if (tiles) {
            const bool s0_ok = ptx::mbar_wait(bar_s0, ph_s0, tile_wait_limit);
            ph_s0 ^= 1u;
            if (!s0_ok) lost |= 4u;
            if (tid == 0) {
                if (s0_ok) {
                    ptx::tc_fence_after_sync();
                    constexpr uint32_t idesc = ptx::idesc_tf32(128, 16);
#pragma unroll
                    for (int kb = 0; kb < 4; ++kb)
#pragma unroll
                        for (int ks = 0; ks < 4; ++ks)
                            ptx::mma_tf32(tmem + kPCol, ptx::smem_desc_sw128(sm_s + kb * kS0Atom + ks * 32),
                                          ptx::smem_desc_sw128(sm_s + kOffQ + kb * kQAtom + ks * 32), idesc,
                                          (kb | ks) != 0);
                }
                ptx::mma_commit(bar_p);
            }
            if (!ptx::mbar_wait(bar_p, ph_p)) lost |= 8u;
            ph_p ^= 1u;
            ptx::tc_fence_after_sync();
            float pr[16];   // columns s: eG S0 k^_s, columns 8 + s: eG S0 q^_s
            ptx::tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + kPCol, pr);
            ptx::tmem_ld_wait();
            if (!lost && vrow < V) {
                // the window's T x T system (forward substitution), then the outputs
                float d[TM];
#pragma unroll
                for (int s = 0; s < TM; ++s) {
                    d[s] = 0.0f;
                    if (s < T) {
                        float r = bw[s] * (bf16w(vcur[s]) - pr[s] - Hk[s]);
#pragma unroll
                        for (int sp = 0; sp < s; ++sp) r = fmaf(-Aw[s * kTMax + sp], d[sp], r);
                        d[s] = r;
                    }
                }
#pragma unroll
                for (int s = 0; s < TM; ++s)
                    if (s < T) {
                        float o = pr[8 + s] + Hq[s];
#pragma unroll
                        for (int sp = 0; sp <= s; ++sp) o = fmaf(Fw[sp * kTMax + s], d[sp], o);
                        out[(((size_t)bb * T + s) * HV + hv) * V + vrow] = __float2bfloat16_rn(P.scale * o);
                        dring[(sh_hv * L + ring_pos(base, W + s, L)) * V + vrow] = d[s];
                    }
            }
        }
        slot = nslot; base = nbase; W = nW; ok = nok;
        ptx::tc_fence_before_sync();
        stop = __syncthreads_or(lost != 0);
        ptx::tc_fence_after_sync();
        if (stop) {
            if (tid == 0) misc[5] = 1;
            if (lost & 1u) ptx::mbar_wait(bar_gram, ph_gram ^ 1u);
            if (lost & 2u) ptx::mbar_wait(bar_dh, ph_dh ^ 1u);
            if (lost & 4u) ptx::mbar_wait(bar_s0, ph_s0 ^ 1u);
            if (lost & 8u) ptx::mbar_wait(bar_p, ph_p ^ 1u);
            break;
        }
    }

    ptx::tc_fence_before_sync();
    __syncthreads();
    if (tid == 0 && misc[5]) atomicOr(C.status, GDN_SPEC_ST_TIMEOUT);
    if (warp == 0) {
        ptx::tc_fence_after_sync();
        ptx::tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace dtc
}  // namespace gdnspec

namespace gdnspec {

namespace {

using EncodeTiledFnD = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                    const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                    const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                    CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFnD encode_fn_d() {
    static EncodeTiledFnD fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFnD>(p);
    });
    return fn;
}

constexpr int kMaxDevicesD = 64;
int g_grid_d[kMaxDevicesD][2];   // per device and window template: grid size, 0 until set up
std::mutex g_mu_d;

template <int TM>
cudaError_t setup_d(int dev, int inst, int *grid) {
    std::lock_guard<std::mutex> lk(g_mu_d);
    if (!g_grid_d[dev][inst]) {
        auto kern = dtc::verify_d_kernel<TM>;
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             dtc::kSmemBytes);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 (int)cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess) return e;
        int sms = 0, smem_sm = 0, smem_rsv = 0;
        if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
        if ((e = cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev)) !=
            cudaSuccess)
            return e;
        if ((e = cudaDeviceGetAttribute(&smem_rsv, cudaDevAttrReservedSharedMemoryPerBlock, dev)) !=
            cudaSuccess)
            return e;
        int per_sm = smem_sm / (dtc::kSmemBytes + smem_rsv);
        if (per_sm > dtc::kCtasPerSm) per_sm = dtc::kCtasPerSm;
        if (per_sm < 1) per_sm = 1;
        g_grid_d[dev][inst] = sms * per_sm;
    }
    *grid = g_grid_d[dev][inst];
    return cudaSuccess;
}

template <int TM>
cudaError_t launch_d_tm(int dev, int inst, const CUtensorMap &tmap, const LayerArgs &P,
                        const CursorArgs &C, float *dring, const int32_t *slot_idx, int B,
                        const void *q, const void *k, const void *v, const void *a, const void *b,
                        const float *A_log, const float *dt_bias, void *out, cudaStream_t stream) {
    int grid = 0;
    cudaError_t e = setup_d<TM>(dev, inst, &grid);
    if (e != cudaSuccess) return e;
    const int nunits = B * P.HV * (P.V / dtc::kBV);
    if (grid > nunits) grid = nunits;
    dtc::verify_d_kernel<TM><<<grid, dtc::kThreads, dtc::kSmemBytes, stream>>>(
        tmap, P, C, dring, slot_idx, nunits, static_cast<const __nv_bfloat16 *>(q),
        static_cast<const __nv_bfloat16 *>(k), static_cast<const __nv_bfloat16 *>(v),
        static_cast<const __nv_bfloat16 *>(a), static_cast<const __nv_bfloat16 *>(b), A_log, dt_bias,
        static_cast<__nv_bfloat16 *>(out), data_wait_limit());
    return cudaGetLastError();
}

}  // namespace

// Shapes of the derived-d verify: those of the tensor-core verify.
bool verify_d_supported(const LayerArgs &P, bool kda, bool bf16) {
    return bf16 && !kda && P.K == dtc::kK && P.V % dtc::kBV == 0 && P.L <= dtc::kLMax &&
           P.T <= dtc::kTMax;
}

cudaError_t launch_verify_d(const LayerArgs &P, const CursorArgs &C, float *dring,
                            const int32_t *slot_idx, int B, const void *q, const void *k,
                            const void *v, const void *a, const void *b, const float *A_log,
                            const float *dt_bias, void *out, cudaStream_t stream) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevicesD) return cudaErrorInvalidDevice;
    EncodeTiledFnD enc = encode_fn_d();
    if (!enc) return cudaErrorNotSupported;
    // the checkpoint as a 2-D tensor [num_slots * HV * V rows, K fp32], boxes
    // of 32 x 128 with the 128-byte swizzle of the MMA operand
    CUtensorMap tmap;
    const cuuint64_t gdim[2] = {(cuuint64_t)P.K, (cuuint64_t)P.num_slots * P.HV * P.V};
    const cuuint64_t gstride[1] = {(cuuint64_t)P.K * sizeof(float)};
    const cuuint32_t box[2] = {32, (cuuint32_t)dtc::kBV};
    const cuuint32_t estride[2] = {1, 1};
    if (enc(&tmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, P.checkpoint, gdim, gstride, box, estride,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    if (P.T <= 4)
        return launch_d_tm<4>(dev, 0, tmap, P, C, dring, slot_idx, B, q, k, v, a, b, A_log, dt_bias, out, stream);
    return launch_d_tm<8>(dev, 1, tmap, P, C, dring, slot_idx, B, q, k, v, a, b, A_log, dt_bias, out, stream);
}

}  // namespace gdnspec
