// verify_kda.cu -- verify kernel for the KDA variant (one gate per key channel,
// prhub summary of sglang PR #36821) on sm_103a: TMA + tcgen05.
//
// Shapes: bf16 I/O, per-key gate, K = 128, V a multiple of 128, ring L <= 64,
// window T <= 8 (an instance for windows of at most 4 and one for 8, so that
// the per-window code of the common case is half as long).  A unit is (batch
// row, v-head, 128 state rows); one persistent CTA of 256 threads per SM.
//
// The math is the GDN verify's output-side UT transform with the scalar decay
// replaced by a vector: with alpha_u = exp(g_u) per channel and
// Gamma(p, r) = prod_{u = r+1 .. p} alpha_u,
//   A[i, r] = beta_i < k^_i o Gamma(i, r), k^_r >   (r < i < n)
//   F[s, r] = < q^_s o Gamma(W+s, r), k^_r >         (r <= W + s)
//   M (I + A) = F, c[j][s] = M[s][j] beta_j,
//   q_eff_s = eG_{W+s} o q^_s - sum_j c[j][s] eG_j o k^_j,   eG_j = prod_{u <= j} alpha_u,
//   o_s = scale (S0 q_eff_s + sum_j c[j][s] v_j).
// The decay now sits inside the contraction over K, so A and F are not a
// Gram matrix scaled afterwards.  They factor through 16-token block
// boundaries: for a target at position p in block b and a source r in an
// earlier block b', Gamma(p, r) = Lin(p) o Mid(b', b) o Rin(r) with
//   Lin(p)    = prod_{u = 16 b .. p} alpha_u          (from the start of p's block),
//   Rin(r)    = prod_{u = r+1 .. 16 b' + 15} alpha_u  (to the end of r's block),
//   Mid(b',b) = the whole blocks strictly between,
// every factor a product of values <= 1, so nothing overflows and no bound on
// the gate is needed.  So A and F outside the diagonal blocks come from one
// tcgen05 kind::tf32 MMA per target block b: D_b = L R_b^T with L's rows
// k^_x o Lin(p_x) (keys and queries, M = 128) and R_b's rows
// k^_r o Rin(r) o Mid(blk r, b) (r < 16 b, N = 16 b).  Inside a diagonal block
// the products are formed directly as running products on the CUDA cores
// (a ratio Lin(p) / Lin(r) could be 0 / 0).  The solve, q_eff (per channel,
// with the running eG_j), the V-term and the checkpoint product (tile by TMA,
// kind::tf32, P = S0 q_eff^T) follow the GDN tensor-core verify.
//
// Side channel: the window's raw k (one writer per k-head), raw v, its per-
// channel g and beta go to ring positions (base + W + s) & (L-1) as the other
// verify kernels write them.
#include <cuda.h>

#include <mutex>
#include <type_traits>

#include "common.cuh"
#include "ptx_sm100.cuh"

namespace gdnspec {
namespace ktc {

constexpr int kThreads = 256;      // two groups of four warps
constexpr int kK = 128;
constexpr int kBV = 128;           // state rows per unit
constexpr int kLMax = 64;          // tokens n = W + T <= L <= 64
constexpr int kTMax = 8;
constexpr int kQRow = 64;          // queries in rows 64 .. 64 + T - 1 of L and X
constexpr int kXRows = 72;
constexpr int kRRows = 96;         // R_1 rows 0..15, R_2 16..47, R_3 48..95
constexpr int kALd = kLMax + 4;

// Shared-memory map (bytes from a 1024-aligned base).
constexpr int kAtomL = 128 * 128;               // one 32-channel slice of L (128 rows); later of S0
constexpr int kOffL = 0;                        // L operand, then the checkpoint tile (64 KiB)
constexpr int kAtomR = kRRows * 128;            // one 32-channel slice of the R operands
constexpr int kOffR = 4 * kAtomL;               // R operands (48 KiB), then the v history
constexpr int kQAtom = 16 * 128;                // one 32-channel slice of q_eff (16 rows)
constexpr int kOffQ = kOffR + 4 * kAtomR;       // q_eff operand (8 KiB)
constexpr int kOffAl = kOffQ + 4 * kQAtom;      // alpha [64][128] fp32
constexpr int kOffX = kOffAl + kLMax * kK * 4;  // raw rows [72][128] bf16 (keys, then queries at 64)
constexpr int kOffA = kOffX + kXRows * kK * 2;  // A [64][kALd] fp32
constexpr int kOffF = kOffA + kLMax * kALd * 4; // F [64][kTMax] fp32 (F[s][r] at r * kTMax + s)
constexpr int kOffC = kOffF + kLMax * kTMax * 4;   // c [64][kTMax] fp32
constexpr int kOffBeta = kOffC + kLMax * kTMax * 4;
constexpr int kOffRn = kOffBeta + kLMax * 4;    // [72] 1/|row|
constexpr int kOffBar = kOffRn + 128 * 4;
constexpr int kOffMisc = kOffBar + 64;
constexpr int kSmemUsed = kOffMisc + 32;
constexpr int kSmemBytes = kSmemUsed + 1024;
static_assert(kOffR % 1024 == 0 && kAtomR % 1024 == 0 && kOffQ % 1024 == 0, "operand bases");
static_assert(kSmemBytes <= 227 * 1024, "shared memory of one CTA");
static_assert(kLMax * kBV * 2 <= 4 * kAtomR, "the v history fits over the R operands");

constexpr uint32_t kTmemCols = 128;
constexpr uint32_t kPCol = 96;      // output product: columns 96 .. 111
// TMEM column of D_b (b = 1, 2, 3): 0, 16, 48; its B operand starts at row
// offset 16 b (b - 1) / 2 of the R region
__host__ __device__ constexpr int dcol(int b) { return 8 * b * (b - 1); }

__device__ __forceinline__ uint32_t sw_f32(int atom, int row, int k) {
    return (uint32_t)((k >> 5) * atom + row * 128 + ((((k & 31) >> 2) ^ (row & 7)) << 4) + (k & 3) * 4);
}
__device__ __forceinline__ float bf(const __nv_bfloat16 *p) { return __bfloat162float(*p); }

// TM: the largest window the instance takes (4 or 8); the shared-memory F and
// c tables keep their kTMax stride either way
template <int TM>
__global__ void __launch_bounds__(kThreads, 1)
verify_kda_kernel(const __grid_constant__ CUtensorMap tmap_s0, LayerArgs P, CursorArgs C,
                  const int32_t *__restrict__ slot_idx, int nunits,
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
    float *const al = reinterpret_cast<float *>(sm + kOffAl);            // alpha [j][c]
    __nv_bfloat16 *const X = reinterpret_cast<__nv_bfloat16 *>(sm + kOffX);   // raw rows [72][128]
    float *const Am = reinterpret_cast<float *>(sm + kOffA);
    float *const Fm = reinterpret_cast<float *>(sm + kOffF);
    float *const Cm = reinterpret_cast<float *>(sm + kOffC);
    float *const betaS = reinterpret_cast<float *>(sm + kOffBeta);
    float *const rn = reinterpret_cast<float *>(sm + kOffRn);
    int *const misc = reinterpret_cast<int *>(sm + kOffMisc);   // [0] TMEM base, [1] error
    const uint32_t bar_ab = sm_s + kOffBar, bar_s0 = sm_s + kOffBar + 8, bar_p = sm_s + kOffBar + 16,
                   bar_vh = sm_s + kOffBar + 24;

    const int T = P.T, L = P.L, HV = P.HV, H = P.H, V = P.V, K = kK;
    const int VB = V / kBV;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int row = tid & (kBV - 1), grp = tid >> 7;
    const __nv_bfloat16 *rawk = reinterpret_cast<const __nv_bfloat16 *>(P.rawk);
    __nv_bfloat16 *rawk_w = reinterpret_cast<__nv_bfloat16 *>(P.rawk);
    const __nv_bfloat16 *rawv = reinterpret_cast<const __nv_bfloat16 *>(P.rawv);
    __nv_bfloat16 *rawv_w = reinterpret_cast<__nv_bfloat16 *>(P.rawv);

    if (tid == 0) {
        misc[1] = 0;
        ptx::mbar_init(bar_ab, 1);
        ptx::mbar_init(bar_s0, 1);
        ptx::mbar_init(bar_p, 1);
        ptx::mbar_init(bar_vh, 1);
        ptx::mbar_init_fence();
        ptx::prefetch_tmap(&tmap_s0);
    }
    if (warp == 0) ptx::tmem_alloc(sm_s + kOffMisc, kTmemCols);
    // q_eff rows of window positions >= T stay zero
    for (int i = tid; i < 4 * kQAtom / 16; i += kThreads)
        reinterpret_cast<float4 *>(sm + kOffQ)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    const uint32_t tmem = static_cast<uint32_t>(misc[0]);
    const uint32_t tl = tmem + ((uint32_t)((warp & 3) * 32) << 16);   // this warp's lanes
    uint32_t ph_ab = 0, ph_s0 = 0, ph_p = 0, ph_vh = 0;
    bool stop = false;

    for (int u = blockIdx.x; u < nunits && !stop; u += gridDim.x) {
        const int vb = u % VB, hv = (u / VB) % HV, bb = u / (VB * HV);
        const int h = hv / P.G, v0 = vb * kBV, vrow = v0 + row;
        const int slot = slot_idx[bb];
        int base = 0, W = 0;
        uint32_t st = 0;
        const bool ok = row_cursor_ok(C, slot, T, L, &base, &W, &st);
        if (!ok) {
            if (st && vb == 0 && hv == 0 && tid == 0) atomicOr(C.status, st);
            if (grp == 0 && vrow < V)
                for (int s = 0; s < T; ++s)
                    out[(((size_t)bb * T + s) * HV + hv) * V + vrow] = __float2bfloat16_rn(0.0f);
            continue;
        }
        const int n = W + T;
        const int nb = (n - 1) >> 4;                 // last target block
        const size_t sh_hv = (size_t)slot * HV + hv, sh_h = (size_t)slot * H + h;
        const bool k_writer = (hv % P.G == 0) && vb == 0;
        uint32_t lost = 0;
        if (tid == 64 && W > 0) {   // the v history into L2 now (read in phase 6)
            const __nv_bfloat16 *rv = rawv + sh_hv * L * V;
            if (V == kBV) {
                const int first = (L - base) < W ? (L - base) : W;
                if (first > 0) ptx::prefetch_l2(rv + (size_t)base * V, first * V * 2);
                if (W > first) ptx::prefetch_l2(rv, (W - first) * V * 2);
            }
        }

        // ---- 1. raw key and query rows into X (two threads per row), their
        //         norms, the key side channel; per-channel gates into alpha;
        //         beta; the window's values (side channel, V-term).  Every
        //         global load of the phase is issued before any is used.
        const int x = tid >> 1, half = tid & 1;
        const bool is_key = x < n, is_q = x >= kQRow && x < kQRow + T;
        const __nv_bfloat16 *src = nullptr;
        if (x < W)
            src = rawk + (sh_h * L + ring_pos(base, x, L)) * K;
        else if (is_key)
            src = k + (((size_t)bb * T + (x - W)) * H + h) * K;
        else if (is_q)
            src = q + (((size_t)bb * T + (x - kQRow)) * H + h) * K;
        uint4 w4[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) w4[c] = make_uint4(0u, 0u, 0u, 0u);
        if (src) {
            const uint4 *s4 = reinterpret_cast<const uint4 *>(src) + 8 * half;
#pragma unroll
            for (int c = 0; c < 8; ++c) w4[c] = s4[c];
        }
        // gates: thread = (4 channels, tokens j0, j0 + 8, ...): the ring's g
        // for history tokens, the raw a (element loads: a and dt_bias carry no
        // alignment promise) for window tokens
        // (a thread's tokens are 8 apart, so at most one of them is in the window)
        const int c4 = 4 * (tid & 31), j0 = tid >> 5;
        float4 gv[kLMax / 8];
#pragma unroll
        for (int m = 0; m < kLMax / 8; ++m) {
            const int j = j0 + 8 * m;
            gv[m] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (j < W) gv[m] = *reinterpret_cast<const float4 *>(P.ring_g + (sh_hv * L + ring_pos(base, j, L)) * K + c4);
        }
        const int jw = W + ((j0 - W) & 7);   // this thread's window token, if jw < n
        float4 aw = make_float4(0.f, 0.f, 0.f, 0.f);
        if (jw < n) {
            const __nv_bfloat16 *ar = a + (((size_t)bb * T + (jw - W)) * HV + hv) * K + c4;
            aw = make_float4(bf(ar), bf(ar + 1), bf(ar + 2), bf(ar + 3));
        }
        float be_in = 0.0f;
        if (tid < W)
            be_in = P.ring_beta[sh_hv * L + ring_pos(base, tid, L)];
        else if (tid < n)
            be_in = bf(bgate + ((size_t)bb * T + (tid - W)) * HV + hv);
        float vwin[TM];
#pragma unroll
        for (int s = 0; s < TM; ++s) vwin[s] = 0.0f;
        __nv_bfloat16 vraw[TM];
        if (grp == 1 && vrow < V) {
#pragma unroll
            for (int s = 0; s < TM; ++s)
                if (s < T) vraw[s] = v[(((size_t)bb * T + s) * HV + hv) * V + vrow];
        }
        const float alog = A_log[hv];
        const float4 dtb4 = make_float4(dt_bias[(size_t)hv * K + c4], dt_bias[(size_t)hv * K + c4 + 1],
                                        dt_bias[(size_t)hv * K + c4 + 2], dt_bias[(size_t)hv * K + c4 + 3]);
        // now use them
        {
            float ss = 0.0f;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const uint32_t ww[4] = {w4[c].x, w4[c].y, w4[c].z, w4[c].w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float lo = __uint_as_float(ww[e] << 16), hi = __uint_as_float(ww[e] & 0xFFFF0000u);
                    ss = fmaf(lo, lo, fmaf(hi, hi, ss));
                }
            }
            ss += __shfl_xor_sync(0xffffffffu, ss, 1);   // the row's other half
            if (src) {
                uint4 *xr = reinterpret_cast<uint4 *>(X + x * K) + 8 * half;
#pragma unroll
                for (int c = 0; c < 8; ++c) xr[c] = w4[c];
                if (half == 0) rn[x] = 1.0f / sqrtf(ss + P.l2_eps);
                if (x >= W && is_key && k_writer) {
                    uint4 *dst = reinterpret_cast<uint4 *>(rawk_w + (sh_h * L + ring_pos(base, x, L)) * K) + 8 * half;
#pragma unroll
                    for (int c = 0; c < 8; ++c) dst[c] = w4[c];
                }
            }
        }
#pragma unroll
        for (int m = 0; m < kLMax / 8; ++m) {
            const int j = j0 + 8 * m;
            if (j >= W) continue;
            const float4 g = gv[m];
            *reinterpret_cast<float4 *>(al + j * K + c4) = make_float4(expf(g.x), expf(g.y), expf(g.z), expf(g.w));
        }
        if (jw < n) {   // the window's gate, written to the ring (side channel)
            const float4 g = make_float4(gate_g(alog, aw.x, dtb4.x), gate_g(alog, aw.y, dtb4.y),
                                         gate_g(alog, aw.z, dtb4.z), gate_g(alog, aw.w, dtb4.w));
            if (vb == 0) *reinterpret_cast<float4 *>(P.ring_g + (sh_hv * L + ring_pos(base, jw, L)) * K + c4) = g;
            *reinterpret_cast<float4 *>(al + jw * K + c4) = make_float4(expf(g.x), expf(g.y), expf(g.z), expf(g.w));
        }
        if (tid < n) {
            float be = be_in;
            if (tid >= W) {
                be = gate_beta(be_in);
                if (vb == 0) P.ring_beta[sh_hv * L + ring_pos(base, tid, L)] = be;
            }
            betaS[tid] = be;
        }
        if (grp == 1 && vrow < V) {
#pragma unroll
            for (int s = 0; s < TM; ++s)
                if (s < T) {
                    vwin[s] = __bfloat162float(vraw[s]);
                    rawv_w[(sh_hv * L + ring_pos(base, W + s, L)) * V + vrow] = vraw[s];
                }
        }
        for (int i = tid; i < kLMax * kALd; i += kThreads) Am[i] = 0.0f;
        for (int i = tid; i < kLMax * kTMax; i += kThreads) Fm[i] = 0.0f;
        __syncthreads();

        // ---- 2. the MMA operands, thread (channel c, group): L rows
        //         k^_x o Lin(p_x) (keys x < n, queries at 64 + s with p = W + s)
        //         and R_b rows k^_r o Rin(r) o Mid(blk r, b) for every target
        //         block b > blk r.  Group 0 takes L and the source block 2,
        //         group 1 the source blocks 0 and 1 (about the same number of
        //         rows); the running products of different blocks are
        //         independent chains, walked side by side.
        {
            const int c = row;
            auto put_l = [&](int xr, float val) {
                *reinterpret_cast<float *>(sm + kOffL + sw_f32(kAtomL, xr, c)) = ptx::round_tf32(val);
            };
            // R rows of source r in block bs: Mid(bs, bt) grows by block bt - 1
            auto put_r = [&](int bs, int r, float val, float blk1, float blk2) {
                for (int bt = bs + 1; bt <= nb; ++bt) {
                    if (bt > bs + 1) val *= (bt == 2 ? blk1 : blk2);
                    *reinterpret_cast<float *>(sm + kOffR + sw_f32(kAtomR, dcol(bt) + r, c)) = ptx::round_tf32(val);
                }
            };
            if (grp == 0) {
                float lin[4] = {1.0f, 1.0f, 1.0f, 1.0f};   // prod_{u = 16 b .. j}
#pragma unroll 2
                for (int jj = 0; jj < 16; ++jj) {
#pragma unroll
                    for (int b = 0; b < 4; ++b) {
                        const int j = 16 * b + jj;
                        if (j < n) {
                            lin[b] *= al[j * K + c];
                            put_l(j, bf(X + j * K + c) * rn[j] * lin[b]);
                            if (j >= W) {   // the query of window position j - W decays like token j
                                const int xq = kQRow + (j - W);
                                put_l(xq, bf(X + xq * K + c) * rn[xq] * lin[b]);
                            }
                        }
                    }
                }
                if (nb >= 3) {
                    float rin = 1.0f;   // prod_{u = r+1 .. 47}
                    for (int r = 47; r >= 32; --r) {
                        if (r < 47) rin *= al[(r + 1) * K + c];
                        put_r(2, r, bf(X + r * K + c) * rn[r] * rin, 1.0f, 1.0f);
                    }
                }
            } else if (nb >= 1) {
                float blk1 = 1.0f, blk2 = 1.0f;
#pragma unroll 4
                for (int jj = 0; jj < 16; ++jj) {
                    if (nb >= 2) blk1 *= al[(16 + jj) * K + c];
                    if (nb >= 3) blk2 *= al[(32 + jj) * K + c];
                }
                float rin0 = 1.0f, rin1 = 1.0f;   // prod_{u = r+1 .. 16 bs + 15}
                for (int rr = 15; rr >= 0; --rr) {
                    if (rr < 15) rin0 *= al[(rr + 1) * K + c];
                    put_r(0, rr, bf(X + rr * K + c) * rn[rr] * rin0, blk1, blk2);
                    if (nb >= 2) {
                        const int r = 16 + rr;
                        if (rr < 15) rin1 *= al[(r + 1) * K + c];
                        put_r(1, r, bf(X + r * K + c) * rn[r] * rin1, blk1, blk2);
                    }
                }
            }
        }
        ptx::fence_proxy_async_smem();
        ptx::tc_fence_before_sync();
        __syncthreads();

        // ---- 3. off-diagonal blocks on the tensor core: D_b = L R_b^T
        if (tid == 0 && nb >= 1) {
            ptx::tc_fence_after_sync();
            for (int bt = 1; bt <= nb; ++bt) {
                const uint32_t idesc = ptx::idesc_tf32(128, 16 * bt);
#pragma unroll
                for (int ks = 0; ks < 16; ++ks)
                    ptx::mma_tf32(tmem + dcol(bt),
                                  ptx::smem_desc_sw128(sm_s + kOffL + (ks >> 2) * kAtomL + (ks & 3) * 32),
                                  ptx::smem_desc_sw128(sm_s + kOffR + dcol(bt) * 128 + (ks >> 2) * kAtomR + (ks & 3) * 32),
                                  idesc, ks != 0);
            }
            ptx::mma_commit(bar_ab);
        }
        // meanwhile the diagonal blocks on the CUDA cores: four threads per
        // target token i (a quarter of K each) walk r down through i's block
        // with z = k^_i o Gamma(i, r) (and, for a window token, zq =
        // q^_s o Gamma(i, r) with s = i - W)
        {
            const int i = tid >> 2, part = tid & 3;
            const bool live = i < n, win = live && i >= W;
            const int s = i - W;
            float2 z[16], zq[16];
#pragma unroll
            for (int m = 0; m < 4; ++m) {   // channels 4 (part + 4 m) .. + 3 and + 16 .. (two 16-byte chunks)
#pragma unroll
                for (int hlf = 0; hlf < 2; ++hlf) {
                    const int ch = 8 * (part + 4 * m) + 4 * hlf;
                    const float ri = live ? rn[i] : 0.0f, rq = win ? rn[kQRow + s] : 0.0f;
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int cc = ch + 2 * e;
                        z[4 * m + 2 * hlf + e] = make_float2(live ? bf(X + i * K + cc) * ri : 0.0f,
                                                             live ? bf(X + i * K + cc + 1) * ri : 0.0f);
                        zq[4 * m + 2 * hlf + e] = make_float2(win ? bf(X + (kQRow + s) * K + cc) * rq : 0.0f,
                                                              win ? bf(X + (kQRow + s) * K + cc + 1) * rq : 0.0f);
                    }
                }
            }
            // F[s][i] = <q^_s, k^_i> (Gamma = 1)
            {
                float2 f2 = make_float2(0.f, 0.f);
#pragma unroll
                for (int m = 0; m < 16; ++m) {
                    const int ch = 8 * (part + 4 * (m >> 2)) + 2 * (m & 3);
                    const float2 kx = make_float2(live ? bf(X + i * K + ch) : 0.0f, live ? bf(X + i * K + ch + 1) : 0.0f);
                    f2 = __ffma2_rn(zq[m], kx, f2);
                }
                float f = f2.x + f2.y;
                f += __shfl_xor_sync(0xffffffffu, f, 1);
                f += __shfl_xor_sync(0xffffffffu, f, 2);
                if (win && part == 0) Fm[i * kTMax + s] = f * rn[i];
            }
            const int i0 = i & ~15;   // first token of i's block
            const float bi = live ? betaS[i] : 0.0f;
            // a warp's eight rows are consecutive tokens of one block: the
            // steps run from the warp's last row down to the block's start
            // (warp-uniform), and only warps holding a window row form zq
            auto walk = [&](auto with_q) {
                constexpr bool WQ = decltype(with_q)::value;
                for (int r = (i | 7) - 1; r >= i0; --r) {
                    const bool act = live && r < i;
                    // z *= alpha_{r+1} for rows that have started (r < i); rows
                    // with r >= i wait with z = k^_i
                    float2 acc2 = make_float2(0.f, 0.f), accq2 = make_float2(0.f, 0.f);
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
#pragma unroll
                        for (int hlf = 0; hlf < 2; ++hlf) {
                            const int ch = 8 * (part + 4 * m) + 4 * hlf;
                            const float4 a4 = *reinterpret_cast<const float4 *>(al + (r + 1) * K + ch);
                            const uint2 kr = *reinterpret_cast<const uint2 *>(X + r * K + ch);
                            const float2 alo = act ? make_float2(a4.x, a4.y) : make_float2(1.f, 1.f);
                            const float2 ahi = act ? make_float2(a4.z, a4.w) : make_float2(1.f, 1.f);
                            const float2 klo = make_float2(__uint_as_float(kr.x << 16), __uint_as_float(kr.x & 0xFFFF0000u));
                            const float2 khi = make_float2(__uint_as_float(kr.y << 16), __uint_as_float(kr.y & 0xFFFF0000u));
                            const int mi = 4 * m + 2 * hlf;
                            z[mi] = __fmul2_rn(z[mi], alo);
                            z[mi + 1] = __fmul2_rn(z[mi + 1], ahi);
                            acc2 = __ffma2_rn(z[mi], klo, acc2);
                            acc2 = __ffma2_rn(z[mi + 1], khi, acc2);
                            if (WQ) {
                                zq[mi] = __fmul2_rn(zq[mi], alo);
                                zq[mi + 1] = __fmul2_rn(zq[mi + 1], ahi);
                                accq2 = __ffma2_rn(zq[mi], klo, accq2);
                                accq2 = __ffma2_rn(zq[mi + 1], khi, accq2);
                            }
                        }
                    }
                    float acc = acc2.x + acc2.y;
                    acc += __shfl_xor_sync(0xffffffffu, acc, 1);
                    acc += __shfl_xor_sync(0xffffffffu, acc, 2);
                    float accq = 0.0f;
                    if (WQ) {
                        accq = accq2.x + accq2.y;
                        accq += __shfl_xor_sync(0xffffffffu, accq, 1);
                        accq += __shfl_xor_sync(0xffffffffu, accq, 2);
                    }
                    if (act && part == 0) {
                        Am[i * kALd + r] = bi * acc * rn[r];
                        if (WQ && win) Fm[r * kTMax + s] = accq * rn[r];
                    }
                }
            };
            if (__any_sync(0xffffffffu, win))
                walk(std::true_type{});
            else
                walk(std::false_type{});
        }
        // the off-diagonal blocks from TMEM: lane x is target row x (key i = x,
        // or query s = x - 64); its block's columns r < 16 blk(p)
        if (nb >= 1) {
            if (!ptx::mbar_wait(bar_ab, ph_ab)) lost |= 1u;
            ph_ab ^= 1u;
        }
        ptx::tc_fence_after_sync();
        // L is dead: the checkpoint tile goes over it now
        bool tile_issued = false;   // (thread 0)
        if (tid == 0 && !lost) {
            tile_issued = true;
            ptx::mbar_expect_tx(bar_s0, 4 * kAtomL);
            const int32_t y = (int32_t)(((size_t)slot * HV + hv) * V + v0);
#pragma unroll
            for (int kb = 0; kb < 4; ++kb) ptx::tma_load_2d(sm_s + kOffL + kb * kAtomL, &tmap_s0, bar_s0, kb * 32, y);
        }
        if (nb >= 1 && grp == 0 && !__any_sync(0xffffffffu, lost != 0)) {
            const int x = row;
            const bool is_key = x < n, is_q = x >= kQRow && x < kQRow + T;
            const int p = is_key ? x : W + (x - kQRow);
            const int b = (is_key || is_q) ? (p >> 4) : 0;
            for (int bt = 1; bt <= nb; ++bt) {   // warp-uniform loads; lane keeps its own block
                for (int cc = 0; cc < bt; ++cc) {
                    float d16[16];
                    ptx::tmem_ld16(tl + dcol(bt) + 16 * cc, d16);
                    ptx::tmem_ld_wait();
                    if (b == bt) {
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            const int r = 16 * cc + e;
                            if (is_key)
                                Am[x * kALd + r] = betaS[x] * d16[e];
                            else
                                Fm[r * kTMax + (x - kQRow)] = d16[e];
                        }
                    }
                }
            }
        }
        __syncthreads();
        if (__syncthreads_or(lost != 0)) {
            stop = true;
        }
        if (!stop) {
            // ---- 5. the v history into the dead R operands (bulk copies), issued
            //         by warp 4 while warps 0..3 solve
            if (warp == 4 && W > 0) {
                ptx::fence_proxy_async_smem();
                if (lane == 0) ptx::mbar_expect_tx(bar_vh, (uint32_t)(W * kBV * 2));
                __syncwarp();
                if (V == kBV) {
                    if (lane == 0) {
                        const int n1 = (L - base) < W ? (L - base) : W;
                        ptx::bulk_copy_g2s(sm_s + kOffR, rawv + (sh_hv * L + base) * V, n1 * kBV * 2, bar_vh);
                        if (W > n1)
                            ptx::bulk_copy_g2s(sm_s + kOffR + n1 * kBV * 2, rawv + sh_hv * L * V, (W - n1) * kBV * 2,
                                               bar_vh);
                    }
                } else {
                    for (int jj = lane; jj < W; jj += 32)
                        ptx::bulk_copy_g2s(sm_s + kOffR + jj * kBV * 2,
                                           rawv + (sh_hv * L + ring_pos(base, jj, L)) * V + v0, kBV * 2, bar_vh);
                }
            }
            // ---- 4. M (I + A) = F^T: the T right-hand sides, s in warp s % 4
            //         (warps 0..3); lane l ends with M[s][l], M[s][l+32]
            if (warp < 4) {
                constexpr int SPW = TM / 4;
                float f0[SPW], f1[SPW];
#pragma unroll
                for (int qq = 0; qq < SPW; ++qq) {
                    const int sq = warp + 4 * qq;
                    f0[qq] = (sq < T && lane < n) ? Fm[lane * kTMax + sq] : 0.0f;
                    f1[qq] = (sq < T && lane + 32 < n) ? Fm[(lane + 32) * kTMax + sq] : 0.0f;
                }
                // four tokens j-3..j per step: their 4 x 4 diagonal block is
                // solved on every lane, then all lanes apply the four updates
                // (which leave f[j-3..j] at their final values)
                int j = n - 1;
                for (; j >= 3; j -= 4) {
                    float ar[4][2];
#pragma unroll
                    for (int x = 0; x < 4; ++x) {
                        ar[x][0] = Am[(j - x) * kALd + lane];
                        ar[x][1] = Am[(j - x) * kALd + 32 + lane];
                    }
                    const float d0 = Am[j * kALd + j - 1], d1 = Am[j * kALd + j - 2], d2 = Am[j * kALd + j - 3];
                    const float d3 = Am[(j - 1) * kALd + j - 2], d4 = Am[(j - 1) * kALd + j - 3];
                    const float d5 = Am[(j - 2) * kALd + j - 3];
#pragma unroll
                    for (int qq = 0; qq < SPW; ++qq) {
                        float fj[4];
#pragma unroll
                        for (int x = 0; x < 4; ++x)
                            fj[x] = __shfl_sync(0xffffffffu, (j - x) < 32 ? f0[qq] : f1[qq], (j - x) & 31);
                        const float m0 = fj[0];
                        const float m1 = fmaf(-d0, m0, fj[1]);
                        const float m2 = fmaf(-d3, m1, fmaf(-d1, m0, fj[2]));
                        const float m3 = fmaf(-d5, m2, fmaf(-d4, m1, fmaf(-d2, m0, fj[3])));
                        f0[qq] = fmaf(-ar[3][0], m3, fmaf(-ar[2][0], m2, fmaf(-ar[1][0], m1, fmaf(-ar[0][0], m0, f0[qq]))));
                        f1[qq] = fmaf(-ar[3][1], m3, fmaf(-ar[2][1], m2, fmaf(-ar[1][1], m1, fmaf(-ar[0][1], m0, f1[qq]))));
                    }
                }
                for (; j >= 0; --j) {
                    const float a0 = Am[j * kALd + lane], a1 = Am[j * kALd + 32 + lane];
#pragma unroll
                    for (int qq = 0; qq < SPW; ++qq) {
                        const float m = __shfl_sync(0xffffffffu, j < 32 ? f0[qq] : f1[qq], j & 31);
                        f0[qq] = fmaf(-a0, m, f0[qq]);
                        f1[qq] = fmaf(-a1, m, f1[qq]);
                    }
                }
#pragma unroll
                for (int hlf = 0; hlf < 2; ++hlf) {
                    const int jj = lane + 32 * hlf;
                    const float bj = jj < n ? betaS[jj] : 0.0f;
#pragma unroll
                    for (int qq = 0; qq < SPW; ++qq) {
                        const int sq = warp + 4 * qq;
                        Cm[jj * kTMax + sq] = (hlf ? f1[qq] : f0[qq]) * bj;
                    }
                }
            }
            __syncthreads();

            float vt[TM];
#pragma unroll
            for (int s = 0; s < TM; ++s) vt[s] = 0.0f;
            if (grp == 0) {
                // ---- 6. q_eff (thread = key channel):
                //         eG_{W+s} q^_s - sum_j c[j][s] eG_j k^_j, eG running
                const int kk = row;
                float acc[TM], eW[TM];
#pragma unroll
                for (int s = 0; s < TM; ++s) acc[s] = eW[s] = 0.0f;
                float e = 1.0f;
                for (int j = 0; j < n; ++j) {
                    e *= al[j * K + kk];
                    const float x = e * bf(X + j * K + kk) * rn[j];
                    float cj[TM];
#pragma unroll
                    for (int q4 = 0; q4 < TM / 4; ++q4) {
                        const float4 c = *reinterpret_cast<const float4 *>(Cm + j * kTMax + 4 * q4);
                        cj[4 * q4] = c.x; cj[4 * q4 + 1] = c.y; cj[4 * q4 + 2] = c.z; cj[4 * q4 + 3] = c.w;
                    }
#pragma unroll
                    for (int s = 0; s < TM; ++s) {
                        acc[s] = fmaf(-cj[s], x, acc[s]);
                        if (j == W + s) eW[s] = e;
                    }
                }
#pragma unroll
                for (int s = 0; s < TM; ++s)
                    if (s < T) {
                        const float qe = acc[s] + eW[s] * bf(X + (kQRow + s) * K + kk) * rn[kQRow + s];
                        *reinterpret_cast<float *>(sm + kOffQ + sw_f32(kQAtom, s, kk)) = qe;
                    }
                ptx::fence_proxy_async_smem();
            } else {
                // ---- 6'. the V-term of this state row: sum_j c[j][s] v_j
                if (W > 0) {
                    if (!ptx::mbar_wait(bar_vh, ph_vh)) lost |= 2u;
                    ph_vh ^= 1u;
                }
                if (vrow < V && !(lost & 2u)) {
                    const __nv_bfloat16 *vh = reinterpret_cast<const __nv_bfloat16 *>(sm + kOffR);
                    for (int jj = 0; jj < W; ++jj) {
                        const float x = __bfloat162float(vh[jj * kBV + row]);
                        float cj[TM];
#pragma unroll
                        for (int q4 = 0; q4 < TM / 4; ++q4) {
                            const float4 c = *reinterpret_cast<const float4 *>(Cm + jj * kTMax + 4 * q4);
                            cj[4 * q4] = c.x; cj[4 * q4 + 1] = c.y; cj[4 * q4 + 2] = c.z; cj[4 * q4 + 3] = c.w;
                        }
#pragma unroll
                        for (int s = 0; s < TM; ++s) vt[s] = fmaf(cj[s], x, vt[s]);
                    }
#pragma unroll
                    for (int s2 = 0; s2 < TM; ++s2) {
                        if (s2 < T) {
                            float cj[TM];
#pragma unroll
                            for (int q4 = 0; q4 < TM / 4; ++q4) {
                                const float4 c = *reinterpret_cast<const float4 *>(Cm + (W + s2) * kTMax + 4 * q4);
                                cj[4 * q4] = c.x; cj[4 * q4 + 1] = c.y; cj[4 * q4 + 2] = c.z; cj[4 * q4 + 3] = c.w;
                            }
#pragma unroll
                            for (int s = 0; s < TM; ++s) vt[s] = fmaf(cj[s], vwin[s2], vt[s]);
                        }
                    }
                }
            }
            const int stop2 = __syncthreads_or(lost != 0);

            // ---- 7. P = S0 q_eff^T (tile by TMA over the dead L), outputs
            if (tid == 0) {
                const bool s0_ok = ptx::mbar_wait(bar_s0, ph_s0, tile_wait_limit);
                if (s0_ok && !stop2) {
                    ptx::tc_fence_after_sync();
                    constexpr uint32_t idesc = ptx::idesc_tf32(128, 16);
#pragma unroll
                    for (int kb = 0; kb < 4; ++kb)
#pragma unroll
                        for (int ks = 0; ks < 4; ++ks)
                            ptx::mma_tf32(tmem + kPCol, ptx::smem_desc_sw128(sm_s + kOffL + kb * kAtomL + ks * 32),
                                          ptx::smem_desc_sw128(sm_s + kOffQ + kb * kQAtom + ks * 32), idesc,
                                          (kb | ks) != 0);
                }
                if (!s0_ok) {
                    lost |= 4u;
                    ptx::mbar_wait(bar_s0, ph_s0);   // drain the tile before the CTA reuses or leaves
                }
                ptx::mma_commit(bar_p);
            }
            ph_s0 ^= 1u;
            if (!ptx::mbar_wait(bar_p, ph_p)) lost |= 8u;
            ph_p ^= 1u;
            ptx::tc_fence_after_sync();
            const int stop3 = __syncthreads_or(lost != 0);
            if (grp == 1) {
                float pr8[8];
                ptx::tmem_ld8(tl + kPCol, pr8);
                ptx::tmem_ld_wait();
                if (!stop2 && !stop3 && vrow < V) {
#pragma unroll
                    for (int s = 0; s < TM; ++s)
                        if (s < T)
                            out[(((size_t)bb * T + s) * HV + hv) * V + vrow] = __float2bfloat16_rn(P.scale * (pr8[s] + vt[s]));
                }
            }
            if (stop2 || stop3) stop = true;
        } else if (tid == 0) {
            // a wait ran out before the solve: drain what is still in flight
            if (nb >= 1 && (lost & 1u)) ptx::mbar_wait(bar_ab, ph_ab ^ 1u);
            if (tile_issued) ptx::mbar_wait(bar_s0, ph_s0);
        }
        if (stop && tid == 0) misc[1] = 1;
        // the tile, the operands and TMEM are reused by the next unit
        ptx::fence_proxy_async_smem();
        ptx::tc_fence_before_sync();
        __syncthreads();
        ptx::tc_fence_after_sync();
    }

    ptx::tc_fence_before_sync();
    __syncthreads();
    if (tid == 0 && misc[1]) atomicOr(C.status, GDN_SPEC_ST_TIMEOUT);
    if (warp == 0) {
        ptx::tc_fence_after_sync();
        ptx::tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace ktc

namespace {

using EncodeTiledFnK = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                    const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                    const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                    CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFnK encode_fn_k() {
    static EncodeTiledFnK fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFnK>(p);
    });
    return fn;
}

constexpr int kMaxDevicesK = 64;
int g_grid_k[kMaxDevicesK];
std::mutex g_mu_k;

cudaError_t setup_k(int dev, int *grid) {
    std::lock_guard<std::mutex> lk(g_mu_k);
    if (!g_grid_k[dev]) {
        cudaError_t e = cudaFuncSetAttribute(ktc::verify_kda_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             ktc::kSmemBytes);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(ktc::verify_kda_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     ktc::kSmemBytes);
        if (e != cudaSuccess) return e;
        int sms = 0;
        if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
        g_grid_k[dev] = sms;   // one CTA per SM (shared memory)
    }
    *grid = g_grid_k[dev];
    return cudaSuccess;
}

}  // namespace

// Shapes of the tensor-core KDA verify.
bool verify_kda_tc_supported(const LayerArgs &P, bool kda, bool bf16) {
    return bf16 && kda && P.K == ktc::kK && P.V % ktc::kBV == 0 && P.L <= ktc::kLMax && P.T <= ktc::kTMax;
}

cudaError_t launch_verify_kda_tc(const LayerArgs &P, const CursorArgs &C, const int32_t *slot_idx, int B,
                                 const void *q, const void *k, const void *v, const void *a, const void *b,
                                 const float *A_log, const float *dt_bias, void *out, cudaStream_t stream) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevicesK) return cudaErrorInvalidDevice;
    int grid = 0;
    if ((e = setup_k(dev, &grid)) != cudaSuccess) return e;
    const int nunits = B * P.HV * (P.V / ktc::kBV);
    if (grid > nunits) grid = nunits;
    if (grid <= 0) return cudaSuccess;
    EncodeTiledFnK enc = encode_fn_k();
    if (!enc) return cudaErrorNotSupported;
    CUtensorMap tmap;
    const cuuint64_t gdim[2] = {(cuuint64_t)P.K, (cuuint64_t)P.num_slots * P.HV * P.V};
    const cuuint64_t gstride[1] = {(cuuint64_t)P.K * sizeof(float)};
    const cuuint32_t box[2] = {32, (cuuint32_t)ktc::kBV};
    const cuuint32_t estride[2] = {1, 1};
    if (enc(&tmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, P.checkpoint, gdim, gstride, box, estride,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    auto kern = P.T <= 4 ? ktc::verify_kda_kernel<4> : ktc::verify_kda_kernel<8>;
    kern<<<grid, ktc::kThreads, ktc::kSmemBytes, stream>>>(
        tmap, P, C, slot_idx, nunits, static_cast<const __nv_bfloat16 *>(q), static_cast<const __nv_bfloat16 *>(k),
        static_cast<const __nv_bfloat16 *>(v), static_cast<const __nv_bfloat16 *>(a),
        static_cast<const __nv_bfloat16 *>(b), A_log, dt_bias, static_cast<__nv_bfloat16 *>(out), data_wait_limit());
    return cudaGetLastError();
}

}  // namespace gdnspec
