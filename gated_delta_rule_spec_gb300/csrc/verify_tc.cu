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
//              (one thread per token; decays are products of alpha, never
//              exponentials of differences of long sums)
//   M          M (I + A) = F^T, backward substitution, one warp per window token
//   q_eff_s    eG_{W+s} q^_s - sum_j M[s, j] beta_j eG_j k^_j       (K-vector)
//   P          P = S0 q_eff^T: the checkpoint tile times T columns
//              -> tcgen05.mma kind::tf32 with S0 staged by TMA.
//   o_s        scale * (P[:, s] + sum_j M[s, j] beta_j v_j)
// The Gram and the checkpoint product are the two dense contractions of the
// path; everything else is O(n) per thread or O(n^2) per CTA on CUDA cores.
//
// Data movement: the checkpoint tile (128 x 128 fp32 = 64 KiB) is the bulk of
// the bytes.  Its L2 prefetch is issued as soon as the cursors are known, as
// is the prefetch of the ring's v history; every other global read of the CTA
// (keys, queries, gates, window values) is issued in one round.  The TMA tile
// load into shared memory is issued after the key buffers are dead, so the
// tile reuses their space and the CTA needs ~73 KiB of shared memory: three
// CTAs per SM.
//
// Side channel (sglang PR #36821 ring-write placement): the window's raw k
// (one writer per k-head), raw v (each V-block its rows) and the fp32 g and
// beta computed here (V-block 0) go to ring positions (base + W + s) & (L-1),
// which no CTA reads in this launch.
#include <cuda.h>

#include <mutex>

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
constexpr int kALd = kLMax + 4;        // row stride (floats) of A: 16-byte rows, conflict-free

// Shared-memory map (bytes from a 1024-aligned base).  R0 holds first the key
// phase (X, A, F, gates, decay products), then the checkpoint tile.  R1 is
// the q_eff operand of the second MMA (16 rows of 128 fp32); rows 8..15 of
// its first two K slices, which only feed output columns that are never read,
// hold c = M beta for the output.
constexpr int kOffX = 0;
constexpr int kOffA = kOffX + 4 * kXAtom;                     // 40960
constexpr int kOffF = kOffA + kLMax * kALd * 4;               // 58368: F, then c eG
constexpr int kOffAlpha = kOffF + kLMax * kTMax * 4;          // 60416
constexpr int kOffBeta = kOffAlpha + kLMax * 4;
constexpr int kOffEG = kOffBeta + kLMax * 4;
constexpr int kOffSuf = kOffEG + kLMax * 4;                   // suffix products, L+1 floats
constexpr int kOffWP = kOffSuf + (kLMax + 4) * 4;             // window products
constexpr int kEndKeyPhase = kOffWP + kTMax * 4;
constexpr int kOffS0 = 0;
constexpr int kR0Bytes = 4 * kS0Atom;                         // 65536
constexpr int kOffQ = kR0Bytes;                               // q_eff operand, 8 KiB
constexpr int kOffBar = kOffQ + 4 * kQAtom;                   // 73728
constexpr int kOffMisc = kOffBar + 32;
constexpr int kSmemUsed = kOffMisc + 32;
constexpr int kSmemBytes = kSmemUsed + 1024;                  // + alignment slack
static_assert(kEndKeyPhase <= kR0Bytes, "key phase must fit under the checkpoint tile");
// the Gram's A operand reads 128 rows of each X slice; slice 3 runs 48 rows
// past X into the A matrix, which is inside shared memory
static_assert(3 * kXAtom + 128 * 128 <= kR0Bytes, "Gram operand overrun leaves R0");
static_assert(3 * (kSmemBytes + 1024) <= 228 * 1024, "three CTAs per SM");

constexpr uint32_t kTmemCols = 128;
// CTAs per SM the kernel is built for: the register cap of the launch bounds
// (65536 / (3 * 128) = 170 per thread) and three TMEM allocations of 128 of
// the SM's 512 columns
constexpr int kCtasPerSm = 3;
static_assert(kCtasPerSm * kTmemCols <= 512, "TMEM columns of the resident CTAs");
constexpr uint32_t kGramCol = 0;
constexpr uint32_t kPCol = 96;

// byte offset of element (row, k) in a K-major SW128 tile of 128-byte rows
__device__ __forceinline__ uint32_t sw128(int atom_bytes, int row, int k) {
    const int atom = k >> 5, byte = (k & 31) * 4, chunk = byte >> 4;
    return atom * atom_bytes + row * 128 + (((chunk ^ (row & 7)) << 4) | (byte & 15));
}

// c[j][s] (j < 64, s < 8) in rows 8..15 of the q_eff operand's first two K slices
__device__ __forceinline__ uint32_t c_off(int j) {
    return kOffQ + (j >> 5) * kQAtom + 1024 + (j & 31) * 32;
}

// warp-wide inclusive prefix product of x
__device__ __forceinline__ float warp_prefix_prod(float x, int lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x *= y;
    }
    return x;
}

// One unit = (batch row, v-head, block of 128 state rows).  Fetching a unit
// means reading its slot and cursors (one thread) and prefetching its
// checkpoint tile and v history into L2.  Inside the unit loop the fetch of
// the next unit is split into stages spread over the current unit, so that no
// stage waits on a load: the slot index, then the cursors, then the checks,
// the prefetch and the hand-over through shared memory.
struct UnitInfo {
    int slot, base, W, ok;
};

__device__ __forceinline__ void unit_coords(int u, int HV, int VB, int &bb, int &hv, int &vb) {
    hv = u % HV;
    const int rest = u / HV;
    vb = rest % VB;
    bb = rest / VB;
}

// Last stage: checks (status bits as row_cursor_ok sets them), L2 prefetch,
// hand-over to dst[0..3].  wp and cbase are only read when the slot is in range.
__device__ __forceinline__ void finish_fetch(const LayerArgs &P, const CursorArgs &C, int u,
                                             int nunits, int VB, int slot, int wp, int cbase,
                                             int *dst) {
    if (u >= nunits) {
        dst[0] = -1; dst[1] = 0; dst[2] = 0; dst[3] = 0;
        return;
    }
    int bb, hv, vb;
    unit_coords(u, P.HV, VB, bb, hv, vb);
    uint32_t st = 0;
    bool ok = false;
    if (slot >= C.num_slots) st = GDN_SPEC_ST_SLOT_OOR;
    else if (slot >= 0) {
        if (wp < 0 || wp > P.L || cbase < 0 || cbase >= P.L) st = GDN_SPEC_ST_CURSOR_CORRUPT;
        else if (wp + P.T > P.L) st = GDN_SPEC_ST_RING_OVERFLOW;
        else ok = true;
    }
    if (st && vb == 0 && hv == 0) atomicOr(C.status, st);
    if (ok) {  // checkpoint tile and v history into L2; used at the end of the unit
        const size_t sh_hv = (size_t)slot * P.HV + hv;
        ptx::prefetch_l2(P.checkpoint + (sh_hv * P.V + vb * kBV) * kK, kBV * kK * 4);
        const __nv_bfloat16 *rv = reinterpret_cast<const __nv_bfloat16 *>(P.rawv) + sh_hv * P.L * P.V;
        if (P.V == kBV) {  // whole records are contiguous: one or two segments
            const int first = (P.L - cbase) < wp ? (P.L - cbase) : wp;
            if (first > 0) ptx::prefetch_l2(rv + (size_t)cbase * P.V, first * P.V * 2);
            if (wp > first) ptx::prefetch_l2(rv, (wp - first) * P.V * 2);
        }
    }
    dst[0] = slot; dst[1] = ok ? cbase : 0; dst[2] = ok ? wp : 0; dst[3] = ok ? 1 : 0;
}

// All stages at once (start-up, and units that have no work to hide it behind).
__device__ __forceinline__ void fetch_unit(const LayerArgs &P, const CursorArgs &C,
                                           const int32_t *slot_idx, int u, int nunits, int VB,
                                           int *dst) {
    int slot = -1, wp = 0, cbase = 0;
    if (u < nunits) {
        int bb, hv, vb;
        unit_coords(u, P.HV, VB, bb, hv, vb);
        slot = slot_idx[bb];
        if (slot >= 0 && slot < C.num_slots) {
            wp = C.write_pos[slot];
            cbase = C.cache_base[slot];
        }
    }
    finish_fetch(P, C, u, nunits, VB, slot, wp, cbase, dst);
}

// The early global reads of a unit, held in registers until its first phase:
// two threads per token row (keys 0..n-1 then the T queries; 128 bytes each),
// the gate inputs of token tid and the window values of state row tid.
template <int TM>
struct UnitLoads {
    uint4 raw[8];
    // raw 32-bit words, converted only when the unit uses them: the ring's
    // fp32 gates, or the window's bf16 gate inputs and values zero-extended
    uint32_t g_in, b_in;
    float alog, dtb;
    uint32_t vwin[TM];
};

__device__ __forceinline__ float bf16_word_to_float(uint32_t w) { return __uint_as_float(w << 16); }

template <int TM>
__device__ __forceinline__ void issue_unit_loads(
    const LayerArgs &P, const UnitInfo &U, int bb, int hv, int vb, int tid,
    const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k,
    const __nv_bfloat16 *__restrict__ v, const __nv_bfloat16 *__restrict__ a,
    const __nv_bfloat16 *__restrict__ bgate, const float *__restrict__ A_log,
    const float *__restrict__ dt_bias, UnitLoads<TM> &R) {
    const int T = P.T, L = P.L, HV = P.HV, H = P.H, V = P.V;
    const int h = hv / P.G, W = U.W, n = W + T, base = U.base;
    const size_t sh_hv = (size_t)U.slot * HV + hv, sh_h = (size_t)U.slot * H + h;
    const __nv_bfloat16 *rawk = reinterpret_cast<const __nv_bfloat16 *>(P.rawk);
    const int t = tid >> 1, half = tid & 1;
    const bool has_row = U.ok && t < n + T;
    const __nv_bfloat16 *src = q;
    if (t < W)
        src = rawk + (sh_h * L + ring_pos(base, t, L)) * kK;
    else if (t < n)
        src = k + (((size_t)bb * T + (t - W)) * H + h) * kK;
    else if (has_row)
        src = q + (((size_t)bb * T + (t - n)) * H + h) * kK;
    // zero first, then guarded loads: nothing here reads a loaded register, so
    // the loads stay in flight until the unit's first phase uses them
#pragma unroll
    for (int c = 0; c < 8; ++c) R.raw[c] = make_uint4(0u, 0u, 0u, 0u);
    if (has_row) {
        const uint4 *s4 = reinterpret_cast<const uint4 *>(src) + 8 * half;
#pragma unroll
        for (int c = 0; c < 8; ++c) R.raw[c] = s4[c];
    }
    R.g_in = R.b_in = 0u;
    R.alog = R.dtb = 0.0f;
    if (U.ok && tid < W) {
        const int pj = ring_pos(base, tid, L);
        R.g_in = reinterpret_cast<const uint32_t *>(P.ring_g)[sh_hv * L + pj];
        R.b_in = reinterpret_cast<const uint32_t *>(P.ring_beta)[sh_hv * L + pj];
    } else if (U.ok && tid < n) {
        const size_t tok = (size_t)bb * T + (tid - W);
        R.g_in = reinterpret_cast<const unsigned short *>(a)[tok * HV + hv];
        R.b_in = reinterpret_cast<const unsigned short *>(bgate)[tok * HV + hv];
        R.alog = A_log[hv];
        R.dtb = dt_bias[hv];
    }
    const int vrow = vb * kBV + tid;
#pragma unroll
    for (int s = 0; s < TM; ++s) R.vwin[s] = 0u;
    if (U.ok && vrow < V) {
#pragma unroll
        for (int s = 0; s < TM; ++s)
            if (s < T)
                R.vwin[s] = reinterpret_cast<const unsigned short *>(v)[(((size_t)bb * T + s) * HV + hv) * V + vrow];
    }
}

// Persistent: each CTA takes units blockIdx.x, blockIdx.x + gridDim.x, ...
// While a unit waits for its checkpoint tile and output MMA, the CTA already
// reads the next unit's cursors and issues that unit's key/gate/value loads.
template <int TM>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
verify_tc_kernel(const __grid_constant__ CUtensorMap tmap_s0, LayerArgs P, CursorArgs C,
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
    float *A = reinterpret_cast<float *>(sm + kOffA);
    float *F = reinterpret_cast<float *>(sm + kOffF);         // F[j][s], later c eG [j][s]
    float *alpha = reinterpret_cast<float *>(sm + kOffAlpha);
    float *betaS = reinterpret_cast<float *>(sm + kOffBeta);
    float *eG = reinterpret_cast<float *>(sm + kOffEG);
    float *suf = reinterpret_cast<float *>(sm + kOffSuf);
    float *wprod = reinterpret_cast<float *>(sm + kOffWP);
    int *misc = reinterpret_cast<int *>(sm + kOffMisc);  // [0..3] next unit, [4] tmem, [5] err
    const uint32_t bar_gram = sm_s + kOffBar, bar_s0 = sm_s + kOffBar + 8,
                   bar_p = sm_s + kOffBar + 16, bar_vh = sm_s + kOffBar + 24;
    // v history of this CTA's rows, staged over the dead A matrix: [W][kBV] bf16
    const __nv_bfloat16 *vh = reinterpret_cast<const __nv_bfloat16 *>(sm + kOffA);

    const int T = P.T, L = P.L, HV = P.HV, H = P.H, V = P.V;
    const int VB = V / kBV;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const __nv_bfloat16 *rawk = reinterpret_cast<const __nv_bfloat16 *>(P.rawk);
    __nv_bfloat16 *rawk_w = reinterpret_cast<__nv_bfloat16 *>(P.rawk);
    const __nv_bfloat16 *rawv = reinterpret_cast<const __nv_bfloat16 *>(P.rawv);
    __nv_bfloat16 *rawv_w = reinterpret_cast<__nv_bfloat16 *>(P.rawv);

    if (tid == 0) {
        misc[5] = 0;
        ptx::mbar_init(bar_gram, 1);
        ptx::mbar_init(bar_s0, 1);
        ptx::mbar_init(bar_p, 1);
        ptx::mbar_init(bar_vh, 1);
        ptx::mbar_init_fence();
        ptx::prefetch_tmap(&tmap_s0);
        fetch_unit(P, C, slot_idx, blockIdx.x, nunits, VB, misc);
    }
    if (warp == 0) ptx::tmem_alloc(sm_s + kOffMisc + 16, kTmemCols);
    // zero the q_eff operand: rows T..7 stay zero; rows 8..15 carry c
    for (int i = tid; i < 4 * kQAtom / 16; i += kThreads)
        reinterpret_cast<float4 *>(sm + kOffQ)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    const uint32_t tmem = static_cast<uint32_t>(misc[4]);
    uint32_t ph_gram = 0, ph_s0 = 0, ph_p = 0, ph_vh = 0;   // mbarrier phase bits

    UnitInfo cur{misc[0], misc[1], misc[2], misc[3]};
    UnitLoads<TM> R;
    int u = blockIdx.x;
    if (u < nunits) {
        const int hv0 = u % HV, rest = u / HV;
        issue_unit_loads<TM>(P, cur, rest / VB, hv0, rest % VB, tid, q, k, v, a, bgate, A_log, dt_bias, R);
    }

    for (; u < nunits; u += gridDim.x) {
        const int hv = u % HV, rest = u / HV, vb = rest % VB, bb = rest / VB;
        const int un = u + gridDim.x;
        const int h = hv / P.G;
        const int v0 = vb * kBV, vrow = v0 + tid;
        const int slot = cur.slot, base = cur.base, W = cur.W;
        const bool ok = cur.ok != 0;
        const int n = W + T;
        const size_t sh_hv = (size_t)slot * HV + hv, sh_h = (size_t)slot * H + h;
        const bool k_writer = (hv % P.G == 0) && vb == 0;
        bool waited = true;
        // waits of this unit that ran out (bit per barrier: Gram, v history,
        // checkpoint tile, output MMA)
        uint32_t lost = 0;
        int f_slot = -1, f_wp = 0, f_base = 0;   // the next unit's fetch (thread 32)
        if (ok && tid == 32 && un < nunits) {     // fetch stage 1: the slot index
            int bbn, hvn, vbn;
            unit_coords(un, HV, VB, bbn, hvn, vbn);
            f_slot = slot_idx[bbn];
        }

        if (ok) {
            // ---- 1. normalise the token rows (loaded earlier) into X (SW128
            //         K-major); gates; ring side channel of the window
            const int half = tid & 1;
            for (int pass = 0; pass < 2; ++pass) {
                if (pass == 1 && n + T <= 64) break;  // a second pass only when W > L - 2T
                const int t = (tid >> 1) + 64 * pass;
                const bool has_row = t < n + T;
                if (pass == 1) {  // rows 64.. (rare): load them now
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
                sq += __shfl_xor_sync(0xffffffffu, sq, 1);   // the row's other half
                if (has_row) {
                    const float r = 1.0f / sqrtf(sq + P.l2_eps);
                    const int row = t < n ? t : kQRow + (t - n);
#pragma unroll
                    for (int c = 0; c < 8; ++c) {  // chunk c of this half: k = 64 half + 8c .. + 7
                        const uint32_t w4[4] = {R.raw[c].x, R.raw[c].y, R.raw[c].z, R.raw[c].w};
                        float f[8];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w4[e]));
                            f[2 * e] = x.x * r;
                            f[2 * e + 1] = x.y * r;
                        }
                        const int k0 = 64 * half + 8 * c;
                        *reinterpret_cast<float4 *>(sm + kOffX + sw128(kXAtom, row, k0)) =
                            make_float4(f[0], f[1], f[2], f[3]);
                        *reinterpret_cast<float4 *>(sm + kOffX + sw128(kXAtom, row, k0 + 4)) =
                            make_float4(f[4], f[5], f[6], f[7]);
                    }
                    if (t >= W && t < n && k_writer) {  // side channel: raw key, bitwise
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
                    g = gate_g(R.alog, bf16_word_to_float(R.g_in), R.dtb);
                    be = gate_beta(bf16_word_to_float(R.b_in));
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

            // ---- 2. Gram on the tensor core (D[i, j] = <X_i, X_j>, M = 128, N = 80),
            //         decay products on CUDA cores meanwhile
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
            if (warp == 1) {  // eG_j = prod_{t <= j} alpha_t, j < n
                const float a0 = 2 * lane < n ? alpha[2 * lane] : 1.0f;
                const float a1 = 2 * lane + 1 < n ? alpha[2 * lane + 1] : 1.0f;
                const float incl = warp_prefix_prod(a0 * a1, lane);
                float excl = __shfl_up_sync(0xffffffffu, incl, 1);
                if (lane == 0) excl = 1.0f;
                eG[2 * lane] = excl * a0;
                eG[2 * lane + 1] = incl;
            } else if (warp == 2) {  // suf[t] = prod_{u=t}^{W-1} alpha_u, t <= W (suf[W] = 1)
                const int u0 = 2 * lane, u1 = 2 * lane + 1;  // reversed index u = W-1-t
                const float a0 = u0 < W ? alpha[W - 1 - u0] : 1.0f;
                const float a1 = u1 < W ? alpha[W - 1 - u1] : 1.0f;
                const float incl = warp_prefix_prod(a0 * a1, lane);
                float excl = __shfl_up_sync(0xffffffffu, incl, 1);
                if (lane == 0) excl = 1.0f;
                if (u0 < W) suf[W - 1 - u0] = excl * a0;
                if (u1 < W) suf[W - 1 - u1] = incl;
                if (lane == 0) suf[W] = 1.0f;
            } else if (warp == 3 && lane == 0) {  // wprod[s] = prod_{t=W}^{W+s} alpha_t
                float c = 1.0f;
#pragma unroll
                for (int s = 0; s < TM; ++s)
                    if (s < T) {
                        c *= alpha[W + s];
                        wprod[s] = c;
                    }
            }
            __syncthreads();
            waited = ptx::mbar_wait(bar_gram, ph_gram);
            ph_gram ^= 1u;
            if (!waited) lost |= 1u;
            ptx::tc_fence_after_sync();
            if (tid == 32 && f_slot >= 0 && f_slot < C.num_slots) {  // fetch stage 2: cursors
                f_wp = C.write_pos[f_slot];
                f_base = C.cache_base[f_slot];
            }

            // ---- 3. per token i (thread i): row i of A (zero above the diagonal), row i of F
            {
                const int i = tid;
                const uint32_t tbase = tmem + ((uint32_t)(warp * 32) << 16) + kGramCol;
                // tcgen05.ld is warp-collective: every load below runs on all lanes
                float gq[16];
                ptx::tmem_ld16(tbase + kQRow, gq);   // columns 64..79: the query columns
                ptx::tmem_ld_wait();
                const bool row_live = i < n;
                const float bi = row_live ? betaS[i] : 0.0f;
                float c = 1.0f;
#pragma unroll 1
                // key columns below n (the bound is the same in every thread),
                // high chunk first
                for (int cc = (n + 15) / 16 - 1; cc >= 0; --cc) {
                    float gk[16];
                    ptx::tmem_ld16(tbase + 16 * cc, gk);
                    ptx::tmem_ld_wait();
                    if (row_live) {
                        float val[16];
#pragma unroll
                        for (int x = 15; x >= 0; --x) {
                            const int r = 16 * cc + x;
                            val[x] = 0.0f;
                            if (r < i) {
                                c *= alpha[r + 1];               // Gamma(i, r)
                                val[x] = bi * c * gk[x];
                            }
                        }
#pragma unroll
                        for (int x = 0; x < 16; x += 4)
                            *reinterpret_cast<float4 *>(A + i * kALd + 16 * cc + x) =
                                make_float4(val[x], val[x + 1], val[x + 2], val[x + 3]);
                    }
                }
                if (row_live) {
                    // Gamma(W+s, i): products of the suffix and window decays
                    const float si = i < W ? suf[i + 1] : 1.0f;
                    float cw = 1.0f;
                    float fr[TM];
#pragma unroll
                    for (int s = 0; s < TM; ++s) {
                        float f = 0.0f;
                        if (s < T) {
                            const int t = W + s;
                            if (i < W) {
                                f = si * wprod[s] * gq[s];
                            } else if (t >= i) {
                                if (t > i) cw *= alpha[t];
                                f = cw * gq[s];
                            }
                        }
                        fr[s] = f;
                    }
#pragma unroll
                    for (int s = 0; s < TM; s += 4)
                        *reinterpret_cast<float4 *>(F + i * TM + s) =
                            make_float4(fr[s], fr[s + 1], fr[s + 2], fr[s + 3]);
                }
            }
            if (!waited && tid == 0) misc[5] = 1;
            __syncthreads();

            // ---- 4. M (I + A) = F^T: the T right-hand sides are independent
            //         systems, s in warp s % 4; lane l ends with M[s][l], M[s][l+32]
            {
                constexpr int SPW = (TM + 3) / 4;   // right-hand sides per warp
                float f0[SPW], f1[SPW];
#pragma unroll
                for (int q = 0; q < SPW; ++q) {
                    const int sq = warp + 4 * q;
                    f0[q] = (sq < T && lane < n) ? F[lane * TM + sq] : 0.0f;
                    f1[q] = (sq < T && lane + 32 < n) ? F[(lane + 32) * TM + sq] : 0.0f;
                }
                // four tokens j-3..j per step: the 4 x 4 diagonal block is solved
                // redundantly on every lane, then all lanes apply the four updates
                // (which also leave f[j-3..j] equal to their final values)
                int j = n - 1;
                for (; j >= 3; j -= 4) {
                    float ar[4][2], d[6];
#pragma unroll
                    for (int qq = 0; qq < 4; ++qq) {
                        ar[qq][0] = A[(j - qq) * kALd + lane];
                        ar[qq][1] = A[(j - qq) * kALd + 32 + lane];
                    }
                    d[0] = A[j * kALd + j - 1];        // A[j][j-1]
                    d[1] = A[j * kALd + j - 2];        // A[j][j-2]
                    d[2] = A[j * kALd + j - 3];        // A[j][j-3]
                    d[3] = A[(j - 1) * kALd + j - 2];  // A[j-1][j-2]
                    d[4] = A[(j - 1) * kALd + j - 3];  // A[j-1][j-3]
                    d[5] = A[(j - 2) * kALd + j - 3];  // A[j-2][j-3]
#pragma unroll
                    for (int q = 0; q < SPW; ++q) {
                        float fj[4];
#pragma unroll
                        for (int qq = 0; qq < 4; ++qq)
                            fj[qq] = __shfl_sync(0xffffffffu, (j - qq) < 32 ? f0[q] : f1[q], (j - qq) & 31);
                        const float m0 = fj[0];
                        const float m1 = fmaf(-d[0], m0, fj[1]);
                        const float m2 = fmaf(-d[3], m1, fmaf(-d[1], m0, fj[2]));
                        const float m3 = fmaf(-d[5], m2, fmaf(-d[4], m1, fmaf(-d[2], m0, fj[3])));
                        f0[q] = fmaf(-ar[3][0], m3, fmaf(-ar[2][0], m2, fmaf(-ar[1][0], m1, fmaf(-ar[0][0], m0, f0[q]))));
                        f1[q] = fmaf(-ar[3][1], m3, fmaf(-ar[2][1], m2, fmaf(-ar[1][1], m1, fmaf(-ar[0][1], m0, f1[q]))));
                    }
                }
                for (; j >= 0; --j) {
                    const float a0 = A[j * kALd + lane], a1 = A[j * kALd + 32 + lane];
#pragma unroll
                    for (int q = 0; q < SPW; ++q) {
                        const float m = __shfl_sync(0xffffffffu, j < 32 ? f0[q] : f1[q], j & 31);
                        f0[q] = fmaf(-a0, m, f0[q]);
                        f1[q] = fmaf(-a1, m, f1[q]);
                    }
                }
                // c = M beta (output) and c eG (effective query), rows j = lane, lane + 32
#pragma unroll
                for (int hlf = 0; hlf < 2; ++hlf) {
                    const int jj = lane + 32 * hlf;
                    const float bj = jj < n ? betaS[jj] : 0.0f, ej = jj < n ? eG[jj] : 0.0f;
#pragma unroll
                    for (int q = 0; q < SPW; ++q) {
                        const int sq = warp + 4 * q;
                        if (sq < TM) {
                            const float cj = (hlf ? f1[q] : f0[q]) * bj;
                            *reinterpret_cast<float *>(sm + c_off(jj) + 4 * sq) = cj;
                            F[jj * TM + sq] = cj * ej;
                        }
                    }
                }
            }
            __syncthreads();

            // ---- 5. the v history of this CTA's rows into the (now dead) A
            //         matrix by 1-D bulk copies: with V = 128 whole records are
            //         contiguous, so the history is one or two ring segments;
            //         otherwise one copy per record, spread over warp 0
            if (warp == 0 && W > 0) {
                ptx::fence_proxy_async_smem();   // the A matrix was last read by generic loads
                if (V == kBV) {
                    if (lane == 0) {
                        ptx::mbar_expect_tx(bar_vh, (uint32_t)W * kBV * 2);
                        const int n1 = (L - base) < W ? (L - base) : W;
                        ptx::bulk_copy_g2s(sm_s + kOffA, rawv + (sh_hv * L + base) * V, n1 * kBV * 2, bar_vh);
                        if (W > n1)
                            ptx::bulk_copy_g2s(sm_s + kOffA + n1 * kBV * 2, rawv + sh_hv * L * V,
                                               (W - n1) * kBV * 2, bar_vh);
                    }
                } else {
                    if (lane == 0) ptx::mbar_expect_tx(bar_vh, (uint32_t)W * kBV * 2);
                    __syncwarp();
                    for (int jj = lane; jj < W; jj += 32)
                        ptx::bulk_copy_g2s(sm_s + kOffA + jj * kBV * 2,
                                           rawv + (sh_hv * L + ring_pos(base, jj, L)) * V + v0, kBV * 2,
                                           bar_vh);
                }
            }
            // q_eff (thread = key channel): eG_{W+s} q^_s - sum_j c[j][s] eG_j k^_j
            {
                const int kk = tid;
                const int katom = kk >> 5, kbyte = (kk & 31) * 4, kch = kbyte >> 4;
                const uint32_t xbase = kOffX + katom * kXAtom + (kbyte & 15);
                float acc[TM];
#pragma unroll
                for (int s = 0; s < TM; ++s) acc[s] = 0.0f;
#pragma unroll 4
                for (int j = 0; j < n; ++j) {
                    const float x = *reinterpret_cast<const float *>(sm + xbase + j * 128 + ((kch ^ (j & 7)) << 4));
#pragma unroll
                    for (int s = 0; s < TM; s += 4) {
                        const float4 c4 = *reinterpret_cast<const float4 *>(F + j * TM + s);
                        acc[s] = fmaf(-c4.x, x, acc[s]);
                        acc[s + 1] = fmaf(-c4.y, x, acc[s + 1]);
                        acc[s + 2] = fmaf(-c4.z, x, acc[s + 2]);
                        acc[s + 3] = fmaf(-c4.w, x, acc[s + 3]);
                    }
                }
#pragma unroll
                for (int s = 0; s < TM; ++s)
                    if (s < T)
                        acc[s] += eG[W + s] * *reinterpret_cast<const float *>(
                                                  sm + xbase + (kQRow + s) * 128 + ((kch ^ ((kQRow + s) & 7)) << 4));
#pragma unroll
                for (int s = 0; s < TM; ++s)
                    if (s < T) *reinterpret_cast<float *>(sm + kOffQ + sw128(kQAtom, s, kk)) = acc[s];
            }
        } else {
            if (tid == 0) fetch_unit(P, C, slot_idx, un, nunits, VB, misc);
            if (vrow < V)
                for (int s = 0; s < T; ++s)
                    out[(((size_t)bb * T + s) * HV + hv) * V + vrow] = __float2bfloat16_rn(0.0f);
        }

        // output part that does not need the checkpoint: sum_j c[j][s] v_j,
        // from the staged v history and the window values
        float vt[TM];
#pragma unroll
        for (int s = 0; s < TM; ++s) vt[s] = 0.0f;
        if (ok) {
            bool vh_ok = true;
            if (W > 0) {
                vh_ok = ptx::mbar_wait(bar_vh, ph_vh);
                ph_vh ^= 1u;
                if (!vh_ok) lost |= 2u;
            }
            if (vrow < V) {
#pragma unroll 4
                for (int j = 0; j < W; ++j) {
                    const float x = __bfloat162float(vh[j * kBV + tid]);
#pragma unroll
                    for (int s = 0; s < TM; s += 4) {
                        const float4 c4 = *reinterpret_cast<const float4 *>(sm + c_off(j) + 4 * s);
                        vt[s] = fmaf(c4.x, x, vt[s]);
                        vt[s + 1] = fmaf(c4.y, x, vt[s + 1]);
                        vt[s + 2] = fmaf(c4.z, x, vt[s + 2]);
                        vt[s + 3] = fmaf(c4.w, x, vt[s + 3]);
                    }
                }
#pragma unroll
                for (int s2 = 0; s2 < TM; ++s2) {
                    if (s2 < T) {
                        const float x = bf16_word_to_float(R.vwin[s2]);
#pragma unroll
                        for (int s = 0; s < TM; s += 4) {
                            const float4 c4 = *reinterpret_cast<const float4 *>(sm + c_off(W + s2) + 4 * s);
                            vt[s] = fmaf(c4.x, x, vt[s]);
                            vt[s + 1] = fmaf(c4.y, x, vt[s + 1]);
                            vt[s + 2] = fmaf(c4.z, x, vt[s + 2]);
                            vt[s + 3] = fmaf(c4.w, x, vt[s + 3]);
                        }
                    }
                }
            }
            if (!vh_ok && tid == 0) misc[5] = 1;
            ptx::fence_proxy_async_smem();
            if (tid == 32)   // fetch stage 3: checks, L2 prefetch, hand-over
                finish_fetch(P, C, un, nunits, VB, f_slot, f_wp, f_base, misc);
        }
        __syncthreads();   // next unit's cursors visible; R0 free for the checkpoint tile

        // ---- 6. checkpoint tile by TMA (over the dead key buffers); the next
        //         unit's loads go out while it is in flight; then P = S0 q_eff^T
        // (every thread fenced its generic shared-memory accesses before the
        // barrier above: no further proxy fence is needed before the TMA)
        if (ok && tid == 0) {
            ptx::mbar_expect_tx(bar_s0, kR0Bytes);
            const int32_t y = (int32_t)((sh_hv * V) + v0);
#pragma unroll
            for (int kb = 0; kb < 4; ++kb)
                ptx::tma_load_2d(sm_s + kOffS0 + kb * kS0Atom, &tmap_s0, bar_s0, kb * 32, y);
        }
        const UnitInfo nxt{misc[0], misc[1], misc[2], misc[3]};
        if (un < nunits) {
            const int hvn = un % HV, restn = un / HV;
            issue_unit_loads<TM>(P, nxt, restn / VB, hvn, restn % VB, tid, q, k, v, a, bgate, A_log,
                                 dt_bias, R);
        }
        if (ok) {
            waited = ptx::mbar_wait(bar_s0, ph_s0, tile_wait_limit);
            ph_s0 ^= 1u;
            if (!waited) lost |= 4u;
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
            const bool p_done = ptx::mbar_wait(bar_p, ph_p);
            ph_p ^= 1u;
            if (!p_done) lost |= 8u;
            waited = p_done && waited;
            ptx::tc_fence_after_sync();
            float pr[16];
            ptx::tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + kPCol, pr);
            ptx::tmem_ld_wait();
            if (!waited) misc[5] = 1;
            if (vrow < V) {
#pragma unroll
                for (int s = 0; s < TM; ++s)
                    if (s < T)
                        out[(((size_t)bb * T + s) * HV + hv) * V + vrow] =
                            __float2bfloat16_rn(P.scale * (pr[s] + vt[s]));
            }
        }
        cur = nxt;
        // the tile and TMEM columns are reused by the next unit
        ptx::tc_fence_before_sync();
        const int stop = __syncthreads_or(lost != 0);
        ptx::tc_fence_after_sync();
        if (stop) {
            // a wait ran out (the status bit is set below): give every copy or
            // MMA this thread saw unfinished one more bounded wait, so that
            // none still writes this CTA's shared memory or TMEM, and leave
            if (tid == 0) misc[5] = 1;
            if (lost & 1u) ptx::mbar_wait(bar_gram, ph_gram ^ 1u);
            if (lost & 2u) ptx::mbar_wait(bar_vh, ph_vh ^ 1u);
            if (lost & 4u) ptx::mbar_wait(bar_s0, ph_s0 ^ 1u);
            if (lost & 8u) ptx::mbar_wait(bar_p, ph_p ^ 1u);
            break;
        }
    }

    // ---- teardown (also after a wait ran out): every TMEM read is
    //      complete; free the columns
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
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// Per-device launch set-up, done once per device and kernel instance: the
// shared-memory attributes and the grid size.  The grid comes from the
// resources themselves (shared memory with the per-CTA reserve, and
// kCtasPerSm): the runtime's occupancy query answers 1 for this kernel
// whatever the sizes, yet the SM holds three of its CTAs (measured: all
// 3 x SMs CTAs of one launch start within a few microseconds), and one per SM
// would leave two thirds of the machine idle.
constexpr int kMaxDevices = 64;
struct DeviceSetup {
    bool done[2];
    int grid_cap;
};
DeviceSetup g_setup[kMaxDevices];
std::mutex g_setup_mu;

template <int TM>
cudaError_t device_setup(int dev, int slot_tm, int *grid_cap) {
    std::lock_guard<std::mutex> lk(g_setup_mu);
    DeviceSetup &d = g_setup[dev];
    if (!d.done[slot_tm]) {
        auto kern = tc::verify_tc_kernel<TM>;
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             tc::kSmemBytes);
        if (e != cudaSuccess) return e;
        // all of the unified L1 / shared storage as shared memory
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
        int per_sm = smem_sm / (tc::kSmemBytes + smem_rsv);
        if (per_sm > tc::kCtasPerSm) per_sm = tc::kCtasPerSm;
        if (per_sm < 1) per_sm = 1;
        d.grid_cap = sms * per_sm;
        d.done[slot_tm] = true;
    }
    *grid_cap = d.grid_cap;
    return cudaSuccess;
}

// The checkpoint as a 2-D tensor [num_slots * HV * V rows, K fp32], boxes of
// 32 x 128 (one 128-byte swizzle span by the CTA's 128 rows).  The map
// depends only on the checkpoint's address and row count, so the last few
// are kept.
constexpr int kMapCache = 16;
struct MapEntry {
    const float *ptr;
    uint64_t rows;
    int dev;
    CUtensorMap map;
};
MapEntry g_maps[kMapCache];
int g_maps_used = 0, g_maps_next = 0;
std::mutex g_maps_mu;

bool tensor_map(const LayerArgs &P, int dev, CUtensorMap *out) {
    const uint64_t rows = (uint64_t)P.num_slots * P.HV * P.V;
    std::lock_guard<std::mutex> lk(g_maps_mu);
    for (int i = 0; i < g_maps_used; ++i)
        if (g_maps[i].ptr == P.checkpoint && g_maps[i].rows == rows && g_maps[i].dev == dev) {
            *out = g_maps[i].map;
            return true;
        }
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    CUtensorMap tmap;
    const cuuint64_t gdim[2] = {(cuuint64_t)P.K, (cuuint64_t)rows};
    const cuuint64_t gstride[1] = {(cuuint64_t)P.K * sizeof(float)};
    const cuuint32_t box[2] = {32, (cuuint32_t)tc::kBV};
    const cuuint32_t estride[2] = {1, 1};
    CUresult r = enc(&tmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, P.checkpoint, gdim, gstride, box,
                     estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return false;
    MapEntry &e = g_maps[g_maps_next];
    e.ptr = P.checkpoint;
    e.rows = rows;
    e.dev = dev;
    e.map = tmap;
    g_maps_next = (g_maps_next + 1) % kMapCache;
    if (g_maps_used < kMapCache) ++g_maps_used;
    *out = tmap;
    return true;
}

template <int TM>
cudaError_t launch_tm(const CUtensorMap &tmap, int grid_cap, const LayerArgs &P, const CursorArgs &C,
                      const int32_t *slot_idx, int B, const void *q, const void *k, const void *v,
                      const void *a, const void *b, const float *A_log, const float *dt_bias,
                      void *out, cudaStream_t stream) {
    const int nunits = B * P.HV * (P.V / tc::kBV);
    const int grid = grid_cap < nunits ? grid_cap : nunits;
    tc::verify_tc_kernel<TM><<<grid, tc::kThreads, tc::kSmemBytes, stream>>>(
        tmap, P, C, slot_idx, nunits, static_cast<const __nv_bfloat16 *>(q),
        static_cast<const __nv_bfloat16 *>(k), static_cast<const __nv_bfloat16 *>(v),
        static_cast<const __nv_bfloat16 *>(a), static_cast<const __nv_bfloat16 *>(b), A_log, dt_bias,
        static_cast<__nv_bfloat16 *>(out), data_wait_limit());
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_verify_tc(const LayerArgs &P, const CursorArgs &C, const int32_t *slot_idx,
                             int B, const void *q, const void *k, const void *v, const void *a,
                             const void *b, const float *A_log, const float *dt_bias, void *out,
                             cudaStream_t stream) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    CUtensorMap tmap;
    if (!tensor_map(P, dev, &tmap)) return cudaErrorInvalidValue;
    int grid_cap = 0;
    if (P.T <= 4) {
        if ((e = device_setup<4>(dev, 0, &grid_cap)) != cudaSuccess) return e;
        return launch_tm<4>(tmap, grid_cap, P, C, slot_idx, B, q, k, v, a, b, A_log, dt_bias, out, stream);
    }
    if ((e = device_setup<8>(dev, 1, &grid_cap)) != cudaSuccess) return e;
    return launch_tm<8>(tmap, grid_cap, P, C, slot_idx, B, q, k, v, a, b, A_log, dt_bias, out, stream);
}

}  // namespace gdnspec
