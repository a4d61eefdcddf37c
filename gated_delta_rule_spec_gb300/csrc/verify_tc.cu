// verify_tc.cu -- verify kernel for the Qwen3-Next-shaped GDN layer on
// sm_103a: TMA + tcgen05 (5th-generation tensor cores, TMEM accumulators).
//
// Shapes: bf16 I/O, scalar (GDN) gate, K = 128, V a multiple of 128, ring
// L <= 64, window T <= 8.  One CTA of 128 threads per unit; no layer axis
// (layers are chain-dependent inside the forward; blog post on sglang PR
// #28695, §1.2).  A unit is (batch row, 128 state rows, NH v-heads of one
// q/k head): with an even number G of v-heads per q/k head and T <= 4, the two
// v-heads of a pair share one unit (NH = 2), so their common work -- the key
// and query rows, their norms and the Gram matrix -- is done once; otherwise
// NH = 1.
//
// The math is the chunked UT transform applied from the output side (see
// verify_generic.cu for the derivation):
//   Gram       G = X X^T over the n = W + T raw keys (rows 0..n-1 of X) and
//              the T raw window queries (rows 64..64+T-1), K = 128
//              contraction -> tcgen05.mma kind::f16 on the bf16 inputs as
//              they are, fp32 accumulator in TMEM; the L2 norms enter as
//              factors 1/|x_i| 1/|x_r| afterwards (exact bf16 products, fp32
//              sums)
//   per row i  A[i, r] = beta_i Gamma(i, r) G^[i, r], F[i, s] = Gamma(W+s, i) G^[i, 64+s]
//              (one thread per token and both heads; decays are products of
//              alpha, never exponentials of differences of long sums)
//   M          M (I + A) = F^T, backward substitution, one warp per window
//              token, both heads interleaved
//   q_eff_s    eG_{W+s} q^_s - sum_j M[s, j] beta_j eG_j k^_j       (K-vector)
//   P          P = S0 q_eff^T: the checkpoint tile times 16 columns (the
//              q_eff of both heads) -> tcgen05.mma kind::tf32 with S0 staged
//              by TMA, one head's tile after the other
//   o_s        scale * (P[:, s] + sum_j M[s, j] beta_j v_j)
// The Gram and the checkpoint product are the two dense contractions of the
// path; everything else is O(n) per thread or O(n^2) per CTA on CUDA cores.
//
// Data movement: each head's checkpoint tile (128 x 128 fp32 = 64 KiB) is the
// bulk of the bytes; it is read once, by a TMA load into shared memory issued
// after the key buffers are dead, so a tile reuses their space and the CTA
// needs ~73 KiB of shared memory: three CTAs per SM, which between them hide
// the loads' DRAM latency.  The ring's v history is prefetched into L2 at the
// start of the unit; every other global read of the unit (keys, queries,
// gates, window values) is issued in one round at the end of the previous
// unit.
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
constexpr int kXAtom = kXRows * 128;   // bytes of one 64-element (bf16) K slice of X
constexpr int kS0Atom = kBV * 128;     // bytes of one 32-float K slice of S0
constexpr int kQAtom = 16 * 128;       // bytes of one 32-float K slice of q_eff (N = 16)
constexpr int kALd = kLMax + 4;        // row stride (floats) of A: 16-byte rows, conflict-free
constexpr int kR0Bytes = 4 * kS0Atom;  // 65536: key phase, then the checkpoint tile

// Shared-memory map (bytes from a 1024-aligned base).  R0 holds first the key
// phase (X, per head A, F, c and the gate tables, the norms), then one head's
// checkpoint tile at a time.  After R0: the q_eff operand of the output MMA
// (16 rows of 128 fp32: head hh in rows 8 hh .. 8 hh + T - 1), the barriers
// and a few words.
template <int TM, int NH>
struct Lay {
    static constexpr int X = 0;
    static constexpr int A = 2 * kXAtom;                            // [NH][64][kALd]
    static constexpr int F = A + NH * kLMax * kALd * 4;             // [NH][64][TM]: F, then c eG / |k|
    static constexpr int Cc = F + NH * kLMax * TM * 4;              // [NH][64][TM]: c = M beta
    static constexpr int Alpha = Cc + NH * kLMax * TM * 4;          // [NH][64]
    static constexpr int Beta = Alpha + NH * kLMax * 4;             // [NH][64]
    static constexpr int EG = Beta + NH * kLMax * 4;                // [NH][64]
    static constexpr int Suf = EG + NH * kLMax * 4;                 // [NH][kLMax + 4]
    static constexpr int WP = Suf + NH * (kLMax + 4) * 4;           // [NH][kTMax]
    static constexpr int Rn = WP + NH * kTMax * 4;                  // [kXRows] 1 / |row of X|
    static constexpr int End = Rn + kXRows * 4;
    static_assert(End <= kR0Bytes, "key phase must fit under the checkpoint tile");
    // the Gram's A operand reads 128 rows of each X slice; slice 1 runs 48 rows
    // past X into the A matrices, which are inside R0
    static_assert(kXAtom + 128 * 128 <= kR0Bytes, "Gram operand overrun leaves R0");
    // each head's v history (up to 64 records of 128 bf16) is staged over its
    // dead A matrix
    static_assert(kLMax * kBV * 2 <= kLMax * kALd * 4, "v history fits over A");
};
constexpr int kOffQ = kR0Bytes;                               // q_eff operand, 8 KiB
constexpr int kOffBar = kOffQ + 4 * kQAtom;                   // 73728
constexpr int kOffMisc = kOffBar + 32;
constexpr int kSmemUsed = kOffMisc + 32;
constexpr int kSmemBytes = kSmemUsed + 1024;                  // + alignment slack
static_assert(3 * (kSmemBytes + 1024) <= 228 * 1024, "three CTAs per SM");

constexpr uint32_t kTmemCols = 128;
// CTAs per SM the kernel is built for: the register cap of the launch bounds
// (65536 / (3 * 128) = 170 per thread) and three TMEM allocations of 128 of
// the SM's 512 columns
constexpr int kCtasPerSm = 3;
static_assert(kCtasPerSm * kTmemCols <= 512, "TMEM columns of the resident CTAs");
constexpr uint32_t kGramCol = 0;
constexpr uint32_t kPCol = 96;   // head hh's product in columns 96 + 16 hh .. + 15

// byte offset of fp32 element (row, k) in a K-major SW128 tile of 128-byte rows
__device__ __forceinline__ uint32_t sw128(int atom_bytes, int row, int k) {
    const int atom = k >> 5, byte = (k & 31) * 4, chunk = byte >> 4;
    return atom * atom_bytes + row * 128 + (((chunk ^ (row & 7)) << 4) | (byte & 15));
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

__device__ __forceinline__ float bf16_word_to_float(uint32_t w) { return __uint_as_float(w << 16); }

// One unit = (batch row, block of 128 state rows, NH v-heads hv0 .. hv0 +
// NH - 1 of one q/k head).  Fetching a unit means reading its slot and cursors
// (one thread).  Inside the unit loop the fetch of the next unit is split into
// stages spread over the current unit, so that no stage waits on a load: the
// slot index, then the cursors, then the checks and the hand-over through
// shared memory.
struct UnitInfo {
    int slot, base, W, ok;
};

__device__ __forceinline__ void unit_coords(int u, int NP, int VB, int &bb, int &pr, int &vb) {
    pr = u % NP;
    const int rest = u / NP;
    vb = rest % VB;
    bb = rest / VB;
}

// L2 prefetch of a unit's v histories (one or two contiguous ring segments
// per head when whole records are contiguous, V = 128).  The checkpoint tiles
// are not prefetched: measured on the Qwen3-Next-shaped layer at B = 128, a
// tile prefetched one unit (or half a unit) ahead of its TMA load was often
// evicted from L2 before the load and read from DRAM twice (DRAM bytes 1.56x /
// 1.10x of the algorithmic bytes against 1.00x without it, and the launch 20%
// / 6% slower); the three resident CTAs hide the load's DRAM latency.
template <int NH>
__device__ __forceinline__ void prefetch_vhist(const LayerArgs &P, int slot, int cbase, int wp, int pr) {
    if (P.V != kBV) return;
#pragma unroll
    for (int hh = 0; hh < NH; ++hh) {
        const size_t sh_hv = (size_t)slot * P.HV + pr * NH + hh;
        const __nv_bfloat16 *rv = reinterpret_cast<const __nv_bfloat16 *>(P.rawv) + sh_hv * P.L * P.V;
        const int first = (P.L - cbase) < wp ? (P.L - cbase) : wp;
        if (first > 0) ptx::prefetch_l2(rv + (size_t)cbase * P.V, first * P.V * 2);
        if (wp > first) ptx::prefetch_l2(rv, (wp - first) * P.V * 2);
    }
}

// Last stage: checks (status bits as row_cursor_ok sets them), hand-over to
// dst[0..3].  wp and cbase are only read when the slot is in range.
template <int NH>
__device__ __forceinline__ void finish_fetch(const LayerArgs &P, const CursorArgs &C, int u,
                                             int nunits, int VB, int slot, int wp, int cbase,
                                             int *dst) {
    if (u >= nunits) {
        dst[0] = -1; dst[1] = 0; dst[2] = 0; dst[3] = 0;
        return;
    }
    int bb, pr, vb;
    unit_coords(u, P.HV / NH, VB, bb, pr, vb);
    uint32_t st = 0;
    bool ok = false;
    if (slot >= C.num_slots) st = GDN_SPEC_ST_SLOT_OOR;
    else if (slot >= 0) {
        if (wp < 0 || wp > P.L || cbase < 0 || cbase >= P.L) st = GDN_SPEC_ST_CURSOR_CORRUPT;
        else if (wp + P.T > P.L) st = GDN_SPEC_ST_RING_OVERFLOW;
        else ok = true;
    }
    if (st && vb == 0 && pr == 0) atomicOr(C.status, st);
    dst[0] = slot; dst[1] = ok ? cbase : 0; dst[2] = ok ? wp : 0; dst[3] = ok ? 1 : 0;
}

// All stages at once (start-up, and units that have no work to hide it behind).
template <int NH>
__device__ __forceinline__ void fetch_unit(const LayerArgs &P, const CursorArgs &C,
                                           const int32_t *slot_idx, int u, int nunits, int VB,
                                           int *dst) {
    int slot = -1, wp = 0, cbase = 0;
    if (u < nunits) {
        int bb, pr, vb;
        unit_coords(u, P.HV / NH, VB, bb, pr, vb);
        slot = slot_idx[bb];
        if (slot >= 0 && slot < C.num_slots) {
            wp = C.write_pos[slot];
            cbase = C.cache_base[slot];
        }
    }
    finish_fetch<NH>(P, C, u, nunits, VB, slot, wp, cbase, dst);
}

// The early global reads of a unit, held in registers until its first phase:
// two threads per token row (keys 0..n-1 then the T queries; 128 bytes each),
// the gate inputs of one (head, token) per thread and the window values of
// state row tid for every head.
template <int TM, int NH>
struct UnitLoads {
    uint4 raw[8];
    // raw 32-bit words, converted only when the unit uses them: the ring's
    // fp32 gates, or the window's bf16 gate inputs and values zero-extended
    uint32_t g_in, b_in;
    float alog, dtb;
    uint32_t vwin[NH][TM];
};

// (head, token) whose gate thread tid computes: with two heads, threads
// 0..63 take head 0 and 64..127 head 1 (n <= 64)
template <int NH>
__device__ __forceinline__ void gate_slot(int tid, int &hh, int &tok) {
    hh = NH == 2 ? (tid >> 6) : 0;
    tok = NH == 2 ? (tid & 63) : tid;
}

template <int TM, int NH>
__device__ __forceinline__ void issue_unit_loads(
    const LayerArgs &P, const UnitInfo &U, int bb, int hv0, int vb, int tid,
    const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k,
    const __nv_bfloat16 *__restrict__ v, const __nv_bfloat16 *__restrict__ a,
    const __nv_bfloat16 *__restrict__ bgate, const float *__restrict__ A_log,
    const float *__restrict__ dt_bias, UnitLoads<TM, NH> &R) {
    const int T = P.T, L = P.L, HV = P.HV, H = P.H, V = P.V;
    const int h = hv0 / P.G, W = U.W, n = W + T, base = U.base;
    const size_t sh_h = (size_t)U.slot * H + h;
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
    int hh, tok;
    gate_slot<NH>(tid, hh, tok);
    const int hv = hv0 + hh;
    const size_t sh_hv = (size_t)U.slot * HV + hv;
    R.g_in = R.b_in = 0u;
    R.alog = R.dtb = 0.0f;
    if (U.ok && tok < W) {
        const int pj = ring_pos(base, tok, L);
        R.g_in = reinterpret_cast<const uint32_t *>(P.ring_g)[sh_hv * L + pj];
        R.b_in = reinterpret_cast<const uint32_t *>(P.ring_beta)[sh_hv * L + pj];
    } else if (U.ok && tok < n) {
        const size_t tk = (size_t)bb * T + (tok - W);
        R.g_in = reinterpret_cast<const unsigned short *>(a)[tk * HV + hv];
        R.b_in = reinterpret_cast<const unsigned short *>(bgate)[tk * HV + hv];
        R.alog = A_log[hv];
        R.dtb = dt_bias[hv];
    }
    const int vrow = vb * kBV + tid;
#pragma unroll
    for (int h2 = 0; h2 < NH; ++h2)
#pragma unroll
        for (int s = 0; s < TM; ++s) R.vwin[h2][s] = 0u;
    if (U.ok && vrow < V) {
#pragma unroll
        for (int h2 = 0; h2 < NH; ++h2)
#pragma unroll
            for (int s = 0; s < TM; ++s)
                if (s < T)
                    R.vwin[h2][s] = reinterpret_cast<const unsigned short *>(
                        v)[(((size_t)bb * T + s) * HV + hv0 + h2) * V + vrow];
    }
}

// Persistent: each CTA takes units blockIdx.x, blockIdx.x + gridDim.x, ...
// While a unit waits for its checkpoint tiles and output MMAs, the CTA already
// reads the next unit's cursors and issues that unit's key/gate/value loads.
template <int TM, int NH>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
verify_tc_kernel(const __grid_constant__ CUtensorMap tmap_s0, LayerArgs P, CursorArgs C,
                 const int32_t *__restrict__ slot_idx, int nunits,
                 const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k,
                 const __nv_bfloat16 *__restrict__ v, const __nv_bfloat16 *__restrict__ a,
                 const __nv_bfloat16 *__restrict__ bgate, const float *__restrict__ A_log,
                 const float *__restrict__ dt_bias, __nv_bfloat16 *__restrict__ out,
                 uint32_t tile_wait_limit) {
    using LY = Lay<TM, NH>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = ptx::smem_addr(smem_raw);
    const uint32_t pad = (1024u - (raw_s & 1023u)) & 1023u;
    uint8_t *sm = smem_raw + pad;
    const uint32_t sm_s = raw_s + pad;
    float *const Am = reinterpret_cast<float *>(sm + LY::A);       // [NH][64][kALd]
    float *const Fm = reinterpret_cast<float *>(sm + LY::F);       // [NH][64][TM]
    float *const Cm = reinterpret_cast<float *>(sm + LY::Cc);      // [NH][64][TM]
    float *const alpha = reinterpret_cast<float *>(sm + LY::Alpha);
    float *const betaS = reinterpret_cast<float *>(sm + LY::Beta);
    float *const eG = reinterpret_cast<float *>(sm + LY::EG);
    float *const suf = reinterpret_cast<float *>(sm + LY::Suf);
    float *const wprod = reinterpret_cast<float *>(sm + LY::WP);
    float *const rn = reinterpret_cast<float *>(sm + LY::Rn);
    int *misc = reinterpret_cast<int *>(sm + kOffMisc);  // [0..3] next unit, [4] tmem, [5] err
    const uint32_t bar_gram = sm_s + kOffBar, bar_s0 = sm_s + kOffBar + 8,
                   bar_p = sm_s + kOffBar + 16, bar_vh = sm_s + kOffBar + 24;

    const int T = P.T, L = P.L, HV = P.HV, H = P.H, V = P.V;
    const int VB = V / kBV, NP = HV / NH;
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
        fetch_unit<NH>(P, C, slot_idx, blockIdx.x, nunits, VB, misc);
    }
    if (warp == 0) ptx::tmem_alloc(sm_s + kOffMisc + 16, kTmemCols);
    // zero the q_eff operand: the rows of window positions >= T stay zero
    for (int i = tid; i < 4 * kQAtom / 16; i += kThreads)
        reinterpret_cast<float4 *>(sm + kOffQ)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    const uint32_t tmem = static_cast<uint32_t>(misc[4]);
    uint32_t ph_gram = 0, ph_s0 = 0, ph_p = 0, ph_vh = 0;   // mbarrier phase bits

    UnitInfo cur{misc[0], misc[1], misc[2], misc[3]};
    UnitLoads<TM, NH> R;
    int u = blockIdx.x;
    if (u < nunits) {
        int bb0, pr0, vb0;
        unit_coords(u, NP, VB, bb0, pr0, vb0);
        issue_unit_loads<TM, NH>(P, cur, bb0, pr0 * NH, vb0, tid, q, k, v, a, bgate, A_log, dt_bias, R);
    }

    for (; u < nunits; u += gridDim.x) {
        int bb, pr, vb;
        unit_coords(u, NP, VB, bb, pr, vb);
        const int hv0 = pr * NH;
        const int un = u + gridDim.x;
        const int h = hv0 / P.G;
        const int v0 = vb * kBV, vrow = v0 + tid;
        const int slot = cur.slot, base = cur.base, W = cur.W;
        const bool ok = cur.ok != 0;
        const int n = W + T;
        const size_t sh_h = (size_t)slot * H + h;
        const bool k_writer = (hv0 % P.G == 0) && vb == 0;
        // waits of this unit that ran out (bit per barrier: Gram, v history,
        // checkpoint tile, output MMA); after one, the unit's remaining copies
        // and MMAs are not issued, and the CTA drains and leaves
        uint32_t lost = 0;
        int f_slot = -1, f_wp = 0, f_base = 0;   // the next unit's fetch (thread 32)
        if (ok && tid == 32 && un < nunits) {     // fetch stage 1: the slot index
            int bbn, prn, vbn;
            unit_coords(un, NP, VB, bbn, prn, vbn);
            f_slot = slot_idx[bbn];
        }
        if (ok && tid == 64) prefetch_vhist<NH>(P, slot, base, W, pr);   // used in phase 5
        float vt[NH][TM];
#pragma unroll
        for (int hh = 0; hh < NH; ++hh)
#pragma unroll
            for (int s = 0; s < TM; ++s) vt[hh][s] = 0.0f;

        if (ok) {
            // ---- 1. raw key and query rows into X (bf16, SW128 K-major: half
            //         `half` of a row is K slice `half`), their norms; gates;
            //         ring side channel of the window
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
                    const int row = t < n ? t : kQRow + (t - n);
                    if (half == 0) rn[row] = 1.0f / sqrtf(sq + P.l2_eps);
                    uint8_t *xr = sm + LY::X + half * kXAtom + row * 128;
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        *reinterpret_cast<uint4 *>(xr + ((c ^ (row & 7)) << 4)) = R.raw[c];
                    if (t >= W && t < n && k_writer) {  // side channel: raw key, bitwise
                        uint4 *dst = reinterpret_cast<uint4 *>(rawk_w + (sh_h * L + ring_pos(base, t, L)) * kK);
#pragma unroll
                        for (int c = 0; c < 8; ++c) dst[8 * half + c] = R.raw[c];
                    }
                }
            }
            {
                int hh, tok;
                gate_slot<NH>(tid, hh, tok);
                if (tok < n) {
                    const size_t sh_hv = (size_t)slot * HV + hv0 + hh;
                    const int pj = ring_pos(base, tok, L);
                    float g = __uint_as_float(R.g_in), be = __uint_as_float(R.b_in);
                    if (tok >= W) {
                        g = gate_g(R.alog, bf16_word_to_float(R.g_in), R.dtb);
                        be = gate_beta(bf16_word_to_float(R.b_in));
                        if (vb == 0) {
                            P.ring_g[sh_hv * L + pj] = g;
                            P.ring_beta[sh_hv * L + pj] = be;
                        }
                    }
                    alpha[hh * kLMax + tok] = expf(g);
                    betaS[hh * kLMax + tok] = be;
                }
            }
#pragma unroll
            for (int hh = 0; hh < NH; ++hh) {
                const size_t sh_hv = (size_t)slot * HV + hv0 + hh;
#pragma unroll
                for (int s = 0; s < TM; ++s)
                    if (s < T && vrow < V) rawv_w[(sh_hv * L + ring_pos(base, W + s, L)) * V + vrow] =
                            __ushort_as_bfloat16((unsigned short)R.vwin[hh][s]);
            }
            ptx::fence_proxy_async_smem();
            __syncthreads();

            // ---- 2. Gram on the tensor core (D[i, j] = <x_i, x_j> of the raw
            //         rows, M = 128, N = 80), decay products on CUDA cores meanwhile
            if (tid == 0) {
                ptx::tc_fence_after_sync();
                constexpr uint32_t idesc = ptx::idesc_bf16(128, kXRows);
#pragma unroll
                for (int kb = 0; kb < 2; ++kb)
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks) {
                        const uint64_t d = ptx::smem_desc_sw128(sm_s + LY::X + kb * kXAtom + ks * 32);
                        ptx::mma_bf16(tmem + kGramCol, d, d, idesc, (kb | ks) != 0);
                    }
                ptx::mma_commit(bar_gram);
            }
            if (warp == 1) {  // eG_j = prod_{t <= j} alpha_t, j < n, per head
#pragma unroll
                for (int hh = 0; hh < NH; ++hh) {
                    const float *al = alpha + hh * kLMax;
                    const float a0 = 2 * lane < n ? al[2 * lane] : 1.0f;
                    const float a1 = 2 * lane + 1 < n ? al[2 * lane + 1] : 1.0f;
                    const float incl = warp_prefix_prod(a0 * a1, lane);
                    float excl = __shfl_up_sync(0xffffffffu, incl, 1);
                    if (lane == 0) excl = 1.0f;
                    eG[hh * kLMax + 2 * lane] = excl * a0;
                    eG[hh * kLMax + 2 * lane + 1] = incl;
                }
            } else if (warp == 2) {  // suf[t] = prod_{u=t}^{W-1} alpha_u, t <= W (suf[W] = 1)
#pragma unroll
                for (int hh = 0; hh < NH; ++hh) {
                    const float *al = alpha + hh * kLMax;
                    float *sf = suf + hh * (kLMax + 4);
                    const int u0 = 2 * lane, u1 = 2 * lane + 1;  // reversed index u = W-1-t
                    const float a0 = u0 < W ? al[W - 1 - u0] : 1.0f;
                    const float a1 = u1 < W ? al[W - 1 - u1] : 1.0f;
                    const float incl = warp_prefix_prod(a0 * a1, lane);
                    float excl = __shfl_up_sync(0xffffffffu, incl, 1);
                    if (lane == 0) excl = 1.0f;
                    if (u0 < W) sf[W - 1 - u0] = excl * a0;
                    if (u1 < W) sf[W - 1 - u1] = incl;
                    if (lane == 0) sf[W] = 1.0f;
                }
            } else if (warp == 3 && lane < NH) {  // wprod[s] = prod_{t=W}^{W+s} alpha_t
                const float *al = alpha + lane * kLMax;
                float c = 1.0f;
#pragma unroll
                for (int s = 0; s < TM; ++s)
                    if (s < T) {
                        c *= al[W + s];
                        wprod[lane * kTMax + s] = c;
                    }
            }
            __syncthreads();
            if (!ptx::mbar_wait(bar_gram, ph_gram)) lost |= 1u;
            ph_gram ^= 1u;
            ptx::tc_fence_after_sync();
            if (tid == 32 && f_slot >= 0 && f_slot < C.num_slots) {  // fetch stage 2: cursors
                f_wp = C.write_pos[f_slot];
                f_base = C.cache_base[f_slot];
            }

            // ---- 3. per token i (thread i), both heads: row i of A (zero above
            //         the diagonal), row i of F.  G^[i, r] = G[i, r] / |x_i| / |x_r|.
            if (warp * 32 < n) {   // (warp-uniform) a warp with a live token row
                const int i = tid;
                const uint32_t tbase = tmem + ((uint32_t)(warp * 32) << 16) + kGramCol;
                // tcgen05.ld is warp-collective: every load below runs on all lanes
                float gq[16];
                ptx::tmem_ld16(tbase + kQRow, gq);   // columns 64..79: the query columns
                ptx::tmem_ld_wait();
                const bool row_live = i < n;
                const float rni = row_live ? rn[i] : 0.0f;
                float bi[NH], c[NH];
#pragma unroll
                for (int hh = 0; hh < NH; ++hh) {
                    bi[hh] = row_live ? betaS[hh * kLMax + i] * rni : 0.0f;
                    c[hh] = 1.0f;
                }
#pragma unroll 1
                // key columns below n (the bound is the same in every thread),
                // high chunk first
                for (int cc = (n + 15) / 16 - 1; cc >= 0; --cc) {
                    float gk[16];
                    ptx::tmem_ld16(tbase + 16 * cc, gk);
                    ptx::tmem_ld_wait();
                    if (row_live) {
                        float val[NH][16];
#pragma unroll
                        for (int x = 15; x >= 0; --x) {
                            const int r = 16 * cc + x;
                            const float g = gk[x] * rn[r];
#pragma unroll
                            for (int hh = 0; hh < NH; ++hh) {
                                val[hh][x] = 0.0f;
                                if (r < i) {
                                    c[hh] *= alpha[hh * kLMax + r + 1];    // Gamma(i, r)
                                    val[hh][x] = bi[hh] * c[hh] * g;
                                }
                            }
                        }
#pragma unroll
                        for (int hh = 0; hh < NH; ++hh)
#pragma unroll
                            for (int x = 0; x < 16; x += 4)
                                *reinterpret_cast<float4 *>(Am + (hh * kLMax + i) * kALd + 16 * cc + x) =
                                    make_float4(val[hh][x], val[hh][x + 1], val[hh][x + 2], val[hh][x + 3]);
                    }
                }
                if (row_live) {
#pragma unroll
                    for (int hh = 0; hh < NH; ++hh) {
                        // Gamma(W+s, i): products of the suffix and window decays
                        const float si = i < W ? suf[hh * (kLMax + 4) + i + 1] : 1.0f;
                        float cw = 1.0f;
                        float fr[TM];
#pragma unroll
                        for (int s = 0; s < TM; ++s) {
                            float f = 0.0f;
                            if (s < T) {
                                const int t = W + s;
                                const float gqs = gq[s] * rni * rn[kQRow + s];
                                if (i < W) {
                                    f = si * wprod[hh * kTMax + s] * gqs;
                                } else if (t >= i) {
                                    if (t > i) cw *= alpha[hh * kLMax + t];
                                    f = cw * gqs;
                                }
                            }
                            fr[s] = f;
                        }
#pragma unroll
                        for (int s = 0; s < TM; s += 4)
                            *reinterpret_cast<float4 *>(Fm + (hh * kLMax + i) * TM + s) =
                                make_float4(fr[s], fr[s + 1], fr[s + 2], fr[s + 3]);
                    }
                }
            }
            __syncthreads();

            // ---- 4. M (I + A) = F^T per head: the T right-hand sides are
            //         independent systems, s in warp s % 4, both heads in the
            //         same steps; lane l ends with M[s][l], M[s][l+32]
            {
                constexpr int SPW = (TM + 3) / 4;   // right-hand sides per warp and head
                float f0[NH][SPW], f1[NH][SPW];
#pragma unroll
                for (int hh = 0; hh < NH; ++hh)
#pragma unroll
                    for (int qq = 0; qq < SPW; ++qq) {
                        const int sq = warp + 4 * qq;
                        const float *Fh = Fm + hh * kLMax * TM;
                        f0[hh][qq] = (sq < T && lane < n) ? Fh[lane * TM + sq] : 0.0f;
                        f1[hh][qq] = (sq < T && lane + 32 < n) ? Fh[(lane + 32) * TM + sq] : 0.0f;
                    }
                // four tokens j-3..j per step: the 4 x 4 diagonal block is solved
                // redundantly on every lane, then all lanes apply the four updates
                // (which also leave f[j-3..j] equal to their final values)
                int j = n - 1;
                for (; j >= 3; j -= 4) {
#pragma unroll
                    for (int hh = 0; hh < NH; ++hh) {
                        const float *Ah = Am + hh * kLMax * kALd;
                        float ar[4][2], d[6];
#pragma unroll
                        for (int qq = 0; qq < 4; ++qq) {
                            ar[qq][0] = Ah[(j - qq) * kALd + lane];
                            ar[qq][1] = Ah[(j - qq) * kALd + 32 + lane];
                        }
                        d[0] = Ah[j * kALd + j - 1];        // A[j][j-1]
                        d[1] = Ah[j * kALd + j - 2];        // A[j][j-2]
                        d[2] = Ah[j * kALd + j - 3];        // A[j][j-3]
                        d[3] = Ah[(j - 1) * kALd + j - 2];  // A[j-1][j-2]
                        d[4] = Ah[(j - 1) * kALd + j - 3];  // A[j-1][j-3]
                        d[5] = Ah[(j - 2) * kALd + j - 3];  // A[j-2][j-3]
#pragma unroll
                        for (int qq = 0; qq < SPW; ++qq) {
                            float fj[4];
#pragma unroll
                            for (int x = 0; x < 4; ++x)
                                fj[x] = __shfl_sync(0xffffffffu, (j - x) < 32 ? f0[hh][qq] : f1[hh][qq], (j - x) & 31);
                            const float m0 = fj[0];
                            const float m1 = fmaf(-d[0], m0, fj[1]);
                            const float m2 = fmaf(-d[3], m1, fmaf(-d[1], m0, fj[2]));
                            const float m3 = fmaf(-d[5], m2, fmaf(-d[4], m1, fmaf(-d[2], m0, fj[3])));
                            f0[hh][qq] = fmaf(-ar[3][0], m3, fmaf(-ar[2][0], m2, fmaf(-ar[1][0], m1, fmaf(-ar[0][0], m0, f0[hh][qq]))));
                            f1[hh][qq] = fmaf(-ar[3][1], m3, fmaf(-ar[2][1], m2, fmaf(-ar[1][1], m1, fmaf(-ar[0][1], m0, f1[hh][qq]))));
                        }
                    }
                }
                for (; j >= 0; --j) {
#pragma unroll
                    for (int hh = 0; hh < NH; ++hh) {
                        const float *Ah = Am + hh * kLMax * kALd;
                        const float a0 = Ah[j * kALd + lane], a1 = Ah[j * kALd + 32 + lane];
#pragma unroll
                        for (int qq = 0; qq < SPW; ++qq) {
                            const float m = __shfl_sync(0xffffffffu, j < 32 ? f0[hh][qq] : f1[hh][qq], j & 31);
                            f0[hh][qq] = fmaf(-a0, m, f0[hh][qq]);
                            f1[hh][qq] = fmaf(-a1, m, f1[hh][qq]);
                        }
                    }
                }
                // c = M beta (the V-term) and c eG / |k_j| (the effective query),
                // rows j = lane, lane + 32
#pragma unroll
                for (int hlf = 0; hlf < 2; ++hlf) {
                    const int jj = lane + 32 * hlf;
                    const float rj = jj < n ? rn[jj] : 0.0f;
#pragma unroll
                    for (int hh = 0; hh < NH; ++hh) {
                        const float bj = jj < n ? betaS[hh * kLMax + jj] : 0.0f;
                        const float ej = jj < n ? eG[hh * kLMax + jj] : 0.0f;
#pragma unroll
                        for (int qq = 0; qq < SPW; ++qq) {
                            const int sq = warp + 4 * qq;
                            if (sq < TM) {
                                const float cj = (hlf ? f1[hh][qq] : f0[hh][qq]) * bj;
                                Cm[(hh * kLMax + jj) * TM + sq] = cj;
                                Fm[(hh * kLMax + jj) * TM + sq] = cj * ej * rj;
                            }
                        }
                    }
                }
            }
            __syncthreads();

            // ---- 5. each head's v history of this CTA's rows into its (now
            //         dead) A matrix by 1-D bulk copies: with V = 128 whole
            //         records are contiguous, so a history is one or two ring
            //         segments; otherwise one copy per record, spread over warp 0
            if (warp == 0 && W > 0) {
                ptx::fence_proxy_async_smem();   // the A matrices were last read by generic loads
                if (lane == 0) ptx::mbar_expect_tx(bar_vh, (uint32_t)(NH * W * kBV * 2));
                __syncwarp();
#pragma unroll
                for (int hh = 0; hh < NH; ++hh) {
                    const size_t sh_hv = (size_t)slot * HV + hv0 + hh;
                    const uint32_t dst = sm_s + LY::A + hh * kLMax * kALd * 4;
                    if (V == kBV) {
                        if (lane == 0) {
                            const int n1 = (L - base) < W ? (L - base) : W;
                            ptx::bulk_copy_g2s(dst, rawv + (sh_hv * L + base) * V, n1 * kBV * 2, bar_vh);
                            if (W > n1)
                                ptx::bulk_copy_g2s(dst + n1 * kBV * 2, rawv + sh_hv * L * V,
                                                   (W - n1) * kBV * 2, bar_vh);
                        }
                    } else {
                        for (int jj = lane; jj < W; jj += 32)
                            ptx::bulk_copy_g2s(dst + jj * kBV * 2,
                                               rawv + (sh_hv * L + ring_pos(base, jj, L)) * V + v0, kBV * 2,
                                               bar_vh);
                    }
                }
            }
            // q_eff (thread = key channel), both heads:
            //   eG_{W+s} q_s / |q_s| - sum_j (c[j][s] eG_j / |k_j|) k_j
            {
                const int kk = tid;
                const uint32_t xbase = LY::X + (kk >> 6) * kXAtom + (kk & 7) * 2;
                const int kch = (kk & 63) >> 3;
                float2 a2[NH][TM / 2];
#pragma unroll
                for (int hh = 0; hh < NH; ++hh)
#pragma unroll
                    for (int s2 = 0; s2 < TM / 2; ++s2) a2[hh][s2] = make_float2(0.f, 0.f);
                auto step = [&](int j, int sw) {
                    const float x = -bf16_word_to_float(
                        *reinterpret_cast<const unsigned short *>(sm + xbase + j * 128 + ((kch ^ sw) << 4)));
                    const float2 x2 = make_float2(x, x);
#pragma unroll
                    for (int hh = 0; hh < NH; ++hh)
#pragma unroll
                        for (int s = 0; s < TM; s += 4) {
                            const float4 c4 = *reinterpret_cast<const float4 *>(Fm + (hh * kLMax + j) * TM + s);
                            a2[hh][s / 2] = __ffma2_rn(make_float2(c4.x, c4.y), x2, a2[hh][s / 2]);
                            a2[hh][s / 2 + 1] = __ffma2_rn(make_float2(c4.z, c4.w), x2, a2[hh][s / 2 + 1]);
                        }
                };
                int j = 0;
                for (; j + 8 <= n; j += 8) {   // (j & 7) is the step's lane in the swizzle
#pragma unroll
                    for (int x = 0; x < 8; ++x) step(j + x, x);
                }
                for (; j < n; ++j) step(j, j & 7);
#pragma unroll
                for (int s = 0; s < TM; ++s)
                    if (s < T) {
                        const int row = kQRow + s;
                        const float xq = bf16_word_to_float(*reinterpret_cast<const unsigned short *>(
                                             sm + xbase + row * 128 + ((kch ^ (row & 7)) << 4))) *
                                         rn[row];
#pragma unroll
                        for (int hh = 0; hh < NH; ++hh) {
                            const float accv = (s & 1) ? a2[hh][s / 2].y : a2[hh][s / 2].x;
                            const float qe = fmaf(eG[hh * kLMax + W + s], xq, accv);
                            *reinterpret_cast<float *>(sm + kOffQ + sw128(kQAtom, 8 * hh + s, kk)) = qe;
                        }
                    }
            }
            // the output part that does not need the checkpoint: sum_j c[j][s] v_j,
            // from the staged v histories and the window values
            if (W > 0) {
                if (!ptx::mbar_wait(bar_vh, ph_vh)) lost |= 2u;
                ph_vh ^= 1u;
            }
            if (vrow < V && !(lost & 2u)) {
#pragma unroll
                for (int hh = 0; hh < NH; ++hh) {
                    const __nv_bfloat16 *vh = reinterpret_cast<const __nv_bfloat16 *>(
                        sm + LY::A + hh * kLMax * kALd * 4);
                    const float *Ch = Cm + hh * kLMax * TM;
                    float2 p2[TM / 2];
#pragma unroll
                    for (int s2 = 0; s2 < TM / 2; ++s2) p2[s2] = make_float2(0.f, 0.f);
#pragma unroll 4
                    for (int jj = 0; jj < W; ++jj) {
                        const float x = __bfloat162float(vh[jj * kBV + tid]);
                        const float2 x2 = make_float2(x, x);
#pragma unroll
                        for (int s = 0; s < TM; s += 4) {
                            const float4 c4 = *reinterpret_cast<const float4 *>(Ch + jj * TM + s);
                            p2[s / 2] = __ffma2_rn(make_float2(c4.x, c4.y), x2, p2[s / 2]);
                            p2[s / 2 + 1] = __ffma2_rn(make_float2(c4.z, c4.w), x2, p2[s / 2 + 1]);
                        }
                    }
#pragma unroll
                    for (int s2 = 0; s2 < TM; ++s2) {
                        if (s2 < T) {
                            const float x = bf16_word_to_float(R.vwin[hh][s2]);
                            const float2 x2 = make_float2(x, x);
#pragma unroll
                            for (int s = 0; s < TM; s += 4) {
                                const float4 c4 = *reinterpret_cast<const float4 *>(Ch + (W + s2) * TM + s);
                                p2[s / 2] = __ffma2_rn(make_float2(c4.x, c4.y), x2, p2[s / 2]);
                                p2[s / 2 + 1] = __ffma2_rn(make_float2(c4.z, c4.w), x2, p2[s / 2 + 1]);
                            }
                        }
                    }
#pragma unroll
                    for (int s2 = 0; s2 < TM / 2; ++s2) {
                        vt[hh][2 * s2] = p2[s2].x;
                        vt[hh][2 * s2 + 1] = p2[s2].y;
                    }
                }
            }
            ptx::fence_proxy_async_smem();
            if (tid == 32)   // fetch stage 3: checks, hand-over
                finish_fetch<NH>(P, C, un, nunits, VB, f_slot, f_wp, f_base, misc);
        } else {
            if (tid == 0) fetch_unit<NH>(P, C, slot_idx, un, nunits, VB, misc);
            if (vrow < V)
#pragma unroll
                for (int hh = 0; hh < NH; ++hh)
                    for (int s = 0; s < T; ++s)
                        out[(((size_t)bb * T + s) * HV + hv0 + hh) * V + vrow] = __float2bfloat16_rn(0.0f);
        }
        // next unit's cursors visible; R0 free for the checkpoint tiles; every
        // thread agrees on whether a wait of this unit ran out
        int stop = __syncthreads_or(lost != 0);

        // ---- 6. each head's checkpoint tile by TMA (over the dead key
        //         buffers, one head after the other); the next unit's loads go
        //         out while the first is in flight; then P = S0 q_eff^T and the
        //         outputs.  (every thread fenced its generic shared-memory
        //         accesses before the barrier above: no further proxy fence is
        //         needed before the TMA)
        const bool tiles = ok && !stop;
        if (tiles && tid == 0) {
            ptx::mbar_expect_tx(bar_s0, kR0Bytes);
            const int32_t y = (int32_t)(((size_t)slot * HV + hv0) * V + v0);
#pragma unroll
            for (int kb = 0; kb < 4; ++kb)
                ptx::tma_load_2d(sm_s + kb * kS0Atom, &tmap_s0, bar_s0, kb * 32, y);
        }
        const UnitInfo nxt{misc[0], misc[1], misc[2], misc[3]};
        if (un < nunits) {
            int bbn, prn, vbn;
            unit_coords(un, NP, VB, bbn, prn, vbn);
            issue_unit_loads<TM, NH>(P, nxt, bbn, prn * NH, vbn, tid, q, k, v, a, bgate, A_log,
                                     dt_bias, R);
        }
        if (tiles) {
            // (kept rolled: one copy of the tile, MMA and output code serves both
            // heads, which keeps the body's instruction footprint smaller)
#pragma unroll 1
            for (int hh = 0; hh < NH; ++hh) {
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
                                ptx::mma_tf32(tmem + kPCol + 16 * hh,
                                              ptx::smem_desc_sw128(sm_s + kb * kS0Atom + ks * 32),
                                              ptx::smem_desc_sw128(sm_s + kOffQ + kb * kQAtom + ks * 32),
                                              idesc, (kb | ks) != 0);
                    }
                    ptx::mma_commit(bar_p);
                }
                if (!ptx::mbar_wait(bar_p, ph_p)) lost |= 8u;
                ph_p ^= 1u;
                ptx::tc_fence_after_sync();
                if (hh + 1 < NH) {
                    // the tile was consumed: the next head's tile may overwrite it
                    // (only if every thread saw this head's waits complete)
                    if (__syncthreads_or(lost != 0)) break;
                    if (tid == 0) {
                        ptx::mbar_expect_tx(bar_s0, kR0Bytes);
                        const int32_t y = (int32_t)(((size_t)slot * HV + hv0 + hh + 1) * V + v0);
#pragma unroll
                        for (int kb = 0; kb < 4; ++kb)
                            ptx::tma_load_2d(sm_s + kb * kS0Atom, &tmap_s0, bar_s0, kb * 32, y);
                    }
                }
                float pr8[8];
                ptx::tmem_ld8(tmem + ((uint32_t)(warp * 32) << 16) + kPCol + 16 * hh + 8 * hh, pr8);
                ptx::tmem_ld_wait();
                if (!lost && vrow < V) {
#pragma unroll
                    for (int s = 0; s < TM; ++s)
                        if (s < T)
                            out[(((size_t)bb * T + s) * HV + hv0 + hh) * V + vrow] =
                                __float2bfloat16_rn(P.scale * (pr8[s] + (NH > 1 && hh ? vt[NH - 1][s] : vt[0][s])));
                }
            }
        }
        cur = nxt;
        // the tile and TMEM columns are reused by the next unit
        ptx::tc_fence_before_sync();
        stop = __syncthreads_or(lost != 0);
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
constexpr int kInstances = 3;   // <4, 2>, <4, 1>, <8, 1>
struct DeviceSetup {
    bool done[kInstances];
    int grid_cap;
};
DeviceSetup g_setup[kMaxDevices];
std::mutex g_setup_mu;

template <int TM, int NH>
cudaError_t device_setup(int dev, int inst, int *grid_cap) {
    std::lock_guard<std::mutex> lk(g_setup_mu);
    DeviceSetup &d = g_setup[dev];
    if (!d.done[inst]) {
        auto kern = tc::verify_tc_kernel<TM, NH>;
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
        d.done[inst] = true;
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

template <int TM, int NH>
cudaError_t launch_tm(int dev, int inst, const CUtensorMap &tmap, const LayerArgs &P,
                      const CursorArgs &C, const int32_t *slot_idx, int B, const void *q,
                      const void *k, const void *v, const void *a, const void *b,
                      const float *A_log, const float *dt_bias, void *out, cudaStream_t stream) {
    int grid_cap = 0;
    cudaError_t e = device_setup<TM, NH>(dev, inst, &grid_cap);
    if (e != cudaSuccess) return e;
    const int nunits = B * (P.HV / NH) * (P.V / tc::kBV);
    const int grid = grid_cap < nunits ? grid_cap : nunits;
    tc::verify_tc_kernel<TM, NH><<<grid, tc::kThreads, tc::kSmemBytes, stream>>>(
        tmap, P, C, slot_idx, nunits, static_cast<const __nv_bfloat16 *>(q),
        static_cast<const __nv_bfloat16 *>(k), static_cast<const __nv_bfloat16 *>(v),
        static_cast<const __nv_bfloat16 *>(a), static_cast<const __nv_bfloat16 *>(b), A_log, dt_bias,
        static_cast<__nv_bfloat16 *>(out), data_wait_limit());
    return cudaGetLastError();
}

}  // namespace

// v-heads per unit of the tensor-core verify: two (a pair of one q/k head)
// when the heads come in even groups and the window fits the paired layout
int verify_tc_heads_per_unit(const LayerArgs &P) { return (P.G % 2 == 0 && P.T <= 4) ? 2 : 1; }

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
    if (P.T <= 4) {
        if (verify_tc_heads_per_unit(P) == 2)
            return launch_tm<4, 2>(dev, 0, tmap, P, C, slot_idx, B, q, k, v, a, b, A_log, dt_bias, out, stream);
        return launch_tm<4, 1>(dev, 1, tmap, P, C, slot_idx, B, q, k, v, a, b, A_log, dt_bias, out, stream);
    }
    return launch_tm<8, 1>(dev, 2, tmap, P, C, slot_idx, B, q, k, v, a, b, A_log, dt_bias, out, stream);
}

}  // namespace gdnspec
