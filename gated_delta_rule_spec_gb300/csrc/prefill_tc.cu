// prefill_tc.cu -- chunk-parallel prefill on the tensor cores: the GDN
// recurrence over a prompt, 64 tokens at a time, in the chunked UT / WY form
// that the blog post on sglang PR #28695 (appendix B.1) names as the prefill
// authority (chunk_gated_delta_rule), for the scalar gate with bf16 I/O,
// K = 128 and V a multiple of 128.  Same contract as the sequential prefill
// kernel (prefill.cu): outputs of every token, final state into the slot's
// checkpoint, cursors reset by the cursor kernel launched after it.
//
// Within a chunk of n tokens starting from state S (V x K), with cumulative
// log-decay G_t = g_1 + ... + g_t, Gam_t = exp(G_t), unit-norm keys k^ and
// queries q^, the per-token recurrence S_t = a_t S_{t-1} + d_t k^_t^T with
// d_t = beta_t (v_t - a_t S_{t-1} k^_t) unrolls to
//     (I + A) D = R,  A[t][i] = beta_t exp(G_t - G_i) <k^_t, k^_i>  (i < t),
//                     R[t]    = beta_t (v_t - Gam_t S k^_t),
//     o_t   = scale (Gam_t S q^_t + sum_{i <= t} exp(G_t - G_i) <q^_t, k^_i> d_i),
//     S_new = Gam_n S + sum_i exp(G_n - G_i) d_i k^_i^T.
// Every decay factor is exp of a difference G_t - G_i <= 0, so nothing
// overflows however strong the decay.
//
// One CTA (256 threads: two groups of four warps, each thread of a group on
// one state row) owns a unit (batch row, v-head, block of 128 state rows) and
// carries its state in tensor memory through the row's chunks:
//   * TMA brings each chunk's k and q rows (bf16, 128-byte swizzle, the MMA
//     operand layout) and v rows into one of two buffers, the next chunk's
//     while this one computes;
//   * tcgen05 kind::f16 computes the raw Gram [K; Q] K^T of the chunk (exact
//     bf16 products, fp32 sums; the L2 norms are applied as factors), and
//     kind::tf32 computes P = S [K^; Gam Q^]^T with the state as the A operand
//     straight from tensor memory;
//   * the first group solves (I + A) D = R, each thread for its own state row,
//     by forward substitution in 16-token blocks (fp32, CUDA cores; a short
//     loop, so that the code stays in the instruction cache), while the second
//     group decays the state and builds the update's key operand;
//   * kind::tf32 MMAs with D from tensor memory add D W^T to Gam Q^ S^T (the
//     outputs) and D (w K^) to the decayed state (the update).  The update's
//     operands are split into tf32 high and low parts (three products), so the
//     state keeps close to fp32 accuracy over long prompts;
//   * a full chunk's outputs are staged over its (dead) v rows and written by
//     one TMA store.
// Tensor memory (512 columns, one CTA per SM): S 0..127, P_k 128..191,
// P_q / outputs 192..255, Gram 256..319, D high 320..383, D low 384..447.
#include <cuda.h>
#include <mutex>

#include "common.cuh"
#include "ptx_sm100.cuh"

namespace gdnspec {
namespace ptc {

constexpr int kC = 64;          // tokens per chunk
constexpr int kK = 128;         // key dim
constexpr int kBV = 128;        // state rows per unit = MMA M
constexpr int kThreads = 256;   // two groups of four warps
// the thread that issues the chunk copies and output stores: outside the
// warps that compute the gates (0, 1) and apart from the MMA issuer (0)
constexpr int kCopier = 64;

// Shared-memory map (bytes from a 1024-aligned base).
constexpr int kAtomKQ = 128 * 128;                 // one 64-channel bf16 slice of [K; Q]
constexpr int kRawV = kC * kBV * 2;                // the chunk's v rows [64][128] bf16
constexpr int kRawBytes = 2 * kAtomKQ + kRawV;     // 49152 per chunk buffer
constexpr int kOffRaw = 0;                         // two chunk buffers
constexpr int kAtomX = 128 * 128;                  // one 32-channel fp32 slice of 128 rows
constexpr int kOffX = 2 * kRawBytes;               // [K^; Gam Q^] fp32, 4 slices
constexpr int kOffKwHi = kOffX;                    // then (w K^)^T high part, 2 slices of 32 tokens
constexpr int kOffKwLo = kOffX + 2 * kAtomX;       //      and low part
constexpr int kAtomW = 64 * 128;                   // one 32-token fp32 slice of 64 rows
constexpr int kOffW = kOffX + 4 * kAtomX;          // W [64 t][64 i] fp32, 2 slices
constexpr int kALd = kC + 4;                       // row stride (floats) of A^T
constexpr int kOffAT = kOffW + 2 * kAtomW;         // A^T [64 i][kALd] fp32: A^T[i][t] = A[t][i]
constexpr int kDRows = kC - 16;                    // deltas kept for later blocks' corrections
constexpr int kOffD = kOffAT + kC * kALd * 4;      // D [48 t][128 rows] fp32
constexpr int kOffF = kOffD + kDRows * kBV * 4;    // G, Gam, beta, wexp [64]; rn [128]; scan [8]
constexpr int kOffBar = kOffF + (4 * kC + 128 + 8) * 4;
constexpr int kOffMisc = kOffBar + 32;             // full[2], mma1, mma2
constexpr int kSmemUsed = kOffMisc + 16;
constexpr int kSmemBytes = kSmemUsed + 1024;       // + alignment slack
static_assert(kRawBytes % 1024 == 0 && kOffX % 1024 == 0 && kOffW % 1024 == 0, "1024-byte operand bases");
static_assert(kOffBar % 8 == 0, "mbarrier alignment");
static_assert(kSmemBytes <= 227 * 1024, "shared memory of one CTA");

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0, kColPk = 128, kColPq = 192, kColGram = 256, kColDhi = 320, kColDlo = 384;

// byte offset of fp32 element (row, k) in a K-major 128-byte-swizzle operand
// whose 32-element K slices are `atom` bytes apart
__device__ __forceinline__ uint32_t sw_f32(int atom, int row, int k) {
    return (uint32_t)((k >> 5) * atom + row * 128 + ((((k & 31) >> 2) ^ (row & 7)) << 4) + (k & 3) * 4);
}
// byte offset of bf16 element (row, c) of a raw [K; Q] chunk buffer
__device__ __forceinline__ uint32_t sw_bf16(int row, int c) {
    return (uint32_t)((c >> 6) * kAtomKQ + row * 128 + ((((c & 63) >> 3) ^ (row & 7)) << 4) + (c & 7) * 2);
}
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Which rows a prefill computes (the oracle's rule); sets *st for the others.
__device__ __forceinline__ bool row_ok(const CursorArgs &C, int slot, int L, int from_zero, uint32_t *st) {
    *st = 0;
    if (slot < 0) return false;
    if (slot >= C.num_slots) { *st = GDN_SPEC_ST_SLOT_OOR; return false; }
    const int wp = C.write_pos[slot], base = C.cache_base[slot];
    if (wp < 0 || wp > L || base < 0 || base >= L) { *st = GDN_SPEC_ST_CURSOR_CORRUPT; return false; }
    if (!from_zero && wp != 0) { *st = GDN_SPEC_ST_UNFOLDED; return false; }
    return true;
}

__global__ void __launch_bounds__(kThreads, 1)
prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_q,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                  LayerArgs P, CursorArgs C,
                  const int32_t *__restrict__ slot_idx, int B, int N,
                  const __nv_bfloat16 *__restrict__ a, const __nv_bfloat16 *__restrict__ bgate,
                  const float *__restrict__ A_log, const float *__restrict__ dt_bias,
                  __nv_bfloat16 *__restrict__ out, int from_zero, uint32_t wait_limit) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = ptx::smem_addr(smem_raw);
    const uint32_t pad = (1024u - (raw_s & 1023u)) & 1023u;
    uint8_t *sm = smem_raw + pad;
    const uint32_t sm_s = raw_s + pad;
    float *const AT = reinterpret_cast<float *>(sm + kOffAT);
    float *const Dsm = reinterpret_cast<float *>(sm + kOffD);
    float *const Gs = reinterpret_cast<float *>(sm + kOffF);
    float *const Gam = Gs + kC;
    float *const betaS = Gam + kC;
    float *const wexp = betaS + kC;
    float *const rn = wexp + kC;        // [128]: 1/|k_t| (rows 0..63), 1/|q_t| (rows 64..127)
    float *const scan = rn + 128;       // per-warp totals of the gate prefix sum
    int *const misc = reinterpret_cast<int *>(sm + kOffMisc);   // [0] TMEM base
    const uint32_t bar_full = sm_s + kOffBar;   // + 8 buf
    const uint32_t bar_m1 = sm_s + kOffBar + 16, bar_m2 = sm_s + kOffBar + 24;

    // threads: two groups of four warps; thread (row, grp) with row = tid % 128
    // is TMEM lane `row` (warp w reaches lanes 32 (w % 4) .. + 31)
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int row = tid & (kBV - 1), grp = tid >> 7;
    const int HV = P.HV, V = P.V;
    const int VB = V / kBV;
    const int nunits = B * HV * VB;
    const int nch = (N + kC - 1) / kC;

    if (tid == 0) {
        ptx::mbar_init(bar_full, 1);
        ptx::mbar_init(bar_full + 8, 1);
        ptx::mbar_init(bar_m1, 1);
        ptx::mbar_init(bar_m2, 1);
        ptx::mbar_init_fence();
        if (N > 0) {
            ptx::prefetch_tmap(&tm_k);
            ptx::prefetch_tmap(&tm_q);
            ptx::prefetch_tmap(&tm_v);
            ptx::prefetch_tmap(&tm_o);
        }
    }
    if (warp == 0) ptx::tmem_alloc(sm_s + kOffMisc, kTmemCols);
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    const uint32_t tmem = static_cast<uint32_t>(misc[0]);
    const uint32_t tl = tmem + ((uint32_t)((warp & 3) * 32) << 16);   // this warp's lanes
    uint32_t ph_full = 0, ph_m1 = 0, ph_m2 = 0;   // phase bits (ph_full: bit per buffer)
    uint32_t inflight = 0;                        // copier: buffers whose copy was not seen landed
    uint32_t pend = 0;                            // MMA barriers whose wait ran out (bit 0: m1, 1: m2)
    int gbuf = 0;                                 // buffer of the next chunk
    bool dead = false;                            // a wait ran out: remaining rows are only marked

    constexpr uint32_t idesc_gram = ptx::idesc_bf16(128, 64);
    constexpr uint32_t idesc_p = ptx::idesc_tf32(128, 128);
    constexpr uint32_t idesc_o = ptx::idesc_tf32(128, 64);
    constexpr uint32_t idesc_u = ptx::idesc_tf32(128, 128);

    for (int u = blockIdx.x; u < nunits; u += gridDim.x) {
        const int vb = u % VB, hv = (u / VB) % HV, bb = u / (VB * HV);
        const int h = hv / P.G, v0 = vb * kBV;
        const int slot = slot_idx[bb];
        uint32_t st = 0;
        if (!row_ok(C, slot, P.L, from_zero, &st)) {
            if (st && hv == 0 && vb == 0 && tid == 0) atomicOr(C.status, st);
            for (int t = grp; t < N; t += 2)   // a skipped row reads out zeros
                out[(((size_t)bb * N + t) * HV + hv) * V + v0 + row] = __float2bfloat16_rn(0.0f);
            continue;
        }
        if (dead) {   // not computed: poisoned by the cursor kernel
            if (tid == 0) C.is_flush[slot] = kFoldFailed;
            continue;
        }
        float *const ck = P.checkpoint + (((size_t)slot * HV + hv) * V + v0 + row) * kK + 64 * grp;

        // ---- this thread's half of its state row into TMEM columns 64 grp ..
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            float r[16];
            if (from_zero) {
#pragma unroll
                for (int e = 0; e < 16; ++e) r[e] = 0.0f;
            } else {
                const float4 *src = reinterpret_cast<const float4 *>(ck + 16 * j);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float4 f = src[e];
                    r[4 * e] = f.x; r[4 * e + 1] = f.y; r[4 * e + 2] = f.z; r[4 * e + 3] = f.w;
                }
            }
            ptx::tmem_st16(tl + kColS + 64 * grp + 16 * j, r);
        }
        ptx::tmem_st_wait();

        const float Alog = A_log[hv], dtb = dt_bias[hv];
        auto issue_chunk = [&](int buf, int tok0) {
            const uint32_t dst = sm_s + kOffRaw + buf * kRawBytes, bar = bar_full + 8 * buf;
            const int z = bb * N + tok0;
            ptx::bulk_wait_read_all();   // an output store may still read this buffer's v rows
            ptx::mbar_expect_tx(bar, kRawBytes);
#pragma unroll
            for (int s = 0; s < 2; ++s) {
                ptx::tma_load_3d(dst + s * kAtomKQ, &tm_k, bar, 64 * s, h, z);
                ptx::tma_load_3d(dst + s * kAtomKQ + 64 * 128, &tm_q, bar, 64 * s, h, z);
            }
            ptx::tma_load_3d(dst + 2 * kAtomKQ, &tm_v, bar, v0, hv, z);
            inflight |= 1u << buf;
        };
        if (tid == kCopier && nch > 0) issue_chunk(gbuf, 0);
        // the gates' raw inputs of the first chunk (threads 0..63, one token
        // each), kept as bf16 bits: converted only when used, so that the
        // loads stay in flight until then
        const unsigned short *a16 = reinterpret_cast<const unsigned short *>(a);
        const unsigned short *b16 = reinterpret_cast<const unsigned short *>(bgate);
        uint32_t ra = 0u, rb = 0u;
        if (tid < kC && tid < N) {
            const size_t o = ((size_t)bb * N + tid) * HV + hv;
            ra = a16[o];
            rb = b16[o];
        }

        for (int c = 0; c < nch; ++c) {
            const int c0 = c * kC, n = N - c0 < kC ? N - c0 : kC;
            const int buf = gbuf;
            if (tid == kCopier && c + 1 < nch) issue_chunk(buf ^ 1, c0 + kC);

            // ---- 1. gates and their prefix sum; next chunk's raw gates
            float gsum = 0.0f, be = 0.0f;
            if (tid < kC) {
                float g = 0.0f;
                if (tid < n) {
                    g = gate_g(Alog, __uint_as_float(ra << 16), dtb);
                    be = gate_beta(__uint_as_float(rb << 16));
                }
                const int tn = c0 + kC + tid;
                ra = rb = 0u;
                if (tn < N) {
                    const size_t o = ((size_t)bb * N + tn) * HV + hv;
                    ra = a16[o];
                    rb = b16[o];
                }
                gsum = g;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const float y = __shfl_up_sync(0xffffffffu, gsum, o);
                    if (lane >= o) gsum += y;
                }
                if (lane == 31) scan[warp] = gsum;
            }
            __syncthreads();
            if (tid < kC) {
                const float G = gsum + (warp == 1 ? scan[0] : 0.0f);
                Gs[tid] = G;
                Gam[tid] = __expf(G);
                betaS[tid] = be;
            }
            // ---- 2. the chunk's rows landed
            const bool landed = ptx::mbar_wait(bar_full + 8 * buf, (ph_full >> buf) & 1u, wait_limit);
            if (landed) {   // (a phase not seen complete stays the one to drain)
                ph_full ^= 1u << buf;
                if (tid == kCopier) inflight &= ~(1u << buf);
            }
            if (__syncthreads_or(!landed)) {
                dead = true;
                break;
            }
            if (tid < kC) wexp[tid] = tid < n ? __expf(Gs[kC - 1] - Gs[tid]) : 0.0f;

            // ---- 3. X = [K^; Gam Q^] (tf32-rounded fp32) and the norms: thread
            //         (row, grp) reads the whole row for its norm and writes
            //         channels 64 grp .. 64 grp + 63
            const uint8_t *raw = sm + kOffRaw + buf * kRawBytes;
            {
                const int r = row, t = r & (kC - 1);
                float x[64];
                float ss = 0.0f;
#pragma unroll
                for (int s = 0; s < 2; ++s) {
                    const int sl = s ^ grp ^ 1;   // own slice last: its values stay in x
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const uint4 w = *reinterpret_cast<const uint4 *>(raw + sl * kAtomKQ + r * 128 +
                                                                         ((j ^ (r & 7)) << 4));
                        const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float lo = bf16_lo(ww[e]), hi = bf16_hi(ww[e]);
                            ss = fmaf(lo, lo, fmaf(hi, hi, ss));
                            x[8 * j + 2 * e] = lo;
                            x[8 * j + 2 * e + 1] = hi;
                        }
                    }
                }
                const bool valid = t < n;
                const float rinv = valid ? rsqrtf(ss + P.l2_eps) : 0.0f;
                const float f = r >= kC ? rinv * Gam[t] : rinv;
                if (grp == 0) rn[r] = rinv;
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    float4 xo = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (valid)
                        xo = make_float4(ptx::round_tf32(x[4 * j] * f), ptx::round_tf32(x[4 * j + 1] * f),
                                         ptx::round_tf32(x[4 * j + 2] * f), ptx::round_tf32(x[4 * j + 3] * f));
                    *reinterpret_cast<float4 *>(sm + kOffX + sw_f32(kAtomX, r, 64 * grp + 4 * j)) = xo;
                }
            }
            ptx::fence_proxy_async_smem();
            ptx::tc_fence_before_sync();
            __syncthreads();

            // ---- 4. Gram of the raw rows; P = S [K^; Gam Q^]^T
            if (tid == 0) {
                ptx::tc_fence_after_sync();
                const uint32_t kq = sm_s + kOffRaw + buf * kRawBytes;
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint64_t d = ptx::smem_desc_sw128(kq + (ks >> 2) * kAtomKQ + (ks & 3) * 32);
                    ptx::mma_bf16(tmem + kColGram, d, d, idesc_gram, ks != 0);
                }
#pragma unroll
                for (int ks = 0; ks < 16; ++ks)
                    ptx::mma_tf32_tmem_a(tmem + kColPk, tmem + kColS + 8 * ks,
                                         ptx::smem_desc_sw128(sm_s + kOffX + (ks >> 2) * kAtomX + (ks & 3) * 32),
                                         idesc_p, ks != 0);
                ptx::mma_commit(bar_m1);
            }
            const bool m1 = ptx::mbar_wait(bar_m1, ph_m1);
            ph_m1 ^= 1u;
            if (__syncthreads_or(!m1)) {
                pend |= 1u;
                dead = true;
                break;
            }
            ptx::tc_fence_after_sync();

            // ---- 5. A^T (key rows: A strictly lower) and W (query rows: lower
            //         with the diagonal) from this lane's Gram row; thread
            //         (row, grp) does columns 32 grp .. 32 grp + 31
            {
                float gr[32];
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    float q16[16];
                    ptx::tmem_ld16(tl + kColGram + 32 * grp + 16 * j, q16);
#pragma unroll
                    for (int e = 0; e < 16; ++e) gr[16 * j + e] = q16[e];
                }
                ptx::tmem_ld_wait();
                const int t = row & (kC - 1), i0 = 32 * grp;
                const float Gt = Gs[t];
                const bool tv = t < n;
                const bool keyrow = row < kC;
                // key rows: A^T[i][t] = beta_t exp(G_t - G_i) <k^_t, k^_i> (i < t);
                // query rows: W[t][i] = exp(G_t - G_i) <q^_t, k^_i> (i <= t)
                const float ft = keyrow ? betaS[t] * rn[t] : rn[kC + t];
#pragma unroll
                for (int i4 = 0; i4 < 8; ++i4) {
                    const float4 g4 = *reinterpret_cast<const float4 *>(Gs + i0 + 4 * i4);
                    const float4 n4 = *reinterpret_cast<const float4 *>(rn + i0 + 4 * i4);
                    const float gi[4] = {g4.x, g4.y, g4.z, g4.w}, ni[4] = {n4.x, n4.y, n4.z, n4.w};
                    float o[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int i = i0 + 4 * i4 + e;
                        const float x = ft * __expf(Gt - gi[e]) * gr[4 * i4 + e] * ni[e];
                        o[e] = (tv && (keyrow ? i < t : i <= t)) ? x : 0.0f;
                    }
                    if (keyrow) {
#pragma unroll
                        for (int e = 0; e < 4; ++e) AT[(i0 + 4 * i4 + e) * kALd + t] = o[e];
                    } else {
                        *reinterpret_cast<float4 *>(sm + kOffW + sw_f32(kAtomW, t, i0 + 4 * i4)) =
                            make_float4(ptx::round_tf32(o[0]), ptx::round_tf32(o[1]), ptx::round_tf32(o[2]),
                                        ptx::round_tf32(o[3]));
                    }
                }
            }
            __syncthreads();

            if (grp == 0) {
                // ---- 6. this state row's corrected deltas, (I + A) D = R, in
                //         blocks of 16 tokens: corrections from the earlier
                //         blocks' deltas, then the block's own triangle
                const __nv_bfloat16 *vr = reinterpret_cast<const __nv_bfloat16 *>(raw + 2 * kAtomKQ);
                for (int b = 0; b < kC / 16; ++b) {
                    float r[16];
                    ptx::tmem_ld16(tl + kColPk + 16 * b, r);
                    ptx::tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int t = 16 * b + j;
                        r[j] = t < n ? betaS[t] * (__bfloat162float(vr[t * kBV + row]) - Gam[t] * r[j]) : 0.0f;
                    }
                    {
                        float2 r2[8];
#pragma unroll
                        for (int q = 0; q < 8; ++q) r2[q] = make_float2(r[2 * q], r[2 * q + 1]);
#pragma unroll 4
                        for (int i = 0; i < 16 * b; ++i) {
                            const float x = -Dsm[i * kBV + row];
                            const float2 x2 = make_float2(x, x);
                            const float4 *ar = reinterpret_cast<const float4 *>(AT + i * kALd + 16 * b);
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                const float4 a4 = ar[q];
                                r2[2 * q] = __ffma2_rn(make_float2(a4.x, a4.y), x2, r2[2 * q]);
                                r2[2 * q + 1] = __ffma2_rn(make_float2(a4.z, a4.w), x2, r2[2 * q + 1]);
                            }
                        }
#pragma unroll
                        for (int q = 0; q < 8; ++q) {
                            r[2 * q] = r2[q].x;
                            r[2 * q + 1] = r2[q].y;
                        }
                    }
#pragma unroll
                    for (int i = 0; i < 15; ++i) {
                        const float x = r[i];
                        const float4 *ar = reinterpret_cast<const float4 *>(AT + (16 * b + i) * kALd + 16 * b);
#pragma unroll
                        for (int q = (i + 1) / 4; q < 4; ++q) {
                            const float4 a4 = ar[q];
                            const float av[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                if (4 * q + e > i) r[4 * q + e] = fmaf(-av[e], x, r[4 * q + e]);
                        }
                    }
                    if (b < kC / 16 - 1) {
#pragma unroll
                        for (int j = 0; j < 16; ++j) Dsm[(16 * b + j) * kBV + row] = r[j];
                    }
                    // D (high and low tf32 parts) into TMEM
                    float lo[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const float hi = ptx::round_tf32(r[j]);
                        lo[j] = r[j] - hi;
                        r[j] = hi;
                    }
                    ptx::tmem_st16(tl + kColDhi + 16 * b, r);
                    ptx::tmem_st16(tl + kColDlo + 16 * b, lo);
                }
            } else {
                // ---- 6'. meanwhile: S <- Gam_n S for this lane's state row, and
                //          (w K^)^T high and low parts (row = channel) over the dead X
                const float gn = Gam[kC - 1];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    float s16[16];
                    ptx::tmem_ld16(tl + kColS + 16 * j, s16);
                    ptx::tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 16; ++e) s16[e] *= gn;
                    ptx::tmem_st16(tl + kColS + 16 * j, s16);
                }
#pragma unroll 4
                for (int i4 = 0; i4 < kC / 4; ++i4) {
                    float hi[4], lo[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int i = 4 * i4 + e;
                        const float kv = __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(raw + sw_bf16(i, row)));
                        const float xk = i < n ? kv * rn[i] * wexp[i] : 0.0f;
                        hi[e] = ptx::round_tf32(xk);
                        lo[e] = xk - hi[e];
                    }
                    const uint32_t off = sw_f32(kAtomX, row, 4 * i4);
                    *reinterpret_cast<float4 *>(sm + kOffKwHi + off) = make_float4(hi[0], hi[1], hi[2], hi[3]);
                    *reinterpret_cast<float4 *>(sm + kOffKwLo + off) = make_float4(lo[0], lo[1], lo[2], lo[3]);
                }
            }
            ptx::tmem_st_wait();
            ptx::fence_proxy_async_smem();
            ptx::tc_fence_before_sync();
            __syncthreads();

            // ---- 7. outputs += D W^T; S += D (w K^) (three tf32 products)
            if (tid == 0) {
                ptx::tc_fence_after_sync();
#pragma unroll
                for (int part = 0; part < 2; ++part)
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks)
                        ptx::mma_tf32_tmem_a(tmem + kColPq, tmem + (part ? kColDlo : kColDhi) + 8 * ks,
                                             ptx::smem_desc_sw128(sm_s + kOffW + (ks >> 2) * kAtomW + (ks & 3) * 32),
                                             idesc_o, 1u);
#pragma unroll
                for (int part = 0; part < 3; ++part)
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks)
                        ptx::mma_tf32_tmem_a(tmem + kColS, tmem + (part == 2 ? kColDlo : kColDhi) + 8 * ks,
                                             ptx::smem_desc_sw128(sm_s + (part == 1 ? kOffKwLo : kOffKwHi) +
                                                                  (ks >> 2) * kAtomX + (ks & 3) * 32),
                                             idesc_u, 1u);
                ptx::mma_commit(bar_m2);
            }
            const bool m2 = ptx::mbar_wait(bar_m2, ph_m2);
            ph_m2 ^= 1u;
            if (__syncthreads_or(!m2)) {
                pend |= 2u;
                dead = true;
                break;
            }
            ptx::tc_fence_after_sync();

            // ---- 8. the chunk's outputs of this state row, tokens 32 grp .. + 31:
            //         a full chunk is staged over its (dead) v rows and leaves by
            //         one TMA store; a ragged one is stored directly
            const bool full = n == kC;
            __nv_bfloat16 *stage = reinterpret_cast<__nv_bfloat16 *>(sm + kOffRaw + buf * kRawBytes + 2 * kAtomKQ);
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                float o16[16];
                ptx::tmem_ld16(tl + kColPq + 32 * grp + 16 * j, o16);
                ptx::tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const int t = 32 * grp + 16 * j + e;
                    const __nv_bfloat16 o = __float2bfloat16_rn(P.scale * o16[e]);
                    if (full)
                        stage[t * kBV + row] = o;
                    else if (t < n)
                        out[(((size_t)bb * N + c0 + t) * HV + hv) * V + v0 + row] = o;
                }
            }
            // the buffer and the TMEM columns are reused by the next chunk
            ptx::fence_proxy_async_smem();
            ptx::tc_fence_before_sync();
            __syncthreads();
            if (full && tid == kCopier) {
                ptx::tma_store_3d(&tm_o, sm_s + kOffRaw + buf * kRawBytes + 2 * kAtomKQ, v0, hv, bb * N + c0);
                ptx::bulk_commit_group();
            }
            gbuf ^= 1;
        }
        if (dead) {
            // a wait ran out: record it, mark this row (the cursor kernel
            // poisons it), and let every copy and MMA still in flight finish
            // before the shared memory and TMEM are released
            if (tid == 0) {
                atomicOr(C.status, GDN_SPEC_ST_TIMEOUT);
                C.is_flush[slot] = kFoldFailed;
            }
            if (tid == kCopier) {
                for (int bf = 0; bf < 2; ++bf)
                    if (inflight & (1u << bf)) ptx::mbar_wait(bar_full + 8 * bf, (ph_full >> bf) & 1u);
                inflight = 0;
            }
            if (pend & 1u) ptx::mbar_wait(bar_m1, ph_m1 ^ 1u);
            if (pend & 2u) ptx::mbar_wait(bar_m2, ph_m2 ^ 1u);
            pend = 0;
            ptx::tc_fence_before_sync();
            __syncthreads();
            continue;
        }

        // ---- the final state into the checkpoint (this thread's half row)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            float s16[16];
            ptx::tmem_ld16(tl + kColS + 64 * grp + 16 * j, s16);
            ptx::tmem_ld_wait();
            float4 *dst = reinterpret_cast<float4 *>(ck + 16 * j);
#pragma unroll
            for (int e = 0; e < 4; ++e)
                dst[e] = make_float4(s16[4 * e], s16[4 * e + 1], s16[4 * e + 2], s16[4 * e + 3]);
        }
        ptx::tc_fence_before_sync();
        __syncthreads();
    }

    if (tid == kCopier) ptx::bulk_wait_all();   // the last output stores
    ptx::tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        ptx::tc_fence_after_sync();
        ptx::tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace ptc

namespace {

using EncodeTiledFnP = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                    const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                    const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                    CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFnP encode_fn_p() {
    static EncodeTiledFnP fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFnP>(p);
    });
    return fn;
}

// A token-major bf16 tensor [tokens][heads][dim] as a 3-D tensor map with
// boxes of (box_x elements of one head) x (64 tokens).
bool token_map(EncodeTiledFnP enc, CUtensorMap *m, const void *base, int dim, int heads,
               long long tokens, uint32_t box_x, bool swizzle) {
    const cuuint64_t gdim[3] = {(cuuint64_t)dim, (cuuint64_t)heads, (cuuint64_t)tokens};
    const cuuint64_t gstride[2] = {(cuuint64_t)dim * 2, (cuuint64_t)heads * dim * 2};
    const cuuint32_t box[3] = {box_x, 1, (cuuint32_t)ptc::kC};
    const cuuint32_t estride[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), gdim, gstride, box,
               estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
               swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

constexpr int kMaxDevicesP = 64;
int g_grid_p[kMaxDevicesP];   // per device: grid size, 0 until set up
std::mutex g_mu_p;

cudaError_t setup_p(int dev, int *grid) {
    std::lock_guard<std::mutex> lk(g_mu_p);
    if (!g_grid_p[dev]) {
        cudaError_t e = cudaFuncSetAttribute(ptc::prefill_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             ptc::kSmemBytes);
        if (e != cudaSuccess) return e;
        int sms = 0;
        if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
        g_grid_p[dev] = sms;   // one CTA per SM (shared memory and all 512 TMEM columns)
    }
    *grid = g_grid_p[dev];
    return cudaSuccess;
}

}  // namespace

// Shapes of the chunk-parallel prefill: GDN scalar gate, bf16 I/O, K = 128,
// V a multiple of 128.
bool prefill_tc_supported(const LayerArgs &P, bool kda, bool bf16) {
    return bf16 && !kda && P.K == ptc::kK && P.V % ptc::kBV == 0;
}

cudaError_t launch_prefill_tc(const LayerArgs &P, const CursorArgs &C, const int32_t *slot_idx, int B,
                              int N, const void *q, const void *k, const void *v, const void *a,
                              const void *b, const float *A_log, const float *dt_bias, void *out,
                              int from_zero, cudaStream_t stream) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevicesP) return cudaErrorInvalidDevice;
    int grid = 0;
    if ((e = setup_p(dev, &grid)) != cudaSuccess) return e;
    const int nunits = B * P.HV * (P.V / ptc::kBV);
    if (grid > nunits) grid = nunits;
    if (grid <= 0) return cudaSuccess;
    EncodeTiledFnP enc = encode_fn_p();
    if (!enc) return cudaErrorNotSupported;
    CUtensorMap mk{}, mq{}, mv{}, mo{};   // N == 0: no copy is issued and the maps stay empty
    if (N > 0) {
        const long long tokens = (long long)B * N;
        if (!token_map(enc, &mk, k, P.K, P.H, tokens, 64, true) ||
            !token_map(enc, &mq, q, P.K, P.H, tokens, 64, true) ||
            !token_map(enc, &mv, v, P.V, P.HV, tokens, ptc::kBV, false) ||
            !token_map(enc, &mo, out, P.V, P.HV, tokens, ptc::kBV, false))
            return cudaErrorInvalidValue;
    }
    ptc::prefill_tc_kernel<<<grid, ptc::kThreads, ptc::kSmemBytes, stream>>>(
        mk, mq, mv, mo, P, C, slot_idx, B, N, static_cast<const __nv_bfloat16 *>(a),
        static_cast<const __nv_bfloat16 *>(b), A_log, dt_bias, static_cast<__nv_bfloat16 *>(out), from_zero,
        data_wait_limit());
    return cudaGetLastError();
}

}  // namespace gdnspec
