// prefill.cu -- prefill of a request's prompt into its slot: the recurrence
// over the N prompt tokens of every row, the output of every token, the final
// state written as the slot's checkpoint, and the slot's cursors reset for
// decode (the prefill -> decode handoff, blog post on sglang PR #28695,
// appendix A.2).  It starts from a zero state or continues from the
// checkpoint, which gives chunked prefill across calls; continuing needs an
// empty ring (write_pos == 0, i.e. folded), else the row is skipped with
// GDN_SPEC_ST_UNFOLDED.
//
// The recurrence is replayed token by token in fp32, as the exact fold does
// (prhub summary of sglang PR #28695, implementation item 3; blog §12.7), with
// the same arrangement: a thread owns a quarter of the K columns of two state
// rows (p and p + 32 of a 64-row block) in registers, raw keys and queries stay
// in shared memory in the I/O dtype and are widened in registers, and the
// scalar decay is carried as a running factor (S = gam R, renormalised below
// 2^-32).  Per token, after the update, the output is
//     o_t = scale S_t q^_t = scale gam_t (R_t q_t) / |q_t|.
// The prompt streams through shared memory in chunks of 64 tokens, brought in
// by 1-D bulk asynchronous copies on an mbarrier (one row per token for k, q
// and the block's v values); the gates are computed from a and b meanwhile.
//
// The same kernel, instantiated with SNAP, is the comparison variant of the
// per-draft snapshot design that the ReplaySSM ring replaces (blog §0-§1, the
// intermediate_ssm buffer): it advances each row's state through the draft
// window from the checkpoint, reads out every position and stores the full
// state after every position (one V x K fp32 state per (row, position,
// v-head)); the checkpoint is only read and no cursor is touched.  Its commit
// copies the state after the accepted tokens back into the checkpoint.
#include "common.cuh"
#include "launch_setup.cuh"
#include "ptx_sm100.cuh"
#include "replay.cuh"

namespace gdnspec {

bool prefill_tc_supported(const LayerArgs &P, bool kda, bool bf16);
cudaError_t launch_prefill_tc(const LayerArgs &P, const CursorArgs &C, const int32_t *slot_idx, int B,
                              int N, const void *q, const void *k, const void *v, const void *a,
                              const void *b, const float *A_log, const float *dt_bias, void *out,
                              int from_zero, cudaStream_t stream);

constexpr int kPreThreads = 128;
constexpr int kPreTPR = 4;                          // threads per pair of state rows
constexpr int kPrePairs = kPreThreads / kPreTPR;    // 32
constexpr int kPreRows = 2 * kPrePairs;             // state rows per work item
constexpr int kPreChunk = 64;                       // prompt tokens per shared-memory chunk

__host__ __device__ constexpr size_t pre_pad16(size_t bytes) { return (bytes + 15) & ~(size_t)15; }

// Shared memory of one chunk: raw k and q rows [64][K] and the block's v
// values [64][64] in the I/O dtype; fp32 (alpha, 1/alpha) [64] (KDA alpha
// [64][K]), beta, 1/|k|, 1/|q| [64].
struct PrefillSmem {
    size_t keys, qs, vals, alpha, beta, rsk, rsq, total;
    __host__ __device__ PrefillSmem(int K, bool kda, size_t io) {
        keys = 0;
        qs = keys + pre_pad16((size_t)kPreChunk * K * io);
        vals = qs + pre_pad16((size_t)kPreChunk * K * io);
        alpha = vals + pre_pad16((size_t)kPreChunk * kPreRows * io);
        beta = alpha + pre_pad16(sizeof(float) * (size_t)kPreChunk * (kda ? K : 2));
        rsk = beta + pre_pad16(sizeof(float) * kPreChunk);
        rsq = rsk + pre_pad16(sizeof(float) * kPreChunk);
        total = rsq + pre_pad16(sizeof(float) * kPreChunk);
    }
};

size_t prefill_smem_bytes(int K, bool kda, bool bf16) { return PrefillSmem(K, kda, bf16 ? 2 : 4).total; }

// Which rows a prefill computes (the oracle's rule); sets *st for the others.
__device__ __forceinline__ bool prefill_row_ok(const CursorArgs &C, int slot, int L, int from_zero,
                                               uint32_t *st) {
    *st = 0;
    if (slot < 0) return false;
    if (slot >= C.num_slots) { *st = GDN_SPEC_ST_SLOT_OOR; return false; }
    const int wp = C.write_pos[slot], base = C.cache_base[slot];
    if (wp < 0 || wp > L || base < 0 || base >= L) { *st = GDN_SPEC_ST_CURSOR_CORRUPT; return false; }
    if (!from_zero && wp != 0) { *st = GDN_SPEC_ST_UNFOLDED; return false; }
    return true;
}

constexpr int kPreCtasPerSm = 3;   // registers: two state rows, a key or query chunk, sums

template <typename IO, bool KDA, int K, bool SNAP>
__global__ void __launch_bounds__(kPreThreads, kPreCtasPerSm)
prefill_kernel(LayerArgs P, CursorArgs C, const int32_t *__restrict__ slot_idx, int B, int N,
               const IO *__restrict__ q, const IO *__restrict__ k, const IO *__restrict__ v,
               const IO *__restrict__ a, const IO *__restrict__ bgate, const float *__restrict__ A_log,
               const float *__restrict__ dt_bias, IO *__restrict__ out, int from_zero,
               float *__restrict__ snap, uint32_t wait_limit) {
    static_assert(K % 32 == 0 && K <= 128, "whole 16-byte key chunks per thread");
    using KC = KeyChunk<IO>;
    constexpr int kPer = KC::kVals;                 // values per 16-byte chunk
    constexpr int kNC = K / kPer / kPreTPR;         // chunks per thread: chunk part + 4 m
    constexpr int kNP = kNC * kPer / 2;             // float2 pairs per thread and row
    extern __shared__ __align__(16) uint8_t smem[];
    __shared__ __align__(8) uint64_t s_bar;
    const int V = P.V, L = P.L, HV = P.HV, H = P.H;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const PrefillSmem lay(K, KDA, sizeof(IO));
    IO *Xk = reinterpret_cast<IO *>(smem + lay.keys);   // [64][K]
    IO *Xq = reinterpret_cast<IO *>(smem + lay.qs);     // [64][K]
    IO *Xv = reinterpret_cast<IO *>(smem + lay.vals);   // [64][64]
    float *alpha = reinterpret_cast<float *>(smem + lay.alpha);
    float *betaS = reinterpret_cast<float *>(smem + lay.beta);
    float *rsk = reinterpret_cast<float *>(smem + lay.rsk);
    float *rsq = reinterpret_cast<float *>(smem + lay.rsq);
    const uint32_t bar = ptx::smem_addr(&s_bar);
    const int vblocks = (V + kPreRows - 1) / kPreRows;
    const long long nitems = (long long)B * HV * vblocks;
    const int pair = tid / kPreTPR, part = tid % kPreTPR;
    uint32_t phase = 0;
    bool failed = false;   // a wait ran out: the rows of the remaining items are only marked

    if (tid == 0) {
        ptx::mbar_init(bar, 1);
        ptx::mbar_init_fence();
    }
    __syncthreads();

    for (long long it = blockIdx.x; it < nitems; it += gridDim.x) {
        const int vbk = (int)(it % vblocks);
        const int hv = (int)((it / vblocks) % HV);
        const int bb = (int)(it / ((long long)vblocks * HV));
        const int h = hv / P.G;
        const int row0 = vbk * kPreRows;
        const int nrows = V - row0 < kPreRows ? V - row0 : kPreRows;   // a multiple of 8
        const int slot = slot_idx[bb];
        uint32_t st = 0;
        const bool row_ok = SNAP ? (slot >= 0 && slot < C.num_slots) : prefill_row_ok(C, slot, L, from_zero, &st);
        if (SNAP && slot >= C.num_slots) st = GDN_SPEC_ST_SLOT_OOR;
        if (!row_ok) {
            if (st && hv == 0 && vbk == 0 && tid == 0) atomicOr(C.status, st);
            // a skipped row reads out zeros
            for (int idx = tid; idx < N * nrows; idx += kPreThreads) {
                const int t = idx / nrows, r = idx - t * nrows;
                out[(((size_t)bb * N + t) * HV + hv) * V + row0 + r] = IO(0.0f);
            }
            continue;
        }
        if (failed) {   // an earlier item's wait ran out: not computed, poisoned by the cursor kernel
            if (!SNAP && tid == 0) C.is_flush[slot] = kFoldFailed;
            continue;
        }
        const size_t sh_hv = (size_t)slot * HV + hv;
        float *ckpt = P.checkpoint;
        const bool valid0 = pair < nrows, valid1 = pair + kPrePairs < nrows;

        // ---- the state rows: zero, or this thread's part of the checkpoint
        float2 S[2][kNP];
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
#pragma unroll
            for (int i = 0; i < kNP; ++i) S[rr][i] = make_float2(0.f, 0.f);
            if ((SNAP || !from_zero) && (rr ? valid1 : valid0)) {
                const float *srow = ckpt + (sh_hv * V + row0 + pair + rr * kPrePairs) * K;
#pragma unroll
                for (int m = 0; m < kNC; ++m) {
                    const float4 *src = reinterpret_cast<const float4 *>(srow + (part + 4 * m) * kPer);
#pragma unroll
                    for (int qq = 0; qq < kPer / 4; ++qq) {
                        const float4 f = src[qq];
                        S[rr][m * (kPer / 2) + 2 * qq] = make_float2(f.x, f.y);
                        S[rr][m * (kPer / 2) + 2 * qq + 1] = make_float2(f.z, f.w);
                    }
                }
            }
        }
        float gam = 1.0f, inv = 1.0f;   // scalar gate: S = gam R (every thread holds the same values)

        for (int c0 = 0; c0 < N; c0 += kPreChunk) {
            const int nt = N - c0 < kPreChunk ? N - c0 : kPreChunk;
            // ---- 1. k, q and v rows of the chunk by bulk copies (warp 0)
            if (warp == 0) {
                const uint32_t rbytes = (uint32_t)(K * sizeof(IO)), vbytes = (uint32_t)(nrows * sizeof(IO));
                if (lane == 0) {
                    ptx::fence_proxy_async_smem();   // the previous chunk's generic reads come first
                    ptx::mbar_expect_tx(bar, (uint32_t)nt * (2 * rbytes + vbytes));
                }
                __syncwarp();
                for (int t = lane; t < nt; t += 32) {
                    const size_t tok = (size_t)bb * N + c0 + t;
                    ptx::bulk_copy_g2s(ptx::smem_addr(Xk + (size_t)t * K), k + (tok * H + h) * K, rbytes, bar);
                    ptx::bulk_copy_g2s(ptx::smem_addr(Xq + (size_t)t * K), q + (tok * H + h) * K, rbytes, bar);
                    ptx::bulk_copy_g2s(ptx::smem_addr(Xv + (size_t)t * kPreRows), v + (tok * HV + hv) * V + row0,
                                       vbytes, bar);
                }
            }
            // ---- 2. gates of the chunk's tokens
            for (int t = tid; t < nt; t += kPreThreads) {
                const size_t tok = (size_t)bb * N + c0 + t;
                if (!KDA) {
                    const float g = gate_g(A_log[hv], to_f32<IO>(a[tok * HV + hv]), dt_bias[hv]);
                    reinterpret_cast<float2 *>(alpha)[t] = make_float2(expf(g), expf(-g));
                }
                betaS[t] = gate_beta(to_f32<IO>(bgate[tok * HV + hv]));
            }
            if (KDA) {
                for (int idx = tid; idx < nt * K; idx += kPreThreads) {
                    const int t = idx / K, kk = idx - t * K;
                    const size_t tok = (size_t)bb * N + c0 + t;
                    alpha[idx] = expf(gate_g(A_log[hv], to_f32<IO>(a[(tok * HV + hv) * K + kk]),
                                             dt_bias[(size_t)hv * K + kk]));
                }
            }
            // ---- 3. the copies land; 1/|k_t| and 1/|q_t| (two threads per token)
            const bool landed = ptx::mbar_wait(bar, phase, wait_limit);
            phase ^= 1u;
            if (__syncthreads_or(!landed)) {   // the same decision in every thread
                // record the failure (and, for prefill, mark the row so that its
                // cursor reset poisons it instead), give the copies one more
                // bounded wait so that none is still writing this CTA's shared
                // memory, and stop
                if (tid == 0) {
                    atomicOr(C.status, GDN_SPEC_ST_TIMEOUT);
                    if (!SNAP) C.is_flush[slot] = kFoldFailed;
                }
                ptx::mbar_wait(bar, phase ^ 1u, kWaitLimitDefault);
                failed = true;
                break;
            }
            {
                const int t = tid >> 1, hf = tid & 1;   // kPreThreads / 2 == kPreChunk
                float sk = 0.0f, sq = 0.0f;
                if (t < nt) {
                    const uint4 *kr = reinterpret_cast<const uint4 *>(Xk + (size_t)t * K) + hf * (K / kPer / 2);
                    const uint4 *qr = reinterpret_cast<const uint4 *>(Xq + (size_t)t * K) + hf * (K / kPer / 2);
#pragma unroll
                    for (int c = 0; c < K / kPer / 2; ++c) {
                        float2 x[kPer / 2], y[kPer / 2];
                        KC::widen(kr[c], x);
                        KC::widen(qr[c], y);
#pragma unroll
                        for (int i = 0; i < kPer / 2; ++i) {
                            sk = fmaf(x[i].y, x[i].y, fmaf(x[i].x, x[i].x, sk));
                            sq = fmaf(y[i].y, y[i].y, fmaf(y[i].x, y[i].x, sq));
                        }
                    }
                }
                sk += __shfl_xor_sync(0xffffffffu, sk, 1);
                sq += __shfl_xor_sync(0xffffffffu, sq, 1);
                if (t < nt && hf == 0) {
                    rsk[t] = 1.0f / sqrtf(sk + P.l2_eps);
                    rsq[t] = 1.0f / sqrtf(sq + P.l2_eps);
                }
            }
            __syncthreads();

            // ---- 4. the chunk's tokens, one after another
            for (int t = 0; t < nt; ++t) {
                float2 x[kNP];
                {
                    const uint4 *xk = reinterpret_cast<const uint4 *>(Xk + (size_t)t * K);
#pragma unroll
                    for (int m = 0; m < kNC; ++m) {
                        float2 c2[kPer / 2];
                        KC::widen(xk[part + 4 * m], c2);
#pragma unroll
                        for (int i = 0; i < kPer / 2; ++i) x[m * (kPer / 2) + i] = c2[i];
                    }
                }
                if (KDA) {
                    const float *al = alpha + (size_t)t * K;
#pragma unroll
                    for (int m = 0; m < kNC; ++m) {
                        const float4 *a4 = reinterpret_cast<const float4 *>(al + (part + 4 * m) * kPer);
#pragma unroll
                        for (int qq = 0; qq < kPer / 4; ++qq) {
                            const float4 av = a4[qq];
                            const int i = m * (kPer / 2) + 2 * qq;
#pragma unroll
                            for (int rr = 0; rr < 2; ++rr) {
                                S[rr][i] = __fmul2_rn(S[rr][i], make_float2(av.x, av.y));
                                S[rr][i + 1] = __fmul2_rn(S[rr][i + 1], make_float2(av.z, av.w));
                            }
                        }
                    }
                } else {
                    const float2 ai = reinterpret_cast<const float2 *>(alpha)[t];   // (alpha, 1 / alpha)
                    gam *= ai.x;
                    inv *= ai.y;
                    if (gam < 0x1p-32f) {   // the same branch in every thread
                        const float2 g2 = make_float2(gam, gam);
#pragma unroll
                        for (int i = 0; i < kNP; ++i) {
                            S[0][i] = __fmul2_rn(S[0][i], g2);
                            S[1][i] = __fmul2_rn(S[1][i], g2);
                        }
                        gam = 1.0f;
                        inv = 1.0f;
                    }
                }
                // delta against the decayed state
                float2 acc[2][2] = {{make_float2(0.f, 0.f), make_float2(0.f, 0.f)},
                                    {make_float2(0.f, 0.f), make_float2(0.f, 0.f)}};
#pragma unroll
                for (int i = 0; i < kNP; ++i) {
                    acc[0][i & 1] = __ffma2_rn(S[0][i], x[i], acc[0][i & 1]);
                    acc[1][i & 1] = __ffma2_rn(S[1][i], x[i], acc[1][i & 1]);
                }
                float u0 = (acc[0][0].x + acc[0][0].y) + (acc[0][1].x + acc[0][1].y);
                float u1 = (acc[1][0].x + acc[1][0].y) + (acc[1][1].x + acc[1][1].y);
                u0 += __shfl_xor_sync(0xffffffffu, u0, 1);
                u1 += __shfl_xor_sync(0xffffffffu, u1, 1);
                u0 += __shfl_xor_sync(0xffffffffu, u0, 2);
                u1 += __shfl_xor_sync(0xffffffffu, u1, 2);
                const float rk = rsk[t], be = betaS[t];
                const float v0 = to_f32<IO>(Xv[(size_t)t * kPreRows + pair]);
                const float v1 = to_f32<IO>(Xv[(size_t)t * kPreRows + pair + kPrePairs]);
                const float d0 = be * (v0 * inv - rk * u0) * rk;   // KDA: inv stays 1
                const float d1 = be * (v1 * inv - rk * u1) * rk;
                const float2 d20 = make_float2(d0, d0), d21 = make_float2(d1, d1);
#pragma unroll
                for (int i = 0; i < kNP; ++i) {
                    S[0][i] = __ffma2_rn(d20, x[i], S[0][i]);
                    S[1][i] = __ffma2_rn(d21, x[i], S[1][i]);
                }
                // output of the token from the updated state
                {
                    const uint4 *xq = reinterpret_cast<const uint4 *>(Xq + (size_t)t * K);
#pragma unroll
                    for (int m = 0; m < kNC; ++m) {
                        float2 c2[kPer / 2];
                        KC::widen(xq[part + 4 * m], c2);
#pragma unroll
                        for (int i = 0; i < kPer / 2; ++i) x[m * (kPer / 2) + i] = c2[i];
                    }
                }
#pragma unroll
                for (int rr = 0; rr < 2; ++rr) {
                    acc[rr][0] = make_float2(0.f, 0.f);
                    acc[rr][1] = make_float2(0.f, 0.f);
                }
#pragma unroll
                for (int i = 0; i < kNP; ++i) {
                    acc[0][i & 1] = __ffma2_rn(S[0][i], x[i], acc[0][i & 1]);
                    acc[1][i & 1] = __ffma2_rn(S[1][i], x[i], acc[1][i & 1]);
                }
                float w0 = (acc[0][0].x + acc[0][0].y) + (acc[0][1].x + acc[0][1].y);
                float w1 = (acc[1][0].x + acc[1][0].y) + (acc[1][1].x + acc[1][1].y);
                w0 += __shfl_xor_sync(0xffffffffu, w0, 1);
                w1 += __shfl_xor_sync(0xffffffffu, w1, 1);
                w0 += __shfl_xor_sync(0xffffffffu, w0, 2);
                w1 += __shfl_xor_sync(0xffffffffu, w1, 2);
                if (part == 0) {
                    const float f = P.scale * gam * rsq[t];
                    const size_t o = (((size_t)bb * N + c0 + t) * HV + hv) * V + row0 + pair;
                    if (valid0) out[o] = IO(f * w0);
                    if (valid1) out[o + kPrePairs] = IO(f * w1);
                }
                if (SNAP) {   // the full state after this position
                    const float2 g2 = make_float2(gam, gam);
#pragma unroll
                    for (int rr = 0; rr < 2; ++rr) {
                        if (!(rr ? valid1 : valid0)) continue;
                        float *drow = snap + ((((size_t)bb * N + c0 + t) * HV + hv) * V + row0 + pair +
                                              rr * kPrePairs) * K;
#pragma unroll
                        for (int m = 0; m < kNC; ++m) {
                            float4 *dst = reinterpret_cast<float4 *>(drow + (part + 4 * m) * kPer);
#pragma unroll
                            for (int qq = 0; qq < kPer / 4; ++qq) {
                                const int i = m * (kPer / 2) + 2 * qq;
                                const float2 x0 = KDA ? S[rr][i] : __fmul2_rn(S[rr][i], g2);
                                const float2 x1 = KDA ? S[rr][i + 1] : __fmul2_rn(S[rr][i + 1], g2);
                                dst[qq] = make_float4(x0.x, x0.y, x1.x, x1.y);
                            }
                        }
                    }
                }
            }
            __syncthreads();   // the chunk's buffers are reused by the next chunk
        }
        if (failed) continue;
        if (SNAP) continue;   // the snapshot variant only reads the checkpoint

        // ---- 5. S = gam R into the checkpoint
        const float2 g2 = make_float2(gam, gam);
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
            if (!(rr ? valid1 : valid0)) continue;
            float *drow = ckpt + (sh_hv * V + row0 + pair + rr * kPrePairs) * K;
#pragma unroll
            for (int m = 0; m < kNC; ++m) {
                float4 *dst = reinterpret_cast<float4 *>(drow + (part + 4 * m) * kPer);
#pragma unroll
                for (int qq = 0; qq < kPer / 4; ++qq) {
                    const int i = m * (kPer / 2) + 2 * qq;
                    const float2 x0 = KDA ? S[rr][i] : __fmul2_rn(S[rr][i], g2);
                    const float2 x1 = KDA ? S[rr][i + 1] : __fmul2_rn(S[rr][i + 1], g2);
                    dst[qq] = make_float4(x0.x, x0.y, x1.x, x1.y);
                }
            }
        }
    }
}

// After the prefill: the cursors of the rows it computed are reset for decode;
// a row whose prefill stopped on a wait that ran out (marked kFoldFailed) is
// poisoned instead (write_pos = -1: CURSOR_CORRUPT until gdn_spec_reset).
__global__ void prefill_cursor_kernel(CursorArgs C, int L, const int32_t *__restrict__ slot_idx, int B,
                                      int from_zero) {
    for (int bb = blockIdx.x * blockDim.x + threadIdx.x; bb < B; bb += gridDim.x * blockDim.x) {
        const int slot = slot_idx[bb];
        uint32_t st;
        if (!prefill_row_ok(C, slot, L, from_zero, &st)) continue;
        if (C.is_flush[slot] == kFoldFailed) {
            C.write_pos[slot] = -1;
            C.is_flush[slot] = 0;
            continue;
        }
        C.write_pos[slot] = 0;
        C.cache_base[slot] = 0;
        C.is_flush[slot] = 0;
    }
}

// checkpoint[slot, hv] = snap[b, accept_len - 1, hv] for 1 <= accept_len <= T
// (0 keeps the state); one CTA per (row, v-head), 16-byte copies
__global__ void snapshot_commit_kernel(LayerArgs P, CursorArgs C, const int32_t *__restrict__ slot_idx,
                                       int B, const int32_t *__restrict__ accept_len,
                                       const float *__restrict__ snap) {
    const int bb = blockIdx.x / P.HV, hv = blockIdx.x % P.HV;
    const int slot = slot_idx[bb];
    if (slot < 0) return;
    if (slot >= C.num_slots) {
        if (hv == 0 && threadIdx.x == 0) atomicOr(C.status, GDN_SPEC_ST_SLOT_OOR);
        return;
    }
    const int acc = accept_len[bb];
    if (acc < 0 || acc > P.T) {
        if (hv == 0 && threadIdx.x == 0) atomicOr(C.status, GDN_SPEC_ST_ACCEPT_RANGE);
        return;
    }
    if (acc == 0) return;
    const size_t n4 = (size_t)P.V * P.K / 4;
    const float4 *src = reinterpret_cast<const float4 *>(snap + (((size_t)bb * P.T + acc - 1) * P.HV + hv) * P.V * P.K);
    float4 *dst = reinterpret_cast<float4 *>(P.checkpoint + ((size_t)slot * P.HV + hv) * P.V * P.K);
    for (size_t i = threadIdx.x; i < n4; i += blockDim.x) dst[i] = src[i];
}

static cudaError_t launch_prefill_cursors(const CursorArgs &C, int L, const int32_t *slot_idx, int B,
                                          int from_zero, cudaStream_t stream) {
    const int cb = (B + 255) / 256;
    prefill_cursor_kernel<<<cb < 1 ? 1 : (cb > 64 ? 64 : cb), 256, 0, stream>>>(C, L, slot_idx, B, from_zero);
    return cudaGetLastError();
}

template <typename IO, bool KDA, int K, bool SNAP>
static cudaError_t launch_prefill_k(const LayerArgs &P, const CursorArgs &C, const int32_t *slot_idx,
                                    int B, int N, const void *q, const void *k, const void *v,
                                    const void *a, const void *b, const float *A_log,
                                    const float *dt_bias, void *out, int from_zero, float *snap,
                                    cudaStream_t stream) {
    const size_t smem = PrefillSmem(K, KDA, sizeof(IO)).total;
    auto kern = prefill_kernel<IO, KDA, K, SNAP>;
    static KernelSetup setup;
    int sms = 0;
    cudaError_t e = kernel_setup(setup, reinterpret_cast<const void *>(kern), smem, &sms);
    if (e != cudaSuccess) return e;
    const long long items = (long long)B * P.HV * ((P.V + kPreRows - 1) / kPreRows);
    const long long cap = (long long)kPreCtasPerSm * sms;
    const int grid = (int)(items < cap ? items : cap);
    if (grid > 0)
        kern<<<grid, kPreThreads, smem, stream>>>(
            P, C, slot_idx, B, N, static_cast<const IO *>(q), static_cast<const IO *>(k),
            static_cast<const IO *>(v), static_cast<const IO *>(a), static_cast<const IO *>(b), A_log,
            dt_bias, static_cast<IO *>(out), from_zero, snap, data_wait_limit());
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (SNAP) return cudaSuccess;
    return launch_prefill_cursors(C, P.L, slot_idx, B, from_zero, stream);
}

template <typename IO, bool KDA, bool SNAP>
static cudaError_t launch_prefill_typed(const LayerArgs &P, const CursorArgs &C, const int32_t *slot_idx,
                                        int B, int N, const void *q, const void *k, const void *v,
                                        const void *a, const void *b, const float *A_log,
                                        const float *dt_bias, void *out, int from_zero, float *snap,
                                        cudaStream_t stream) {
    switch (P.K) {
        case 32: return launch_prefill_k<IO, KDA, 32, SNAP>(P, C, slot_idx, B, N, q, k, v, a, b, A_log, dt_bias, out, from_zero, snap, stream);
        case 64: return launch_prefill_k<IO, KDA, 64, SNAP>(P, C, slot_idx, B, N, q, k, v, a, b, A_log, dt_bias, out, from_zero, snap, stream);
        case 128: return launch_prefill_k<IO, KDA, 128, SNAP>(P, C, slot_idx, B, N, q, k, v, a, b, A_log, dt_bias, out, from_zero, snap, stream);
        default: return cudaErrorInvalidValue;
    }
}

template <bool SNAP>
static cudaError_t launch_any(const LayerArgs &P, const CursorArgs &C, bool kda, bool bf16,
                              const int32_t *slot_idx, int B, int N, const void *q, const void *k,
                              const void *v, const void *a, const void *b, const float *A_log,
                              const float *dt_bias, void *out, int from_zero, float *snap,
                              cudaStream_t stream) {
    if (bf16)
        return kda ? launch_prefill_typed<__nv_bfloat16, true, SNAP>(P, C, slot_idx, B, N, q, k, v, a, b, A_log, dt_bias, out, from_zero, snap, stream)
                   : launch_prefill_typed<__nv_bfloat16, false, SNAP>(P, C, slot_idx, B, N, q, k, v, a, b, A_log, dt_bias, out, from_zero, snap, stream);
    return kda ? launch_prefill_typed<float, true, SNAP>(P, C, slot_idx, B, N, q, k, v, a, b, A_log, dt_bias, out, from_zero, snap, stream)
               : launch_prefill_typed<float, false, SNAP>(P, C, slot_idx, B, N, q, k, v, a, b, A_log, dt_bias, out, from_zero, snap, stream);
}

cudaError_t launch_prefill(const LayerArgs &P, const CursorArgs &C, bool kda, bool bf16,
                           const int32_t *slot_idx, int B, int N, const void *q, const void *k,
                           const void *v, const void *a, const void *b, const float *A_log,
                           const float *dt_bias, void *out, int from_zero, cudaStream_t stream) {
    if (prefill_tc_supported(P, kda, bf16)) {   // chunk-parallel form on the tensor cores
        cudaError_t e = launch_prefill_tc(P, C, slot_idx, B, N, q, k, v, a, b, A_log, dt_bias, out,
                                          from_zero, stream);
        if (e != cudaSuccess) return e;
        return launch_prefill_cursors(C, P.L, slot_idx, B, from_zero, stream);
    }
    return launch_any<false>(P, C, kda, bf16, slot_idx, B, N, q, k, v, a, b, A_log, dt_bias, out,
                             from_zero, nullptr, stream);
}

cudaError_t launch_snapshot_verify(const LayerArgs &P, const CursorArgs &C, bool kda, bool bf16,
                                   const int32_t *slot_idx, int B, const void *q, const void *k,
                                   const void *v, const void *a, const void *b, const float *A_log,
                                   const float *dt_bias, void *out, float *snap, cudaStream_t stream) {
    return launch_any<true>(P, C, kda, bf16, slot_idx, B, P.T, q, k, v, a, b, A_log, dt_bias, out, 0,
                            snap, stream);
}

cudaError_t launch_snapshot_commit(const LayerArgs &P, const CursorArgs &C, const int32_t *slot_idx,
                                   int B, const int32_t *accept_len, const float *snap,
                                   cudaStream_t stream) {
    snapshot_commit_kernel<<<B * P.HV, 256, 0, stream>>>(P, C, slot_idx, B, accept_len, snap);
    return cudaGetLastError();
}

}  // namespace gdnspec
