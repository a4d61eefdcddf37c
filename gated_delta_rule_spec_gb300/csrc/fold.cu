// fold.cu -- exact fold of the committed ring history into the checkpoint.
//
// sglang PR #28695 replaced the chunked (I+A)^{-1} flush, which is
// ill-conditioned and let long outputs drift, by a closed-loop fold that
// replays the raw (v, k, g, beta) records with the recurrence itself (blog
// post on PR #28695, §12.5-12.7; prhub summary of PR #28695, implementation
// item 3).  This kernel does exactly that, in fp32, token by token:
//     S <- exp(g_t) S   (KDA: S diag(exp(g_t)))
//     d  = beta_t (v_t - S k^_t),   S <- S + d k^_t^T
// Rows of S are independent under the recurrence (row i only sees v_t[i]),
// so four threads own one state row (K/4 values each, in registers; the row's
// dot product takes two shuffles) and replay the records one after another.
// The elementwise work uses Blackwell's packed fp32x2 instructions.
//
// Only the rows whose is_flush is set do any work, and in steady state that
// is a small share of the batch per step.  So the grid is persistent: every
// CTA scans the batch's flags, builds the same compact list of rows to fold,
// and takes work items (row, layer, v-head, block of 32 state rows)
// round-robin from it.  For an item every global read (keys, gates, values,
// the state rows) is issued in one round.  Folding runs after sampling,
// outside the forward, so the layers are independent here and one launch
// folds all of them (the blog's §2.1 observation about replay outside the
// forward).  The cursors move in a separate launch after every layer.
#include "common.cuh"

namespace gdnspec {

constexpr int kFoldThreads = 128;
constexpr int kFoldTPR = 4;                          // threads per state row
constexpr int kFoldRows = kFoldThreads / kFoldTPR;   // state rows per work item
constexpr int kFoldMaxL = 128;   // ring length limit of this kernel
constexpr int kFoldScan = kFoldThreads;

// Shared memory of one item: raw keys [L][K] fp32, alpha [L] (KDA [L][K]),
// beta [L], 1/|k| [L], values [L][32 rows] fp32, and the compacted row list.
size_t fold_smem_bytes(int K, int L, bool kda) {
    return sizeof(float) * ((size_t)L * K + (size_t)L * (kda ? K : 1) + 2 * L + (size_t)L * kFoldRows) +
           sizeof(int) * 2 * kFoldScan;
}

template <typename IO, bool KDA, int K>
__global__ void __launch_bounds__(kFoldThreads, 4)
fold_kernel(LayerArgs P, FoldLayers FL, int n_layers, CursorArgs C,
            const int32_t *__restrict__ slot_idx, int B) {
    static_assert(K % 32 == 0 && K <= 128, "K/4 state values per thread, in float4 chunks");
    constexpr int KC = K / 16;   // float4 chunks per thread: chunk c4 = part + 4 m
    extern __shared__ __align__(16) float sm[];
    __shared__ int s_count, s_warp_off[kFoldThreads / 32];
    const int V = P.V, L = P.L, HV = P.HV, H = P.H;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    float *Xs = sm;                                  // [L][K]
    float *alpha = Xs + (size_t)L * K;               // [L] or [L][K]
    float *betaS = alpha + (size_t)L * (KDA ? K : 1);
    float *rsS = betaS + L;                          // [L] 1 / |k_t|
    float *vv = rsS + L;                             // [L][kFoldRows]
    int *rows = reinterpret_cast<int *>(vv + (size_t)L * kFoldRows);
    int *meta = rows + kFoldScan;
    const int vblocks = (V + kFoldRows - 1) / kFoldRows;
    const int per_row = n_layers * HV * vblocks;
    long long item_base = 0;  // items enumerated in earlier scan passes

    for (int b0 = 0; b0 < B; b0 += kFoldScan) {
        // ---- scan kFoldScan batch rows, compact the flagged ones (same list in every CTA)
        const int bb = b0 + tid;
        int flag = 0, wp = 0, base = 0;
        if (bb < B) {
            const int slot = slot_idx[bb];
            if (slot >= 0 && slot < C.num_slots && C.is_flush[slot]) {
                wp = C.write_pos[slot];
                base = C.cache_base[slot];
                flag = (wp > 0 && wp <= L && base >= 0 && base < L) ? 1 : 0;
            }
        }
        const unsigned ball = __ballot_sync(0xffffffffu, flag);
        if (lane == 0) s_warp_off[warp] = __popc(ball);
        __syncthreads();
        if (tid == 0) {
            int acc = 0;
            for (int w = 0; w < kFoldThreads / 32; ++w) {
                const int c = s_warp_off[w];
                s_warp_off[w] = acc;
                acc += c;
            }
            s_count = acc;
        }
        __syncthreads();
        if (flag) {
            const int pos = s_warp_off[warp] + __popc(ball & ((1u << lane) - 1u));
            rows[pos] = bb;
            meta[pos] = (wp << 16) | base;
        }
        __syncthreads();
        const long long nitems = (long long)s_count * per_row;

        // ---- this CTA's items of the pass
        long long first = ((long long)blockIdx.x - item_base) % gridDim.x;
        if (first < 0) first += gridDim.x;
        for (long long it = first; it < nitems; it += gridDim.x) {
            const int e = (int)(it / per_row);
            int rem = (int)(it - (long long)e * per_row);
            const int li = rem / (HV * vblocks);
            rem -= li * HV * vblocks;
            const int hv = rem / vblocks, vbk = rem - hv * vblocks;
            const int h = hv / P.G;
            const int slot = slot_idx[rows[e]];
            const int W = meta[e] >> 16, base = meta[e] & 0xFFFF;
            const int r = tid / kFoldTPR, part = tid % kFoldTPR;
            const int vr = vbk * kFoldRows + r;   // this thread's state row
            const bool valid = vr < V;
            const size_t sh_hv = (size_t)slot * HV + hv, sh_h = (size_t)slot * H + h;
            const IO *rawk = reinterpret_cast<const IO *>(FL.rawk[li]);
            const IO *rawv = reinterpret_cast<const IO *>(FL.rawv[li]);
            const float *ring_g = FL.ring_g[li];
            const float *ring_beta = FL.ring_beta[li];
            float *ckpt = FL.checkpoint[li];

            // ---- one round of reads: the state row slice, keys (two threads per
            //      record), gates (thread per record), values
            float2 S2[2 * KC];
            const float4 *srow = reinterpret_cast<const float4 *>(ckpt + (sh_hv * V + (valid ? vr : 0)) * K);
#pragma unroll
            for (int m = 0; m < KC; ++m) {
                const float4 t4 = valid ? srow[part + 4 * m] : make_float4(0.f, 0.f, 0.f, 0.f);
                S2[2 * m] = make_float2(t4.x, t4.y);
                S2[2 * m + 1] = make_float2(t4.z, t4.w);
            }
            // keys stay raw in shared memory; rs[t] = 1 / |k_t| (with eps) is
            // applied in the replay.  All loads of the item are issued before
            // any of them is used: keys of records tid/2 (+64 per pass), the
            // gates of record tid, the values of this thread's records.
            constexpr int KH = K / 2;                    // key elements per thread
            constexpr int kPer = 16 / (int)sizeof(IO);
            constexpr int kChunks = KH / kPer;
            const int half = tid & 1;
            uint4 kraw[kChunks];
            {
                const int j = tid >> 1;
                if (j < W) {
                    const uint4 *src = reinterpret_cast<const uint4 *>(
                        rawk + (sh_h * L + ring_pos(base, j, L)) * K + half * KH);
#pragma unroll
                    for (int c = 0; c < kChunks; ++c) kraw[c] = src[c];
                }
            }
            float g_in = 0.f, b_in = 0.f;
            if (tid < W) {
                const int p = ring_pos(base, tid, L);
                if (!KDA) g_in = ring_g[sh_hv * L + p];
                b_in = ring_beta[sh_hv * L + p];
            }
            float xv[kFoldMaxL / kFoldTPR];
#pragma unroll
            for (int u = 0; u < kFoldMaxL / kFoldTPR; ++u) {
                const int j = part + kFoldTPR * u;
                xv[u] = (j < W && valid) ? to_f32<IO>(rawv[(sh_hv * L + ring_pos(base, j, L)) * V + vr])
                                         : 0.0f;
            }
            // keys -> shared memory (first 64 records from the registers above)
            for (int pass = 0; pass * (kFoldThreads / 2) < W; ++pass) {
                const int j = pass * (kFoldThreads / 2) + (tid >> 1);
                if (pass > 0 && j < W) {
                    const uint4 *src = reinterpret_cast<const uint4 *>(
                        rawk + (sh_h * L + ring_pos(base, j, L)) * K + half * KH);
#pragma unroll
                    for (int c = 0; c < kChunks; ++c) kraw[c] = src[c];
                }
                float ss = 0.0f;
                if (j < W) {
#pragma unroll
                    for (int c = 0; c < kChunks; ++c) {
                        float x[kPer];
                        const uint4 u4 = kraw[c];
                        if constexpr (sizeof(IO) == 2) {
                            const uint32_t w[4] = {u4.x, u4.y, u4.z, u4.w};
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w[e]));
                                x[2 * e] = f.x;
                                x[2 * e + 1] = f.y;
                            }
                        } else {
                            x[0] = __uint_as_float(u4.x); x[1] = __uint_as_float(u4.y);
                            x[2] = __uint_as_float(u4.z); x[3] = __uint_as_float(u4.w);
                        }
#pragma unroll
                        for (int e = 0; e < kPer; e += 4) {
                            ss = fmaf(x[e], x[e], ss); ss = fmaf(x[e + 1], x[e + 1], ss);
                            ss = fmaf(x[e + 2], x[e + 2], ss); ss = fmaf(x[e + 3], x[e + 3], ss);
                            *reinterpret_cast<float4 *>(Xs + j * K + half * KH + c * kPer + e) =
                                make_float4(x[e], x[e + 1], x[e + 2], x[e + 3]);
                        }
                    }
                }
                ss += __shfl_xor_sync(0xffffffffu, ss, 1);
                if (j < W && half == 0) rsS[j] = 1.0f / sqrtf(ss + P.l2_eps);
            }
            if (KDA) {
                for (int idx = tid; idx < W * K; idx += kFoldThreads) {
                    const int j = idx / K, kk = idx - j * K;
                    alpha[idx] = expf(ring_g[(sh_hv * L + ring_pos(base, j, L)) * K + kk]);
                }
            } else if (tid < W) {
                alpha[tid] = expf(g_in);
            }
            if (tid < W) betaS[tid] = b_in;
            for (int j = kFoldThreads + tid; j < W; j += kFoldThreads) {  // records >= 128 (none: L <= 128)
                if (!KDA) alpha[j] = expf(ring_g[sh_hv * L + ring_pos(base, j, L)]);
                betaS[j] = ring_beta[sh_hv * L + ring_pos(base, j, L)];
            }
#pragma unroll
            for (int u = 0; u < kFoldMaxL / kFoldTPR; ++u) {
                const int j = part + kFoldTPR * u;
                if (j < W) vv[j * kFoldRows + r] = xv[u];
            }
            __syncthreads();

            // ---- replay (decay, then the delta against the decayed state)
            for (int t = 0; t < W; ++t) {
                const float4 *xk = reinterpret_cast<const float4 *>(Xs + t * K);
                float2 acc[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
                if (KDA) {
                    const float4 *al = reinterpret_cast<const float4 *>(alpha + (size_t)t * K);
#pragma unroll
                    for (int m = 0; m < KC; ++m) {
                        const float4 a4 = al[part + 4 * m], x4 = xk[part + 4 * m];
                        S2[2 * m] = __fmul2_rn(S2[2 * m], make_float2(a4.x, a4.y));
                        S2[2 * m + 1] = __fmul2_rn(S2[2 * m + 1], make_float2(a4.z, a4.w));
                        acc[0] = __ffma2_rn(S2[2 * m], make_float2(x4.x, x4.y), acc[0]);
                        acc[1] = __ffma2_rn(S2[2 * m + 1], make_float2(x4.z, x4.w), acc[1]);
                    }
                } else {
                    const float a = alpha[t];
                    const float2 a2 = make_float2(a, a);
#pragma unroll
                    for (int m = 0; m < KC; ++m) {
                        const float4 x4 = xk[part + 4 * m];
                        S2[2 * m] = __fmul2_rn(S2[2 * m], a2);
                        S2[2 * m + 1] = __fmul2_rn(S2[2 * m + 1], a2);
                        acc[0] = __ffma2_rn(S2[2 * m], make_float2(x4.x, x4.y), acc[0]);
                        acc[1] = __ffma2_rn(S2[2 * m + 1], make_float2(x4.z, x4.w), acc[1]);
                    }
                }
                float u = (acc[0].x + acc[0].y) + (acc[1].x + acc[1].y);
                u += __shfl_xor_sync(0xffffffffu, u, 1);
                u += __shfl_xor_sync(0xffffffffu, u, 2);
                const float rs = rsS[t];
                const float d = betaS[t] * (vv[t * kFoldRows + r] - rs * u) * rs;
                const float2 d2 = make_float2(d, d);
#pragma unroll
                for (int m = 0; m < KC; ++m) {
                    const float4 x4 = xk[part + 4 * m];
                    S2[2 * m] = __ffma2_rn(d2, make_float2(x4.x, x4.y), S2[2 * m]);
                    S2[2 * m + 1] = __ffma2_rn(d2, make_float2(x4.z, x4.w), S2[2 * m + 1]);
                }
            }
            if (valid) {
                float4 *dst = reinterpret_cast<float4 *>(ckpt + (sh_hv * V + vr) * K);
#pragma unroll
                for (int m = 0; m < KC; ++m)
                    dst[part + 4 * m] = make_float4(S2[2 * m].x, S2[2 * m].y, S2[2 * m + 1].x, S2[2 * m + 1].y);
            }
            __syncthreads();  // the item's buffers are reused by the next item
        }
        item_base += nitems;
        __syncthreads();  // the row list is rebuilt by the next pass
    }
}

template <typename IO, bool KDA, int K>
static cudaError_t launch_fold_k(const LayerArgs &P, const FoldLayers &FL, int n_layers,
                                 const CursorArgs &C, const int32_t *slot_idx, int B,
                                 cudaStream_t stream) {
    const size_t smem = fold_smem_bytes(K, P.L, KDA);
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    auto kern = fold_kernel<IO, KDA, K>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    // enough CTAs for every item of a typical step to run at once; the ones
    // without an item leave after the flag scan
    kern<<<4 * sms, kFoldThreads, smem, stream>>>(P, FL, n_layers, C, slot_idx, B);
    return cudaGetLastError();
}

template <typename IO, bool KDA>
static cudaError_t launch_fold_typed(const LayerArgs &P, const FoldLayers &FL, int n_layers,
                                     const CursorArgs &C, const int32_t *slot_idx, int B,
                                     cudaStream_t stream) {
    switch (P.K) {
        case 32: return launch_fold_k<IO, KDA, 32>(P, FL, n_layers, C, slot_idx, B, stream);
        case 64: return launch_fold_k<IO, KDA, 64>(P, FL, n_layers, C, slot_idx, B, stream);
        case 128: return launch_fold_k<IO, KDA, 128>(P, FL, n_layers, C, slot_idx, B, stream);
        default: return cudaErrorInvalidValue;
    }
}

bool fold_supported(int K, int L) { return (K == 32 || K == 64 || K == 128) && L <= kFoldMaxL; }

cudaError_t launch_fold(const LayerArgs &P, const FoldLayers &FL, int n_layers, bool kda,
                        bool bf16, const CursorArgs &C, const int32_t *slot_idx, int B,
                        cudaStream_t stream) {
    if (bf16)
        return kda ? launch_fold_typed<__nv_bfloat16, true>(P, FL, n_layers, C, slot_idx, B, stream)
                   : launch_fold_typed<__nv_bfloat16, false>(P, FL, n_layers, C, slot_idx, B, stream);
    return kda ? launch_fold_typed<float, true>(P, FL, n_layers, C, slot_idx, B, stream)
               : launch_fold_typed<float, false>(P, FL, n_layers, C, slot_idx, B, stream);
}

}  // namespace gdnspec
