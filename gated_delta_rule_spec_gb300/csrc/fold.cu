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
// so the work is parallel over V and sequential over the W records.
//
// Only the rows whose is_flush is set do any work, and in steady state that
// is a small share of the batch per step.  So the grid is persistent: every
// CTA scans the batch's flags, builds the same compact list of rows to fold,
// and takes work items (row, layer, v-head, block of 32 state rows)
// round-robin from it.  For an item, every global read (keys, gates, values)
// is issued in one round; then four threads per state row hold K/4 state
// values each in registers and replay the records.  Folding runs after
// sampling, outside the forward, so the layers are independent here and one
// launch folds all of them (the blog's §2.1 observation about replay outside
// the forward).  The cursors move in a separate launch after every layer.
#include "common.cuh"

namespace gdnspec {

constexpr int kFoldThreads = 128;
constexpr int kFoldRows = kFoldThreads / 4;  // state rows per work item
constexpr int kFoldMaxL = 128;               // ring length limit of this kernel
constexpr int kFoldScan = kFoldThreads;      // batch rows scanned per pass

size_t fold_smem_bytes(int K, int L, bool kda) {
    // keys [L][K], alpha [L] or [L][K], beta [L], values [L][kFoldRows], row list
    return sizeof(float) * ((size_t)L * K + (size_t)L * (kda ? K : 1) + L + (size_t)L * kFoldRows) +
           sizeof(int) * 2 * kFoldScan;
}

template <typename IO, bool KDA, int KC>
__global__ void __launch_bounds__(kFoldThreads)
fold_kernel(LayerArgs P, FoldLayers FL, int n_layers, CursorArgs C,
            const int32_t *__restrict__ slot_idx, int B) {
    extern __shared__ __align__(16) float sm[];
    __shared__ int s_count, s_warp_off[kFoldThreads / 32];
    const int K = P.K, V = P.V, L = P.L, HV = P.HV, H = P.H;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    float *Xs = sm;                                  // [L][K]
    float *alpha = Xs + (size_t)L * K;               // [L] or [L][K]
    float *betaS = alpha + (size_t)L * (KDA ? K : 1);
    float *vv = betaS + L;                           // [L][kFoldRows]
    int *rows = reinterpret_cast<int *>(vv + (size_t)L * kFoldRows);  // [kFoldScan] row, [kFoldScan] W|base
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
            const int v0 = vbk * kFoldRows;
            const size_t sh_hv = (size_t)slot * HV + hv, sh_h = (size_t)slot * H + h;
            const IO *rawk = reinterpret_cast<const IO *>(FL.rawk[li]);
            const IO *rawv = reinterpret_cast<const IO *>(FL.rawv[li]);
            const float *ring_g = FL.ring_g[li];
            const float *ring_beta = FL.ring_beta[li];
            float *ckpt = FL.checkpoint[li];

            // one round of reads: keys (warp-per-record), gates, values
            constexpr int kRecPerWarp = kFoldMaxL / (kFoldThreads / 32);  // 32
            constexpr int KPL = KC / 2;  // key elements per lane per record (K / 32)
            for (int j0 = 0; j0 < W; j0 += kRecPerWarp * (kFoldThreads / 32) / 4) {
                // records j0 + warp + 4 i, i < 8: keys loaded together, then normalised
                float kx[8][KPL];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int j = j0 + warp + 4 * i;
#pragma unroll
                    for (int m = 0; m < KPL; ++m) kx[i][m] = 0.0f;
                    if (j < W) {
                        const IO *src = rawk + (sh_h * L + ring_pos(base, j, L)) * K;
#pragma unroll
                        for (int m = 0; m < KPL; ++m)
                            if (lane + 32 * m < K) kx[i][m] = to_f32<IO>(src[lane + 32 * m]);
                    }
                }
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int j = j0 + warp + 4 * i;
                    float ss = 0.0f;
#pragma unroll
                    for (int m = 0; m < KPL; ++m) ss += kx[i][m] * kx[i][m];
                    ss = warp_sum(ss);
                    const float r = 1.0f / sqrtf(ss + P.l2_eps);
                    if (j < W) {
#pragma unroll
                        for (int m = 0; m < KPL; ++m)
                            if (lane + 32 * m < K) Xs[j * K + lane + 32 * m] = kx[i][m] * r;
                    }
                }
            }
            if (KDA) {
                for (int idx = tid; idx < W * K; idx += kFoldThreads) {
                    const int j = idx / K, kk = idx - j * K;
                    alpha[idx] = expf(ring_g[(sh_hv * L + ring_pos(base, j, L)) * K + kk]);
                }
            } else {
                for (int j = tid; j < W; j += kFoldThreads)
                    alpha[j] = expf(ring_g[sh_hv * L + ring_pos(base, j, L)]);
            }
            for (int j = tid; j < W; j += kFoldThreads)
                betaS[j] = ring_beta[sh_hv * L + ring_pos(base, j, L)];
            {
                const int r = tid & (kFoldRows - 1), jq = tid / kFoldRows;  // 4 record lanes
                const int vr = v0 + r;
                constexpr int kVals = kFoldMaxL / (kFoldThreads / kFoldRows);  // 32
                float x[kVals];
#pragma unroll
                for (int i = 0; i < kVals; ++i) {
                    const int j = jq + 4 * i;
                    x[i] = (j < W && vr < V)
                               ? to_f32<IO>(rawv[(sh_hv * L + ring_pos(base, j, L)) * V + vr])
                               : 0.0f;
                }
#pragma unroll
                for (int i = 0; i < kVals; ++i) {
                    const int j = jq + 4 * i;
                    if (j < W) vv[j * kFoldRows + r] = x[i];
                }
            }
            __syncthreads();

            // replay: thread (row r, part) holds state columns 4 (part + 4 m) .. + 3
            const int r = tid >> 2, part = tid & 3;
            const int vr = v0 + r;
            const bool valid = vr < V;
            const int K4 = K / 4;
            float4 S[KC];
            float4 *row = reinterpret_cast<float4 *>(ckpt + (sh_hv * V + (valid ? vr : 0)) * K);
#pragma unroll
            for (int m = 0; m < KC; ++m) {
                const int c4 = part + 4 * m;
                S[m] = (valid && c4 < K4) ? row[c4] : make_float4(0.f, 0.f, 0.f, 0.f);
            }
            for (int t = 0; t < W; ++t) {
                const float4 *xk = reinterpret_cast<const float4 *>(Xs + t * K);
                float4 u4 = make_float4(0.f, 0.f, 0.f, 0.f);
                if (KDA) {
                    const float4 *al = reinterpret_cast<const float4 *>(alpha + (size_t)t * K);
#pragma unroll
                    for (int m = 0; m < KC; ++m) {
                        const int c4 = part + 4 * m;
                        if (c4 < K4) {
                            const float4 a4 = al[c4], x4 = xk[c4];
                            S[m].x *= a4.x; S[m].y *= a4.y; S[m].z *= a4.z; S[m].w *= a4.w;
                            u4.x = fmaf(S[m].x, x4.x, u4.x); u4.y = fmaf(S[m].y, x4.y, u4.y);
                            u4.z = fmaf(S[m].z, x4.z, u4.z); u4.w = fmaf(S[m].w, x4.w, u4.w);
                        }
                    }
                } else {
                    const float al = alpha[t];
#pragma unroll
                    for (int m = 0; m < KC; ++m) {
                        const int c4 = part + 4 * m;
                        if (c4 < K4) {
                            const float4 x4 = xk[c4];
                            S[m].x *= al; S[m].y *= al; S[m].z *= al; S[m].w *= al;
                            u4.x = fmaf(S[m].x, x4.x, u4.x); u4.y = fmaf(S[m].y, x4.y, u4.y);
                            u4.z = fmaf(S[m].z, x4.z, u4.z); u4.w = fmaf(S[m].w, x4.w, u4.w);
                        }
                    }
                }
                float u = (u4.x + u4.y) + (u4.z + u4.w);
                u += __shfl_xor_sync(0xffffffffu, u, 1);
                u += __shfl_xor_sync(0xffffffffu, u, 2);
                const float d = betaS[t] * (vv[t * kFoldRows + r] - u);
#pragma unroll
                for (int m = 0; m < KC; ++m) {
                    const int c4 = part + 4 * m;
                    if (c4 < K4) {
                        const float4 x4 = xk[c4];
                        S[m].x = fmaf(d, x4.x, S[m].x); S[m].y = fmaf(d, x4.y, S[m].y);
                        S[m].z = fmaf(d, x4.z, S[m].z); S[m].w = fmaf(d, x4.w, S[m].w);
                    }
                }
            }
            if (valid) {
#pragma unroll
                for (int m = 0; m < KC; ++m) {
                    const int c4 = part + 4 * m;
                    if (c4 < K4) row[c4] = S[m];
                }
            }
            __syncthreads();  // the item's buffers are reused by the next item
        }
        item_base += nitems;
        __syncthreads();  // the row list is rebuilt by the next pass
    }
}

template <typename IO, bool KDA>
static cudaError_t launch_fold_typed(const LayerArgs &P, const FoldLayers &FL, int n_layers,
                                     const CursorArgs &C, const int32_t *slot_idx, int B,
                                     cudaStream_t stream) {
    const size_t smem = fold_smem_bytes(P.K, P.L, KDA);
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const int grid = 2 * sms;
#define GDN_FOLD_LAUNCH(KCV)                                                                   \
    do {                                                                                       \
        auto kern = fold_kernel<IO, KDA, KCV>;                                                 \
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem); \
        if (e != cudaSuccess) return e;                                                        \
        kern<<<grid, kFoldThreads, smem, stream>>>(P, FL, n_layers, C, slot_idx, B);           \
    } while (0)
    if (P.K <= 32) GDN_FOLD_LAUNCH(2);
    else if (P.K <= 64) GDN_FOLD_LAUNCH(4);
    else if (P.K <= 128) GDN_FOLD_LAUNCH(8);
    else GDN_FOLD_LAUNCH(16);
#undef GDN_FOLD_LAUNCH
    return cudaGetLastError();
}

bool fold_supported(int K, int L) { return K <= 256 && L <= kFoldMaxL; }

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
