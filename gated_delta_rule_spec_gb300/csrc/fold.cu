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
// Four threads share a row: each holds K/4 state values in registers and the
// row's dot product is reduced with two shuffles.  The grid has a layer axis:
// folding runs after sampling, outside the forward, so layers are independent
// there (the same observation as the blog's §2.1 on replay outside the
// forward).  The cursors move in a separate launch after every layer is done.
#include "common.cuh"

namespace gdnspec {

constexpr int kFoldThreads = 128;
constexpr int kFoldRows = kFoldThreads / 4;  // rows of S per CTA

size_t fold_smem_bytes(int K, int L, bool kda) {
    // keys [L][K], alpha [L] or [L][K], beta [L], values [L][kFoldRows]
    return sizeof(float) * ((size_t)L * K + (size_t)L * (kda ? K : 1) + L + (size_t)L * kFoldRows);
}

template <typename IO, bool KDA, int KC>
__global__ void __launch_bounds__(kFoldThreads)
fold_kernel(LayerArgs P, FoldLayers FL, CursorArgs C, const int32_t *__restrict__ slot_idx) {
    extern __shared__ __align__(16) float sm[];
    __shared__ int s_slot, s_base, s_W, s_ok;
    const int K = P.K, V = P.V, L = P.L, HV = P.HV, H = P.H;
    const int li = blockIdx.z / HV, hv = blockIdx.z - li * HV;
    const int h = hv / P.G;
    const int bb = blockIdx.y;
    const int v0 = blockIdx.x * kFoldRows;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    if (tid == 0) {
        int slot = slot_idx[bb];
        int ok = 0, W = 0, base = 0;
        if (slot >= 0 && slot < C.num_slots && C.is_flush[slot]) {
            W = C.write_pos[slot];
            base = C.cache_base[slot];
            ok = (W > 0 && W <= L && base >= 0 && base < L) ? 1 : 0;
        }
        s_slot = slot;
        s_base = base;
        s_W = W;
        s_ok = ok;
    }
    __syncthreads();
    if (!s_ok) return;
    const int slot = s_slot, base = s_base, W = s_W;
    const size_t sh_hv = (size_t)slot * HV + hv, sh_h = (size_t)slot * H + h;
    float *Xs = sm;                                  // [L][K]
    float *alpha = Xs + (size_t)L * K;               // [L] or [L][K]
    float *betaS = alpha + (size_t)L * (KDA ? K : 1);
    float *vv = betaS + L;                           // [L][kFoldRows]
    const IO *rawk = reinterpret_cast<const IO *>(FL.rawk[li]);
    const IO *rawv = reinterpret_cast<const IO *>(FL.rawv[li]);
    const float *ring_g = FL.ring_g[li];
    const float *ring_beta = FL.ring_beta[li];
    float *ckpt = FL.checkpoint[li];

    for (int j = warp; j < W; j += kFoldThreads / 32) {
        const IO *src = rawk + (sh_h * L + ring_pos(base, j, L)) * K;
        float ss = 0.0f;
        for (int kk = lane; kk < K; kk += 32) {
            float x = to_f32<IO>(src[kk]);
            Xs[j * K + kk] = x;
            ss += x * x;
        }
        ss = warp_sum(ss);
        const float r = 1.0f / sqrtf(ss + P.l2_eps);
        for (int kk = lane; kk < K; kk += 32) Xs[j * K + kk] *= r;
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
    for (int j = tid; j < W; j += kFoldThreads) betaS[j] = ring_beta[sh_hv * L + ring_pos(base, j, L)];
    for (int idx = tid; idx < W * kFoldRows; idx += kFoldThreads) {
        const int j = idx / kFoldRows, r = idx - j * kFoldRows;
        const int vr = v0 + r;
        vv[idx] = vr < V ? to_f32<IO>(rawv[(sh_hv * L + ring_pos(base, j, L)) * V + vr]) : 0.0f;
    }
    __syncthreads();

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
        float u = 0.0f;
        if (KDA) {
            const float4 *al = reinterpret_cast<const float4 *>(alpha + (size_t)t * K);
#pragma unroll
            for (int m = 0; m < KC; ++m) {
                const int c4 = part + 4 * m;
                if (c4 < K4) {
                    const float4 a4 = al[c4], x4 = xk[c4];
                    S[m].x *= a4.x; S[m].y *= a4.y; S[m].z *= a4.z; S[m].w *= a4.w;
                    u += S[m].x * x4.x + S[m].y * x4.y + S[m].z * x4.z + S[m].w * x4.w;
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
                    u += S[m].x * x4.x + S[m].y * x4.y + S[m].z * x4.z + S[m].w * x4.w;
                }
            }
        }
        u += __shfl_xor_sync(0xffffffffu, u, 1);
        u += __shfl_xor_sync(0xffffffffu, u, 2);
        const float d = betaS[t] * (vv[t * kFoldRows + r] - u);
#pragma unroll
        for (int m = 0; m < KC; ++m) {
            const int c4 = part + 4 * m;
            if (c4 < K4) {
                const float4 x4 = xk[c4];
                S[m].x += d * x4.x; S[m].y += d * x4.y; S[m].z += d * x4.z; S[m].w += d * x4.w;
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
}

template <typename IO, bool KDA>
static cudaError_t launch_fold_typed(const LayerArgs &P, const FoldLayers &FL, int n_layers,
                                     const CursorArgs &C, const int32_t *slot_idx, int B,
                                     cudaStream_t stream) {
    const size_t smem = fold_smem_bytes(P.K, P.L, KDA);
    dim3 grid((P.V + kFoldRows - 1) / kFoldRows, B, n_layers * P.HV);
    cudaError_t e;
#define GDN_FOLD_LAUNCH(KCV)                                                                   \
    do {                                                                                       \
        auto kern = fold_kernel<IO, KDA, KCV>;                                                 \
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem); \
        if (e != cudaSuccess) return e;                                                        \
        kern<<<grid, kFoldThreads, smem, stream>>>(P, FL, C, slot_idx);                        \
    } while (0)
    if (P.K <= 32) GDN_FOLD_LAUNCH(2);
    else if (P.K <= 64) GDN_FOLD_LAUNCH(4);
    else if (P.K <= 128) GDN_FOLD_LAUNCH(8);
    else GDN_FOLD_LAUNCH(16);
#undef GDN_FOLD_LAUNCH
    return cudaGetLastError();
}

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
