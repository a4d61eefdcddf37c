// verify_generic.cu -- CUDA-core verify kernel for any supported shape
// (fp32 or bf16 I/O, GDN or KDA gate, K in {32, 64, 128}, L <= 128).
//
// One CTA per (V-block of 128 rows, batch row, v-head); no layer axis, since
// layers are chain-dependent inside the forward (blog post on sglang PR
// #28695, §1.2).  The draft window's outputs come from the frozen checkpoint
// S0 and the ring history by the chunked UT transform (blog §12.3-12.4):
// with tokens j = 0..n-1 (W history records, then the T window tokens),
// alpha_j = exp(g_j), Gamma(i, r) = prod_{t=r+1..i} alpha_t and
// eG_j = prod_{t<=j} alpha_t (KDA: all per key channel),
//
//     A[i, r] = beta_i <k^_i, Gamma(i, r) k^_r>                 (r < i)
//     F[r, s] = <k^_r, Gamma(W+s, r) q^_s>                       (r <= W+s)
//     R_j     = beta_j (v_j - S0 (eG_j k^_j))
//     D = (I + A)^{-1} R,   o_s = S0 (eG_{W+s} q^_s) + sum_r F[r, s] d_r.
//
// The kernel applies (I + A)^{-1} from the output side instead of forming D:
// M = F^T (I + A)^{-1} (T x n, one backward substitution per window token),
// c[s, j] = M[s, j] beta_j, and
//
//     q_eff_s = eG_{W+s} q^_s - sum_j c[s, j] eG_j k^_j              (K-vector)
//     o_s     = scale * ( S0 q_eff_s + sum_j c[s, j] v_j ).
//
// Same result in exact arithmetic; the checkpoint is then read once, in a
// T-column product, and no n x V matrix is ever formed.  Decays are running
// products of per-token alpha (never exp of a difference of large prefix sums,
// never exp(-G)), so nothing overflows when cumulative decays reach -3000.
//
// The ring write is a side channel: window records go to positions
// (base + W + s) & (L-1), disjoint from the history positions the CTA reads,
// and hold the raw inputs (pre-normalisation k, v as given) plus the fp32 g
// and beta computed here.  rawk is written by one CTA per k-head (hv % G == 0,
// V-block 0), g and beta by V-block 0 (sglang PR #36821 ring-write placement).
#include "common.cuh"
#include "launch_setup.cuh"
#include "ptx_sm100.cuh"

namespace gdnspec {

constexpr int kGenThreads = 128;
constexpr int kGenMaxT = 16;

struct GenSmem {
    int KP;        // padded row length of X (floats)
    int L;
    int T;
    int K;
    bool kda;
    // offsets in floats
    size_t x, alpha, beta, A, F, c, qeff, total;
};

__host__ __device__ inline GenSmem gen_smem_layout(int K, int L, int T, bool kda) {
    GenSmem s;
    s.KP = K + 4;
    s.L = L;
    s.T = T;
    s.K = K;
    s.kda = kda;
    // every region starts on 16 bytes (a multiple of 4 floats): float4 reads
    auto up4 = [](size_t x) { return (x + 3) & ~(size_t)3; };
    size_t off = 0;
    s.x = off;     off = up4(off + (size_t)(L + T) * s.KP);   // rows: n keys then T queries (n <= L)
    s.alpha = off; off = up4(off + (size_t)L * (kda ? K : 1));
    s.beta = off;  off = up4(off + (size_t)L);
    s.A = off;     off = up4(off + (size_t)L * (L + 1));
    s.F = off;     off = up4(off + (size_t)T * L);
    s.c = off;     off = up4(off + (size_t)T * L);
    s.qeff = off;  off = up4(off + (size_t)T * K);
    s.total = off;
    return s;
}

size_t verify_generic_smem_bytes(int K, int L, int T, bool kda) {
    return gen_smem_layout(K, L, T, kda).total * sizeof(float);
}

template <typename IO, bool KDA>
__global__ void __launch_bounds__(kGenThreads)
verify_generic_kernel(LayerArgs P, CursorArgs C, const int32_t *__restrict__ slot_idx,
                      const IO *__restrict__ q, const IO *__restrict__ k,
                      const IO *__restrict__ v, const IO *__restrict__ a,
                      const IO *__restrict__ bgate, const float *__restrict__ A_log,
                      const float *__restrict__ dt_bias, IO *__restrict__ out) {
    extern __shared__ __align__(16) float sm[];
    __shared__ int s_slot, s_base, s_W, s_ok;

    const int vb = blockIdx.x, bb = blockIdx.y, hv = blockIdx.z;
    const int K = P.K, V = P.V, T = P.T, L = P.L, HV = P.HV, H = P.H;
    const int h = hv / P.G;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int v0 = vb * kGenThreads;
    const GenSmem lay = gen_smem_layout(K, L, T, KDA);
    float *X = sm + lay.x;
    float *alpha = sm + lay.alpha;
    float *betaS = sm + lay.beta;
    float *Am = sm + lay.A;
    float *Fm = sm + lay.F;
    float *cm = sm + lay.c;
    float *qeff = sm + lay.qeff;
    const int KP = lay.KP;
    const int LA = L + 1;  // row stride of A

    if (tid == 0) {
        int slot = slot_idx[bb], base = 0, W = 0;
        uint32_t st = 0;
        bool ok = row_cursor_ok(C, slot, T, L, &base, &W, &st);
        if (st && vb == 0 && hv == 0) atomicOr(C.status, st);
        s_slot = slot;
        s_base = base;
        s_W = W;
        s_ok = ok ? 1 : 0;
    }
    __syncthreads();
    const int vrow = v0 + tid;
    if (!s_ok) {
        if (vrow < V)
            for (int s = 0; s < T; ++s)
                out[(((size_t)bb * T + s) * HV + hv) * V + vrow] = from_f32<IO>(0.0f);
        return;
    }
    const int slot = s_slot, base = s_base, W = s_W;
    const int n = W + T;
    const size_t sh_hv = (size_t)slot * HV + hv;   // (slot, v-head) index
    const size_t sh_h = (size_t)slot * H + h;      // (slot, k-head) index
    const IO *rawk = reinterpret_cast<const IO *>(P.rawk);
    const IO *rawv = reinterpret_cast<const IO *>(P.rawv);
    IO *rawk_w = reinterpret_cast<IO *>(P.rawk);
    IO *rawv_w = reinterpret_cast<IO *>(P.rawv);
    const bool k_writer = (hv % P.G == 0) && vb == 0;
    if (tid == 0) {   // the history and the checkpoint tile into L2 now, ahead of their reads
        // the ring history is one or two contiguous segments of each array
        const int first = (L - base) < W ? (L - base) : W;
        if (first > 0)
            ptx::prefetch_l2(rawk + (sh_h * L + base) * K, (uint32_t)(first * K * sizeof(IO)));
        if (W > first) ptx::prefetch_l2(rawk + sh_h * L * K, (uint32_t)((W - first) * K * sizeof(IO)));
        if (KDA) {   // one gate per key channel: K floats per record
            if (first > 0) ptx::prefetch_l2(P.ring_g + (sh_hv * L + base) * K, (uint32_t)first * K * 4);
            if (W > first) ptx::prefetch_l2(P.ring_g + sh_hv * L * K, (uint32_t)(W - first) * K * 4);
        }
        const int rows = V - v0 < kGenThreads ? V - v0 : kGenThreads;
        ptx::prefetch_l2(P.checkpoint + (sh_hv * V + v0) * K, (uint32_t)rows * K * 4);
        if (V == kGenThreads) {   // whole v records are contiguous
            if (first > 0)
                ptx::prefetch_l2(rawv + (sh_hv * L + base) * V, (uint32_t)(first * V * sizeof(IO)));
            if (W > first) ptx::prefetch_l2(rawv + sh_hv * L * V, (uint32_t)((W - first) * V * sizeof(IO)));
        }
    }

    // ---- 1. keys (history + window) and window queries, L2-normalised into X.
    //         A warp takes four rows at a time (rows jb .. jb + 3) and issues the
    //         loads of all four before it uses any of them.
    {
        constexpr int kRows = 4, kPerLane = 4;   // K <= 128: four values per lane and row
        for (int jb = warp * kRows; jb < n + T; jb += kRows * (kGenThreads / 32)) {
            const IO *src[kRows];
            float xv[kRows][kPerLane];
#pragma unroll
            for (int rr = 0; rr < kRows; ++rr) {
                const int j = jb + rr;
                src[rr] = nullptr;
                if (j < W)
                    src[rr] = rawk + (sh_h * L + ring_pos(base, j, L)) * K;
                else if (j < n)
                    src[rr] = k + (((size_t)bb * T + (j - W)) * H + h) * K;
                else if (j < n + T)
                    src[rr] = q + (((size_t)bb * T + (j - n)) * H + h) * K;
            }
#pragma unroll
            for (int rr = 0; rr < kRows; ++rr)
#pragma unroll
                for (int c = 0; c < kPerLane; ++c) {
                    const int kk = lane + 32 * c;
                    xv[rr][c] = (src[rr] != nullptr && kk < K) ? to_f32<IO>(src[rr][kk]) : 0.0f;
                }
#pragma unroll
            for (int rr = 0; rr < kRows; ++rr) {
                const int j = jb + rr;
                if (j >= n + T) break;   // the same in every lane of the warp
                float ss = 0.0f;
#pragma unroll
                for (int c = 0; c < kPerLane; ++c) ss = fmaf(xv[rr][c], xv[rr][c], ss);
                ss = warp_sum(ss);
                const float r = 1.0f / sqrtf(ss + P.l2_eps);
#pragma unroll
                for (int c = 0; c < kPerLane; ++c) {
                    const int kk = lane + 32 * c;
                    if (kk < K) X[j * KP + kk] = xv[rr][c] * r;
                }
                if (j >= W && j < n && k_writer) {  // side channel: raw key, bitwise
                    IO *dst = rawk_w + (sh_h * L + ring_pos(base, j, L)) * K;
                    for (int kk = lane; kk < K; kk += 32) dst[kk] = src[rr][kk];
                }
            }
        }
    }
    // ---- 2. gates: history from the ring, window computed (and written to the ring)
    if (KDA) {   // n K gates: sixteen loads in flight per thread before any is used
        constexpr int kB = 16;
        for (int idx0 = tid; idx0 < n * K; idx0 += kB * kGenThreads) {
            float raw[kB];
#pragma unroll
            for (int u = 0; u < kB; ++u) {
                const int idx = idx0 + u * kGenThreads;
                const int j = idx / K, kk = idx - j * K;
                raw[u] = 0.0f;
                if (idx < n * K) {
                    if (j < W)
                        raw[u] = P.ring_g[(sh_hv * L + ring_pos(base, j, L)) * K + kk];
                    else
                        raw[u] = to_f32<IO>(a[(((size_t)bb * T + (j - W)) * HV + hv) * K + kk]);
                }
            }
#pragma unroll
            for (int u = 0; u < kB; ++u) {
                const int idx = idx0 + u * kGenThreads;
                if (idx < n * K) {
                    const int j = idx / K, kk = idx - j * K;
                    float g = raw[u];
                    if (j >= W) {
                        g = gate_g(A_log[hv], raw[u], dt_bias[(size_t)hv * K + kk]);
                        if (vb == 0) P.ring_g[(sh_hv * L + ring_pos(base, j, L)) * K + kk] = g;
                    }
                    alpha[j * K + kk] = expf(g);
                }
            }
        }
    } else {
        for (int j = tid; j < n; j += kGenThreads) {
            const int p = ring_pos(base, j, L);
            float g;
            if (j < W) {
                g = P.ring_g[sh_hv * L + p];
            } else {
                const size_t tok = (size_t)bb * T + (j - W);
                g = gate_g(A_log[hv], to_f32<IO>(a[tok * HV + hv]), dt_bias[hv]);
                if (vb == 0) P.ring_g[sh_hv * L + p] = g;
            }
            alpha[j] = expf(g);
        }
    }
    for (int j = tid; j < n; j += kGenThreads) {
        const int p = ring_pos(base, j, L);
        float be;
        if (j < W) {
            be = P.ring_beta[sh_hv * L + p];
        } else {
            const size_t tok = (size_t)bb * T + (j - W);
            be = gate_beta(to_f32<IO>(bgate[tok * HV + hv]));
            if (vb == 0) P.ring_beta[sh_hv * L + p] = be;
        }
        betaS[j] = be;
    }
    if (vrow < V) {  // side channel: raw values of this V-block, bitwise
        for (int s = 0; s < T; ++s)
            rawv_w[(sh_hv * L + ring_pos(base, W + s, L)) * V + vrow] =
                v[(((size_t)bb * T + s) * HV + hv) * V + vrow];
    }
    for (int idx = tid; idx < T * L; idx += kGenThreads) Fm[idx] = 0.0f;
    __syncthreads();

    // ---- 3. A and F: four threads per token row i (a quarter of K each)
    //         walk r down from i - 1 with the decay Gamma(i, r) as a running
    //         product; a window row i = W + s also forms F[s, r] against q^_s.
    //         Rows are interleaved over the warps (the triangle stays
    //         balanced) and every loop bound is the same in a warp, so the
    //         two-level shuffles of the dot products are warp-wide.
    {
        // a thread owns the 16-byte chunks part, part + 4, part + 8, ... of a
        // row (chunk c = channels 4c..4c+3): the four parts of a row read
        // consecutive chunks, so their shared-memory reads share no bank
        constexpr int KQ = 32;                 // channels per thread, K <= 128
        constexpr int KQ4 = KQ / 4;
        const int part = tid & 3, grp = tid >> 2;
        const int kq4 = K / 16;                // chunks per thread
        const float *Q = X + (size_t)n * KP;
        for (int pass = 0; pass * 32 < n; ++pass) {
            const int i = pass * 32 + (grp & 7) * 4 + warp;
            const bool live = i < n, win = live && i >= W;
            const int s = i - W;
            float xi[KQ], xq[KQ], c[KQ];
#pragma unroll
            for (int m = 0; m < KQ; ++m) {
                const bool in = (m >> 2) < kq4;
                const int ch = 4 * (part + 4 * (m >> 2)) + (m & 3);
                xi[m] = (in && live) ? X[i * KP + ch] : 0.0f;
                xq[m] = (in && win) ? Q[s * KP + ch] : 0.0f;
                c[m] = 1.0f;
            }
            float cs = 1.0f;
            {   // F[s, i] = <k^_i, q^_s> (Gamma = 1)
                float acc = 0.0f;
#pragma unroll
                for (int m = 0; m < KQ; ++m) acc = fmaf(xi[m], xq[m], acc);
                acc += __shfl_xor_sync(0xffffffffu, acc, 1);
                acc += __shfl_xor_sync(0xffffffffu, acc, 2);
                if (win && part == 0) Fm[s * L + i] = acc;
            }
            const float bi = live ? betaS[i] : 0.0f;
            const int top = min(pass * 32 + 28 + warp, n - 1);   // largest row of this warp
            for (int r = top - 1; r >= 0; --r) {
                const bool act = live && r < i;
                if (KDA) {
#pragma unroll
                    for (int m4 = 0; m4 < KQ4; ++m4) {
                        if (m4 < kq4) {
                            const float4 a4 = *reinterpret_cast<const float4 *>(alpha + (r + 1) * K + 4 * (part + 4 * m4));
                            c[4 * m4] *= act ? a4.x : 1.0f;
                            c[4 * m4 + 1] *= act ? a4.y : 1.0f;
                            c[4 * m4 + 2] *= act ? a4.z : 1.0f;
                            c[4 * m4 + 3] *= act ? a4.w : 1.0f;
                        }
                    }
                } else if (act) {
                    cs *= alpha[r + 1];
                }
                float acc = 0.0f, accq = 0.0f;
#pragma unroll
                for (int m4 = 0; m4 < KQ4; ++m4) {
                    if (m4 < kq4) {
                        const float4 x4 = *reinterpret_cast<const float4 *>(X + r * KP + 4 * (part + 4 * m4));
                        const float xs[4] = {x4.x, x4.y, x4.z, x4.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float w = c[4 * m4 + e] * xs[e];
                            acc = fmaf(xi[4 * m4 + e], w, acc);
                            accq = fmaf(xq[4 * m4 + e], w, accq);
                        }
                    }
                }
                acc += __shfl_xor_sync(0xffffffffu, acc, 1);
                accq += __shfl_xor_sync(0xffffffffu, accq, 1);
                acc += __shfl_xor_sync(0xffffffffu, acc, 2);
                accq += __shfl_xor_sync(0xffffffffu, accq, 2);
                if (act && part == 0) {
                    Am[i * LA + r] = bi * acc * cs;
                    if (win) Fm[s * L + r] = accq * cs;
                }
            }
        }
    }
    __syncthreads();

    // ---- 4. M = F^T (I + A)^{-1}: backward substitution, one warp per window token
    for (int s = warp; s < T; s += kGenThreads / 32) {
        float *f = Fm + s * L;
        for (int j = W + s; j >= 0; --j) {  // f_j = 0 beyond the causal limit W + s
            __syncwarp();
            const float m = f[j];
            if (lane == 0) cm[s * L + j] = m * betaS[j];
            for (int i = lane; i < j; i += 32) f[i] -= Am[j * LA + i] * m;
        }
        for (int j = W + s + 1 + lane; j < n; j += 32) cm[s * L + j] = 0.0f;
    }
    __syncthreads();

    // ---- 5. q_eff_s = eG_{W+s} q^_s - sum_j c[s, j] eG_j k^_j
    for (int kk = tid; kk < K; kk += kGenThreads) {
        for (int s = 0; s < T; ++s) {
            float e = 1.0f, acc = 0.0f;
            for (int j = 0; j <= W + s; ++j) {
                e *= KDA ? alpha[j * K + kk] : alpha[j];
                acc -= cm[s * L + j] * e * X[j * KP + kk];
            }
            acc += e * X[(n + s) * KP + kk];
            qeff[s * K + kk] = acc;
        }
    }
    __syncthreads();

    // ---- 6. o_s = scale (S0 q_eff_s + sum_j c[s, j] v_j) for this thread's row;
    //         global reads in batches (eight 16-byte checkpoint chunks, sixteen
    //         values), so that a batch costs one round trip
    if (vrow < V) {
        constexpr int kBatch = 8, kVBatch = 16;
        float acc[kGenMaxT];
#pragma unroll
        for (int s = 0; s < kGenMaxT; ++s) acc[s] = 0.0f;
        const float4 *srow =
            reinterpret_cast<const float4 *>(P.checkpoint + (sh_hv * V + vrow) * K);
        for (int k4 = 0; k4 < K / 4; k4 += kBatch) {   // K / 4 is a multiple of 8
            float4 sv[kBatch];
#pragma unroll
            for (int u = 0; u < kBatch; ++u) sv[u] = srow[k4 + u];
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
#pragma unroll
                for (int s = 0; s < kGenMaxT; ++s) {
                    if (s < T) {
                        const float4 qe = *reinterpret_cast<const float4 *>(qeff + s * K + 4 * (k4 + u));
                        acc[s] += sv[u].x * qe.x + sv[u].y * qe.y + sv[u].z * qe.z + sv[u].w * qe.w;
                    }
                }
            }
        }
        for (int j0 = 0; j0 < n; j0 += kVBatch) {
            float vj[kVBatch];
#pragma unroll
            for (int u = 0; u < kVBatch; ++u) {
                const int j = j0 + u;
                vj[u] = 0.0f;
                if (j < W)
                    vj[u] = to_f32<IO>(rawv[(sh_hv * L + ring_pos(base, j, L)) * V + vrow]);
                else if (j < n)
                    vj[u] = to_f32<IO>(v[(((size_t)bb * T + (j - W)) * HV + hv) * V + vrow]);
            }
#pragma unroll
            for (int u = 0; u < kVBatch; ++u) {
                if (j0 + u < n) {
#pragma unroll
                    for (int s = 0; s < kGenMaxT; ++s)
                        if (s < T) acc[s] += cm[s * L + j0 + u] * vj[u];
                }
            }
        }
#pragma unroll
        for (int s = 0; s < kGenMaxT; ++s)
            if (s < T)
                out[(((size_t)bb * T + s) * HV + hv) * V + vrow] = from_f32<IO>(P.scale * acc[s]);
    }
}

template <typename IO, bool KDA>
static cudaError_t launch_one(const LayerArgs &P, const CursorArgs &C, const int32_t *slot_idx,
                              int B, const void *q, const void *k, const void *v, const void *a,
                              const void *b, const float *A_log, const float *dt_bias, void *out,
                              cudaStream_t stream) {
    const size_t smem = verify_generic_smem_bytes(P.K, P.L, P.T, KDA);
    auto kern = verify_generic_kernel<IO, KDA>;
    static KernelSetup setup;
    int sms = 0;
    cudaError_t e = kernel_setup(setup, reinterpret_cast<const void *>(kern), smem, &sms);
    if (e != cudaSuccess) return e;
    dim3 grid((P.V + kGenThreads - 1) / kGenThreads, B, P.HV);
    kern<<<grid, kGenThreads, smem, stream>>>(
        P, C, slot_idx, static_cast<const IO *>(q), static_cast<const IO *>(k),
        static_cast<const IO *>(v), static_cast<const IO *>(a), static_cast<const IO *>(b),
        A_log, dt_bias, static_cast<IO *>(out));
    return cudaGetLastError();
}

cudaError_t launch_verify_generic(const LayerArgs &P, const CursorArgs &C, bool kda, bool bf16,
                                  const int32_t *slot_idx, int B, const void *q, const void *k,
                                  const void *v, const void *a, const void *b,
                                  const float *A_log, const float *dt_bias, void *out,
                                  cudaStream_t stream) {
    if (bf16) {
        return kda ? launch_one<__nv_bfloat16, true>(P, C, slot_idx, B, q, k, v, a, b, A_log,
                                                     dt_bias, out, stream)
                   : launch_one<__nv_bfloat16, false>(P, C, slot_idx, B, q, k, v, a, b, A_log,
                                                      dt_bias, out, stream);
    }
    return kda ? launch_one<float, true>(P, C, slot_idx, B, q, k, v, a, b, A_log, dt_bias, out,
                                         stream)
               : launch_one<float, false>(P, C, slot_idx, B, q, k, v, a, b, A_log, dt_bias, out,
                                          stream);
}

}  // namespace gdnspec
