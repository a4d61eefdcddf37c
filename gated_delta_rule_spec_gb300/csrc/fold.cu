// fold.cu -- exact fold of the committed ring history into the checkpoint.
//
// sglang PR #28695 replaced the chunked (I+A)^{-1} flush, which is
// ill-conditioned and let long outputs drift, by a closed-loop fold that
// replays the raw (v, k, g, beta) records with the recurrence itself (blog
// post on PR #28695, §12.5-12.7; prhub summary of PR #28695, implementation
// item 3).  This kernel does exactly that, in fp32, token by token:
//     S <- exp(g_t) S   (KDA: S diag(exp(g_t)))
//     d  = beta_t (v_t - S k^_t),   S <- S + d k^_t^T
//
// Rows of S are independent under the recurrence (row i only sees v_t[i]).
// A group of eight threads holds four state rows, each thread an eighth of
// their K columns (at K = 32 four threads and a quarter), so every key value
// it reads from shared memory serves four rows.  The four rows' dot products
// are reduced over the group by a reduce-scatter: two shuffles split the
// rows between the threads (each keeps two rows' sums, then one), a third
// finishes the sum (at K = 32 the two splits do), each thread computes the
// delta of the row it ends with, and four shuffles hand the deltas to the
// group.  The keys stay in shared
// memory as the raw I/O-dtype records (bf16: half the bytes of fp32) and are
// widened in registers: per record and state row this reads 64 bytes of
// keys.  The elementwise work uses Blackwell's packed fp32x2 instructions.
//
// With one gate per (token, v-head) the decay is carried as a running scalar
// instead of being applied to every element: S = gam * R with gam the product
// of the decays so far, so a record costs a dot product and a rank-1 update of
// R and nothing else:
//     gam <- gam * exp(g_t),  u = R k^_t,  R <- R + beta_t (v_t / gam - u) k^_t^T
// (since exp(g_t) S_{t-1} = gam_t R_{t-1}).  When gam drops below 2^-32 it is
// multiplied into R and reset to 1, which keeps every value in range; the
// stored checkpoint is gam * R.  This is the same recurrence, record by
// record, with the decay multiplications moved, not a chunked form.
//
// Only the rows whose is_flush is set do any work, and in steady state that
// is a small share of the batch per step.  So the grid is persistent: every
// CTA scans the batch's flags, builds the same compact list of slots to
// fold, and takes work items (row, layer, v-head, block of 32 state rows; 64
// with per-channel decays) round-robin from it.  The kernel is launched
// dependent on the commit before it in the stream and waits on that grid
// before its first global access.  An item's keys (one or two contiguous ring segments)
// and values (one short run per record) arrive by bulk asynchronous copies
// on an mbarrier while the CTA reads the gates and loads its state rows into
// registers.  Folding runs after sampling, outside the forward, so the
// layers are independent here and one launch folds all of them (the blog's
// §2.1 observation about replay outside the forward).  The cursors move in
// a separate launch after every layer.
//
// When a bounded wait runs out, the item's row is marked (is_flush =
// kFoldFailed) and the CTA goes on; the cursor move then poisons that row
// instead of moving it, since some of its layers and v-heads may be folded
// and others not.
#include "common.cuh"
#include "launch_setup.cuh"
#include "ptx_sm100.cuh"
#include "replay.cuh"

namespace gdnspec {

constexpr int kFoldMaxL = 128;                        // ring length limit of this kernel

// Threads per group of four state rows: eight at K >= 64, four at K = 32.
// An item has 64 threads with one gate per (token, v-head): 32 state rows at
// K >= 64 (small items spread a step's few flagged rows over the SMs); with
// per-channel decays 128 threads and 64 rows, so that the item's fp32 decay
// table [L][K] serves twice the rows and a step's items fit on the SMs at
// once.  The flag scan takes kFoldScanPer batch rows per thread.
constexpr int kFoldScanPer = 4;   // batch rows per thread and flag-scan pass

template <int K, bool KDA>
struct FoldGeom {
    static constexpr int Threads = KDA ? 128 : 64;
    static constexpr int TPR = K >= 64 ? 8 : 4;
    static constexpr int RPT = 4;                     // state rows per thread
    static constexpr int Groups = Threads / TPR;
    static constexpr int Rows = RPT * Groups;         // state rows per work item
    static constexpr int CtasPerSm = KDA ? 4 : 8;
};

__host__ __device__ constexpr size_t fold_pad16(size_t bytes) { return (bytes + 15) & ~(size_t)15; }

// Shared memory of one item (every region starts on 16 bytes): raw keys
// [L][K] and raw values [L][rows of the item] in the I/O dtype, then fp32 (alpha,
// 1/alpha) [L] (KDA: alpha [L][K]), beta [L], 1/|k| [L], and the compacted
// slot list with its cursors.
struct FoldSmem {
    size_t keys, vals, alpha, beta, rs, rows, meta, total;
    __host__ __device__ FoldSmem(int K, int L, bool kda, size_t io) {
        const int item_rows = K >= 64 ? (kda ? FoldGeom<128, true>::Rows : FoldGeom<128, false>::Rows)
                                      : (kda ? FoldGeom<32, true>::Rows : FoldGeom<32, false>::Rows);
        const int scan = kFoldScanPer * (kda ? FoldGeom<128, true>::Threads : FoldGeom<128, false>::Threads);
        keys = 0;
        vals = keys + fold_pad16((size_t)L * K * io);
        alpha = vals + fold_pad16((size_t)L * item_rows * io);
        beta = alpha + fold_pad16(sizeof(float) * (size_t)L * (kda ? K : 2));
        rs = beta + fold_pad16(sizeof(float) * L);
        rows = rs + fold_pad16(sizeof(float) * L);
        meta = rows + sizeof(int) * scan;
        total = meta + sizeof(int) * scan;
    }
};

size_t fold_smem_bytes(int K, int L, bool kda, bool bf16) {
    return FoldSmem(K, L, kda, bf16 ? 2 : 4).total;
}

template <typename IO, bool KDA, int K>
__global__ void __launch_bounds__(FoldGeom<K, KDA>::Threads, FoldGeom<K, KDA>::CtasPerSm)
fold_kernel(LayerArgs P, FoldLayers FL, int n_layers, CursorArgs C,
            const int32_t *__restrict__ slot_idx, int B, uint32_t wait_limit) {
    static_assert(K % 32 == 0 && K <= 128, "whole 16-byte key chunks per thread");
    using KC = KeyChunk<IO>;
    constexpr int kFoldThreads = FoldGeom<K, KDA>::Threads;
    constexpr int kFoldScan = kFoldScanPer * kFoldThreads;   // batch rows per scan pass
    constexpr int kFoldTPR = FoldGeom<K, KDA>::TPR;
    constexpr int kGroups = FoldGeom<K, KDA>::Groups;
    constexpr int kRPT = FoldGeom<K, KDA>::RPT;
    constexpr int kFoldRows = FoldGeom<K, KDA>::Rows;
    constexpr int kPer = KC::kVals;                 // key values per 16-byte chunk
    constexpr int kNC = K / kPer / kFoldTPR;        // chunks per thread: chunk part + TPR m
    constexpr int kNP = kNC * kPer / 2;             // float2 pairs per thread and row
    static_assert(kNC >= 1, "at least one chunk per thread");
    extern __shared__ __align__(16) uint8_t smem[];
    __shared__ int s_count, s_warp_off[kFoldScanPer][kFoldThreads / 32];
    __shared__ __align__(8) uint64_t s_bar;
    const int V = P.V, L = P.L, HV = P.HV, H = P.H;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const FoldSmem lay(K, L, KDA, sizeof(IO));
    IO *Xk = reinterpret_cast<IO *>(smem + lay.keys);      // [L][K]
    IO *Xv = reinterpret_cast<IO *>(smem + lay.vals);      // [L][kFoldRows]
    float *alpha = reinterpret_cast<float *>(smem + lay.alpha);
    float *betaS = reinterpret_cast<float *>(smem + lay.beta);
    float *rsS = reinterpret_cast<float *>(smem + lay.rs);
    int *rows = reinterpret_cast<int *>(smem + lay.rows);
    int *meta = reinterpret_cast<int *>(smem + lay.meta);
    const uint32_t bar = ptx::smem_addr(&s_bar);
    const int vblocks = (V + kFoldRows - 1) / kFoldRows;
    const int per_row = n_layers * HV * vblocks;
    const int grp = tid / kFoldTPR, part = tid % kFoldTPR;
    // the dot products of the group's four rows are reduced over its TPR
    // threads by splitting on two bits of part (S1, S0): each thread ends with
    // the full sum of row 2 h1 + h0 and computes that row's delta
    constexpr int S1 = kFoldTPR == 8 ? 2 : 1, S0 = S1 - 1;
    const int h1 = (part >> S1) & 1, h0 = (part >> S0) & 1;
    const int own = 2 * h1 + h0;
    const int lane_base = lane & ~(kFoldTPR - 1);
    long long item_base = 0;  // items enumerated in earlier scan passes
    uint32_t phase = 0;
    // set when a drain wait ran out too: copies may still land in the buffers,
    // so the CTA only marks the rows of its remaining items as failed
    bool dead = false;

    if (tid == 0) {
        ptx::mbar_init(bar, 1);
        ptx::mbar_init_fence();
    }
    grid_dep_wait();   // the commit's flags and cursors (the cursor move starts as this grid exits)
    __syncthreads();

    for (int b0 = 0; b0 < B; b0 += kFoldScan) {
        // ---- scan kFoldScan batch rows, compact the flagged ones (same list in
        //      every CTA, ordered by (k, warp, lane)); a row's flag and cursors
        //      are read together, every load of the pass before any is used
        int slot[kFoldScanPer], fl[kFoldScanPer], wp[kFoldScanPer], base[kFoldScanPer];
#pragma unroll
        for (int k = 0; k < kFoldScanPer; ++k) {
            const int bb = b0 + k * kFoldThreads + tid;
            slot[k] = bb < B ? slot_idx[bb] : -1;
        }
#pragma unroll
        for (int k = 0; k < kFoldScanPer; ++k) {
            fl[k] = wp[k] = base[k] = 0;
            if (slot[k] >= 0 && slot[k] < C.num_slots) {
                fl[k] = C.is_flush[slot[k]];
                wp[k] = C.write_pos[slot[k]];
                base[k] = C.cache_base[slot[k]];
            }
        }
        unsigned ball[kFoldScanPer];
#pragma unroll
        for (int k = 0; k < kFoldScanPer; ++k) {
            fl[k] = (fl[k] && wp[k] > 0 && wp[k] <= L && base[k] >= 0 && base[k] < L) ? 1 : 0;
            ball[k] = __ballot_sync(0xffffffffu, fl[k]);
            if (lane == 0) s_warp_off[k][warp] = __popc(ball[k]);
        }
        __syncthreads();
        if (tid == 0) {
            int acc = 0;
            for (int k = 0; k < kFoldScanPer; ++k)
                for (int w = 0; w < kFoldThreads / 32; ++w) {
                    const int c = s_warp_off[k][w];
                    s_warp_off[k][w] = acc;
                    acc += c;
                }
            s_count = acc;
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < kFoldScanPer; ++k)
            if (fl[k]) {
                const int pos = s_warp_off[k][warp] + __popc(ball[k] & ((1u << lane) - 1u));
                rows[pos] = slot[k];
                meta[pos] = (wp[k] << 16) | base[k];
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
            const int slot_e = rows[e];
            const int W = meta[e] >> 16, base_e = meta[e] & 0xFFFF;
            const int row0 = vbk * kFoldRows;
            const int nrows = V - row0 < kFoldRows ? V - row0 : kFoldRows;   // a multiple of 8
            const size_t sh_hv = (size_t)slot_e * HV + hv, sh_h = (size_t)slot_e * H + h;
            const IO *rawk = reinterpret_cast<const IO *>(FL.rawk[li]);
            const IO *rawv = reinterpret_cast<const IO *>(FL.rawv[li]);
            const float *ring_g = FL.ring_g[li];
            const float *ring_beta = FL.ring_beta[li];
            float *ckpt = FL.checkpoint[li];
            if (dead) {
                if (tid == 0) C.is_flush[slot_e] = kFoldFailed;
                continue;
            }

            // ---- 1. keys and values by bulk copies (warp 0): the keys are one
            //         or two contiguous ring segments, the values one run of
            //         nrows per record
            if (warp == 0) {
                const uint32_t kbytes = (uint32_t)(K * sizeof(IO)), vbytes = (uint32_t)(nrows * sizeof(IO));
                if (lane == 0) {
                    ptx::fence_proxy_async_smem();   // the previous item's generic reads come first
                    ptx::mbar_expect_tx(bar, (uint32_t)W * (kbytes + vbytes));
                    const int n1 = (L - base_e) < W ? (L - base_e) : W;
                    ptx::bulk_copy_g2s(ptx::smem_addr(Xk), rawk + (sh_h * L + base_e) * K, n1 * kbytes, bar);
                    if (W > n1)
                        ptx::bulk_copy_g2s(ptx::smem_addr(Xk + (size_t)n1 * K), rawk + sh_h * L * K,
                                           (W - n1) * kbytes, bar);
                }
                __syncwarp();
                for (int j = lane; j < W; j += 32)
                    ptx::bulk_copy_g2s(ptx::smem_addr(Xv + (size_t)j * kFoldRows),
                                       rawv + (sh_hv * L + ring_pos(base_e, j, L)) * V + row0, vbytes, bar);
            }
            // ---- 2. this thread's four state rows (loads issued first: their latency
            //         overlaps the gate loads below and the copies)
            float2 S[kRPT][kNP];
#pragma unroll
            for (int rr = 0; rr < kRPT; ++rr) {
#pragma unroll
                for (int i = 0; i < kNP; ++i) S[rr][i] = make_float2(0.f, 0.f);
                if (grp + kGroups * rr < nrows) {
                    const float *srow = ckpt + (sh_hv * V + row0 + grp + kGroups * rr) * K;
#pragma unroll
                    for (int m = 0; m < kNC; ++m) {
                        const float4 *src = reinterpret_cast<const float4 *>(srow + (part + kFoldTPR * m) * kPer);
#pragma unroll
                        for (int q = 0; q < kPer / 4; ++q) {
                            const float4 f = src[q];
                            S[rr][m * (kPer / 2) + 2 * q] = make_float2(f.x, f.y);
                            S[rr][m * (kPer / 2) + 2 * q + 1] = make_float2(f.z, f.w);
                        }
                    }
                }
            }
            // ---- 2'. gates (thread per record); their loads are in flight with the state rows'
            for (int j = tid; j < W; j += kFoldThreads) {
                const int p = ring_pos(base_e, j, L);
                if (!KDA) {
                    const float gj = ring_g[sh_hv * L + p];
                    reinterpret_cast<float2 *>(alpha)[j] = make_float2(expf(gj), expf(-gj));
                }
                betaS[j] = ring_beta[sh_hv * L + p];
            }
            if (KDA) {
                for (int idx = tid; idx < W * K; idx += kFoldThreads) {
                    const int j = idx / K, kk = idx - j * K;
                    alpha[idx] = expf(ring_g[(sh_hv * L + ring_pos(base_e, j, L)) * K + kk]);
                }
            }
            // ---- 3. the copies land; 1 / |k_t| for every record (two threads each)
            const bool landed = ptx::mbar_wait(bar, phase, wait_limit);
            phase ^= 1u;
            if (__syncthreads_or(!landed)) {   // the same decision in every thread
                // record the failure and mark the row (its other items may be
                // folded already: the cursor move poisons it), give the copies
                // one more bounded wait so that none is still writing this
                // CTA's shared memory, and go on with the next item.  The flag
                // stays non-zero, so every CTA still builds the same slot list.
                if (tid == 0) {
                    atomicOr(C.status, GDN_SPEC_ST_TIMEOUT);
                    C.is_flush[slot_e] = kFoldFailed;
                }
                const bool drained = ptx::mbar_wait(bar, phase ^ 1u, kWaitLimitDefault);
                if (__syncthreads_or(!drained)) dead = true;
                continue;
            }
            // 1 / |k_j| of the raw keys (two threads per record; the trip count
            // is the same in every thread: the shuffle is warp-wide)
            for (int j0 = 0; j0 < W; j0 += kFoldThreads / 2) {
                const int j = j0 + (tid >> 1);
                float ss = 0.0f;
                if (j < W) {
                    const uint4 *kr =
                        reinterpret_cast<const uint4 *>(Xk + (size_t)j * K) + (tid & 1) * (K / kPer / 2);
#pragma unroll
                    for (int c = 0; c < K / kPer / 2; ++c) {
                        float2 x[kPer / 2];
                        KC::widen(kr[c], x);
#pragma unroll
                        for (int i = 0; i < kPer / 2; ++i) ss = fmaf(x[i].y, x[i].y, fmaf(x[i].x, x[i].x, ss));
                    }
                }
                ss += __shfl_xor_sync(0xffffffffu, ss, 1);
                if (j < W && (tid & 1) == 0) rsS[j] = 1.0f / sqrtf(ss + P.l2_eps);
            }
            __syncthreads();

            // ---- 4. replay (decay, then the delta against the decayed state)
            // this thread's chunks of key t, widened
            auto load_key = [&](int t, float2 (&x)[kNP]) {
                const uint4 *xk = reinterpret_cast<const uint4 *>(Xk + (size_t)t * K);
#pragma unroll
                for (int m = 0; m < kNC; ++m) {
                    float2 c2[kPer / 2];
                    KC::widen(xk[part + kFoldTPR * m], c2);
#pragma unroll
                    for (int i = 0; i < kPer / 2; ++i) x[m * (kPer / 2) + i] = c2[i];
                }
            };
            // S x for the group's four rows, reduced over the group's threads;
            // returns the full dot product of this thread's own row.  The first
            // split keeps rows 2 h1, 2 h1 + 1 and sends the other two, the
            // second keeps row 2 h1 + h0; the remaining bits sum what is left.
            auto dot_own = [&](const float2 (&x)[kNP]) {
                float u[kRPT];
#pragma unroll
                for (int rr = 0; rr < kRPT; ++rr) {
                    float2 acc[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
                    for (int i = 0; i < kNP; ++i) acc[i & 1] = __ffma2_rn(S[rr][i], x[i], acc[i & 1]);
                    const float2 a2 = __fadd2_rn(acc[0], acc[1]);
                    u[rr] = a2.x + a2.y;
                }
                float k0 = h1 ? u[2] : u[0], k1 = h1 ? u[3] : u[1];
                const float s0 = h1 ? u[0] : u[2], s1 = h1 ? u[1] : u[3];
                k0 += __shfl_xor_sync(0xffffffffu, s0, 1 << S1);
                k1 += __shfl_xor_sync(0xffffffffu, s1, 1 << S1);
                float uo = h0 ? k1 : k0;
                uo += __shfl_xor_sync(0xffffffffu, h0 ? k0 : k1, 1 << S0);
#pragma unroll
                for (int o = 1; o < (1 << S0); o <<= 1) uo += __shfl_xor_sync(0xffffffffu, uo, o);
                return uo;
            };
            // S += d_rr x^T for the group's four rows, each row's delta from the
            // thread that owns it
            auto update = [&](float dow, const float2 (&x)[kNP]) {
#pragma unroll
                for (int rr = 0; rr < kRPT; ++rr) {
                    const float d = __shfl_sync(0xffffffffu, dow, lane_base | ((rr >> 1) << S1) | ((rr & 1) << S0));
                    const float2 d2 = make_float2(d, d);
#pragma unroll
                    for (int i = 0; i < kNP; ++i) S[rr][i] = __ffma2_rn(d2, x[i], S[rr][i]);
                }
            };
            const IO *vown = Xv + grp + kGroups * own;
            float gam = 1.0f, inv = 1.0f;   // scalar gate: S = gam R (every thread holds the same values)
            for (int t = 0; t < W; ++t) {
                float2 x[kNP];
                load_key(t, x);
                if (KDA) {
                    const float *al = alpha + (size_t)t * K;
#pragma unroll
                    for (int m = 0; m < kNC; ++m) {
                        const float4 *a4 = reinterpret_cast<const float4 *>(al + (part + kFoldTPR * m) * kPer);
#pragma unroll
                        for (int q = 0; q < kPer / 4; ++q) {
                            const float4 a = a4[q];
                            const int i = m * (kPer / 2) + 2 * q;
#pragma unroll
                            for (int rr = 0; rr < kRPT; ++rr) {
                                S[rr][i] = __fmul2_rn(S[rr][i], make_float2(a.x, a.y));
                                S[rr][i + 1] = __fmul2_rn(S[rr][i + 1], make_float2(a.z, a.w));
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
                        for (int rr = 0; rr < kRPT; ++rr)
#pragma unroll
                            for (int i = 0; i < kNP; ++i) S[rr][i] = __fmul2_rn(S[rr][i], g2);
                        gam = 1.0f;
                        inv = 1.0f;
                    }
                }
                const float uo = dot_own(x);
                const float rs = rsS[t], be = betaS[t];
                // KDA: S itself (inv stays 1); scalar gate: R, with v_t / gam
                update(be * (to_f32<IO>(vown[(size_t)t * kFoldRows]) * inv - rs * uo) * rs, x);
            }
            // ---- 5. S = gam R back into the checkpoint
            const float2 g2 = make_float2(gam, gam);
#pragma unroll
            for (int rr = 0; rr < kRPT; ++rr) {
                if (grp + kGroups * rr >= nrows) continue;
                float *drow = ckpt + (sh_hv * V + row0 + grp + kGroups * rr) * K;
#pragma unroll
                for (int m = 0; m < kNC; ++m) {
                    float4 *dst = reinterpret_cast<float4 *>(drow + (part + kFoldTPR * m) * kPer);
#pragma unroll
                    for (int q = 0; q < kPer / 4; ++q) {
                        const int i = m * (kPer / 2) + 2 * q;
                        const float2 a = KDA ? S[rr][i] : __fmul2_rn(S[rr][i], g2);
                        const float2 b = KDA ? S[rr][i + 1] : __fmul2_rn(S[rr][i + 1], g2);
                        dst[q] = make_float4(a.x, a.y, b.x, b.y);
                    }
                }
            }
            __syncthreads();  // the item's buffers are reused by the next item
        }
        item_base += nitems;
        __syncthreads();  // the slot list is rebuilt by the next pass
    }
}

template <typename IO, bool KDA, int K>
static cudaError_t launch_fold_k(const LayerArgs &P, const FoldLayers &FL, int n_layers,
                                 const CursorArgs &C, const int32_t *slot_idx, int B,
                                 cudaStream_t stream) {
    const size_t smem = FoldSmem(K, P.L, KDA, sizeof(IO)).total;
    auto kern = fold_kernel<IO, KDA, K>;
    static KernelSetup setup;
    int sms = 0;
    cudaError_t e = kernel_setup(setup, reinterpret_cast<const void *>(kern), smem, &sms);
    if (e != cudaSuccess) return e;
    // enough CTAs for every item of a typical step to run at once; the ones
    // without an item leave after the flag scan
    using FG = FoldGeom<K, KDA>;
    return launch_dependent(kern, dim3(FG::CtasPerSm * sms), dim3(FG::Threads), smem, stream, P, FL, n_layers, C,
                            slot_idx, B, data_wait_limit());
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
