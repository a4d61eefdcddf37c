// cursors.cu -- device-side cursor arithmetic (commit, fold's cursor move,
// reset).  Pure integer work on [num_slots] arrays, read and written on the
// device so the whole decode step stays capturable in a CUDA graph (blog post
// on sglang PR #28695, §1.3 and appendix A.2).  The commit and the cursor move
// are launched dependent on the kernel before them (launch_setup.cuh): each
// waits on that grid before reading anything and lets the next kernel start
// its launch right after.
#include "common.cuh"
#include "launch_setup.cuh"

namespace gdnspec {

constexpr int kCursorThreads = 256;

// commit: write_pos += accept_len; is_flush = (write_pos + 2T > L)  (blog §4.2, §8.1-8.2).
// A row whose cursors are out of range (write_pos outside [0, L] or cache_base
// outside [0, L), as row_cursor_ok rejects them) is skipped with CURSOR_CORRUPT.
__global__ void commit_kernel(CursorArgs C, int T, int L, const int32_t *__restrict__ slot_idx,
                              int B, const int32_t *__restrict__ accept_len) {
    grid_dep_wait();   // the verify that read these cursors
    grid_dep_launch();
    for (int bb = blockIdx.x * blockDim.x + threadIdx.x; bb < B; bb += gridDim.x * blockDim.x) {
        const int slot = slot_idx[bb];
        if (slot < 0) continue;
        if (slot >= C.num_slots) { atomicOr(C.status, GDN_SPEC_ST_SLOT_OOR); continue; }
        const int acc = accept_len[bb];
        if (acc < 0 || acc > T) { atomicOr(C.status, GDN_SPEC_ST_ACCEPT_RANGE); continue; }
        const int wp0 = C.write_pos[slot], base = C.cache_base[slot];
        if (wp0 < 0 || wp0 > L || base < 0 || base >= L) {
            atomicOr(C.status, GDN_SPEC_ST_CURSOR_CORRUPT);
            continue;
        }
        const int wp = wp0 + acc;
        C.write_pos[slot] = wp;
        C.is_flush[slot] = (wp + 2 * T > L) ? 1 : 0;
    }
}

// after the fold of every layer: cache_base = (cache_base + write_pos) & (L-1),
// write_pos = 0, is_flush = 0, for the rows whose is_flush was set.  A row the
// fold could not finish (a bounded wait ran out; the fold kernel marked it with
// is_flush = kFoldFailed) is poisoned instead: write_pos = -1, so that every
// later call reports CURSOR_CORRUPT for it until gdn_spec_reset.
__global__ void fold_cursor_kernel(CursorArgs C, int L, const int32_t *__restrict__ slot_idx, int B) {
    grid_dep_wait();   // the fold that read these cursors
    grid_dep_launch();
    for (int bb = blockIdx.x * blockDim.x + threadIdx.x; bb < B; bb += gridDim.x * blockDim.x) {
        const int slot = slot_idx[bb];
        if (slot < 0) continue;
        if (slot >= C.num_slots) { atomicOr(C.status, GDN_SPEC_ST_SLOT_OOR); continue; }
        const int flag = C.is_flush[slot];
        if (!flag) continue;
        if (flag == kFoldFailed) {
            C.write_pos[slot] = -1;
            C.is_flush[slot] = 0;
            continue;
        }
        const int wp = C.write_pos[slot], base = C.cache_base[slot];
        if (wp < 0 || wp > L || base < 0 || base >= L) {
            atomicOr(C.status, GDN_SPEC_ST_CURSOR_CORRUPT);
            continue;
        }
        C.cache_base[slot] = ring_pos(base, wp, L);
        C.write_pos[slot] = 0;
        C.is_flush[slot] = 0;
    }
}

// prefill -> decode handoff: write_pos = cache_base = 0, is_flush = 0
__global__ void reset_kernel(CursorArgs C, const int32_t *__restrict__ slot_idx, int B) {
    for (int bb = blockIdx.x * blockDim.x + threadIdx.x; bb < B; bb += gridDim.x * blockDim.x) {
        const int slot = slot_idx[bb];
        if (slot < 0) continue;
        if (slot >= C.num_slots) { atomicOr(C.status, GDN_SPEC_ST_SLOT_OOR); continue; }
        C.write_pos[slot] = 0;
        C.cache_base[slot] = 0;
        C.is_flush[slot] = 0;
    }
}

static int cursor_blocks(int B) {
    int nb = (B + kCursorThreads - 1) / kCursorThreads;
    return nb < 1 ? 1 : (nb > 64 ? 64 : nb);
}

cudaError_t launch_commit(const CursorArgs &C, int T, int L, const int32_t *slot_idx, int B,
                          const int32_t *accept_len, cudaStream_t stream) {
    return launch_dependent(commit_kernel, dim3(cursor_blocks(B)), dim3(kCursorThreads), 0, stream, C, T, L,
                            slot_idx, B, accept_len);
}

cudaError_t launch_fold_cursors(const CursorArgs &C, int L, const int32_t *slot_idx, int B,
                                cudaStream_t stream) {
    return launch_dependent(fold_cursor_kernel, dim3(cursor_blocks(B)), dim3(kCursorThreads), 0, stream, C, L,
                            slot_idx, B);
}

cudaError_t launch_reset(const CursorArgs &C, const int32_t *slot_idx, int B, cudaStream_t stream) {
    reset_kernel<<<cursor_blocks(B), kCursorThreads, 0, stream>>>(C, slot_idx, B);
    return cudaGetLastError();
}

}  // namespace gdnspec
