// common.cuh -- device helpers and by-value kernel parameters shared by the
// libgdnspec kernels.  The math follows the GDN recurrence of sglang PR
// #28695 "[GDN] Support ReplaySSM Ring Spec-Verify" and the blog post that
// explains it ("PR #28695 详解", §12.1): g = -exp(A_log) softplus(a + dt_bias),
// beta = sigmoid(b), decay first and then the delta against the decayed state.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include "gdn_spec.h"

namespace gdnspec {

// Everything a kernel needs about one layer, passed by value.
struct LayerArgs {
    int H, HV, G, K, V, T, L, num_slots;
    float scale, l2_eps;
    float *checkpoint;
    void *rawv, *rawk;
    float *ring_g, *ring_beta;
};

struct CursorArgs {
    int num_slots;
    int32_t *write_pos, *cache_base, *is_flush;
    uint32_t *status;
};

// is_flush value with which the fold marks a row it could not finish (a bounded
// wait ran out); its cursor move then poisons the row (write_pos = -1).
constexpr int kFoldFailed = 2;

// Default iteration limit of a bounded mbarrier wait (polls of at most about
// 256 ns each: 0.3 s at most).
constexpr uint32_t kWaitLimitDefault = 1u << 20;

// Iteration limit of the first wait on each data copy (verify's checkpoint
// tile, the fold's ring records, prefill's prompt chunks), set by
// gdn_spec_set_wait_limit; the waits that drain copies after a failure always
// use kWaitLimitDefault.
uint32_t data_wait_limit();

// Layers folded by one launch (the grid's z axis is layer * HV + v-head).
constexpr int kFoldMaxLayers = 48;
struct FoldLayers {
    float *checkpoint[kFoldMaxLayers];
    void *rawv[kFoldMaxLayers];
    void *rawk[kFoldMaxLayers];
    float *ring_g[kFoldMaxLayers];
    float *ring_beta[kFoldMaxLayers];
};

template <typename IO> __device__ __forceinline__ float to_f32(IO x);
template <> __device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) {
    return __bfloat162float(x);
}

template <typename IO> __device__ __forceinline__ IO from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// softplus with beta = 1 and the linear branch above 20
__device__ __forceinline__ float softplus_f(float x) {
    return x > 20.0f ? x : log1pf(expf(x));
}

// g = -exp(A_log) * softplus(a + dt_bias)
__device__ __forceinline__ float gate_g(float A_log, float a, float dt_bias) {
    return -expf(A_log) * softplus_f(a + dt_bias);
}

__device__ __forceinline__ float gate_beta(float b) {
    return 1.0f / (1.0f + expf(-b));
}

// Ring position of logical offset o from cache_base (L a power of two).
__device__ __forceinline__ int ring_pos(int base, int o, int L) { return (base + o) & (L - 1); }

// Validate a row's slot and cursors.  Returns true when the row is computed;
// otherwise *status_bits says why (0 for a padding row).
__device__ __forceinline__ bool row_cursor_ok(const CursorArgs &C, int slot, int T, int L,
                                              int *base, int *wp, uint32_t *status_bits) {
    *status_bits = 0;
    if (slot < 0) return false;
    if (slot >= C.num_slots) { *status_bits = GDN_SPEC_ST_SLOT_OOR; return false; }
    int w = C.write_pos[slot], bs = C.cache_base[slot];
    if (w < 0 || w > L || bs < 0 || bs >= L) { *status_bits = GDN_SPEC_ST_CURSOR_CORRUPT; return false; }
    if (w + T > L) { *status_bits = GDN_SPEC_ST_RING_OVERFLOW; return false; }
    *base = bs;
    *wp = w;
    return true;
}

}  // namespace gdnspec
