// replay.cuh -- pieces shared by the kernels that replay the recurrence token
// by token over state rows held in registers (fold, prefill).
#pragma once

#include <cstdint>

#include "common.cuh"

namespace gdnspec {

// 16 bytes of raw keys -> fp32 pairs (bf16: 8 values, fp32: 4)
template <typename IO> struct KeyChunk;
template <> struct KeyChunk<__nv_bfloat16> {
    static constexpr int kVals = 8;
    __device__ __forceinline__ static void widen(const uint4 &w, float2 (&x)[4]) {
        const uint32_t q[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)   // the low half is the element at the lower address
            x[i] = make_float2(__uint_as_float(q[i] << 16), __uint_as_float(q[i] & 0xFFFF0000u));
    }
};
template <> struct KeyChunk<float> {
    static constexpr int kVals = 4;
    __device__ __forceinline__ static void widen(const uint4 &w, float2 (&x)[2]) {
        x[0] = make_float2(__uint_as_float(w.x), __uint_as_float(w.y));
        x[1] = make_float2(__uint_as_float(w.z), __uint_as_float(w.w));
    }
};

}  // namespace gdnspec
