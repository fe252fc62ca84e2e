// Common device helpers for libmla: element types, the per-device error word, RoPE angles.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>
#include <math.h>

#include "mla.h"

namespace mla {

typedef __nv_bfloat16 bf16;

// Per-device error word (first error wins).  Read and cleared by mla_get_device_error().
__device__ int g_device_error = 0;
// Bounded-wait limit for spin loops in nanoseconds (set from the host before launches).
__device__ unsigned long long g_wait_limit_ns = 2000000000ull;

__device__ __forceinline__ void set_device_error(int code) { atomicCAS(&g_device_error, 0, code); }

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(bf16 v) { return __bfloat162float(v); }

template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ bf16 from_f32<bf16>(float v) { return __float2bfloat16_rn(v); }

// RoPE for interleaved pair i of a d_r-wide vector at position pos: angle = pos*base^(-2i/d_r),
// evaluated in double so long positions keep full angle precision.
__device__ __forceinline__ void rope_cos_sin(int pos, int i, int d_r, float base, float* c, float* s) {
    double theta = pow((double)base, -2.0 * (double)i / (double)d_r);
    double ang = (double)pos * theta;
    double sd, cd;
    sincos(ang, &sd, &cd);
    *c = (float)cd;
    *s = (float)sd;
}

__device__ __forceinline__ unsigned long long globaltimer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

}  // namespace mla
