// Common device helpers for libmla: element types, the per-device error word, RoPE angles.
#pragma once

#include <cmath>

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>
#include <math.h>

#include "mla.h"

namespace mla {

typedef __nv_bfloat16 bf16;

// Per-device error word (first error wins).  Read and cleared by mla_get_device_error().
__device__ int g_device_error = 0;

__device__ __forceinline__ void set_device_error(int code) { atomicCAS(&g_device_error, 0, code); }

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(bf16 v) { return __bfloat162float(v); }

template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ bf16 from_f32<bf16>(float v) { return __float2bfloat16_rn(v); }

// RoPE frequencies theta_i = base^(-2i/d_r) of the interleaved pairs (2i, 2i+1), evaluated in
// double on the host and passed by value (d_r <= 1024).
constexpr int MAX_ROPE_PAIRS = 512;
struct RopeFreq {
    double theta[MAX_ROPE_PAIRS];
};

inline void rope_freq_fill(RopeFreq* f, int d_r, float base) {
    for (int i = 0; i < d_r / 2 && i < MAX_ROPE_PAIRS; ++i)
        f->theta[i] = std::pow((double)base, -2.0 * (double)i / (double)d_r);
}

// cos and sin of the angle pos * theta.  The product and its reduction to [-pi, pi] are done
// in double, so the angle keeps full precision at long positions; sin and cos of the reduced
// angle are then taken in float (absolute error below 1e-6, far under bf16 rounding).
__device__ __forceinline__ void rope_cos_sin(int pos, double theta, float* c, float* s) {
    const double ang = (double)pos * theta;
    const double k = rint(ang * 0.15915494309189535);   // 1 / (2 pi)
    const float r = (float)fma(-k, 6.283185307179586, ang);
    sincosf(r, s, c);
}

// Programmatic dependent launch: a kernel launched with programmatic stream serialisation may
// start before its predecessor ends; griddepcontrol.wait blocks the calling thread until the
// predecessor grid has completed and its writes are visible.  launch_dependents lets the next
// such kernel be scheduled early.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

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
