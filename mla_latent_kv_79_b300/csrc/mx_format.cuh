// MX block formats of the low-precision latent cache.
//
// The institutepm explainer ("Multi-Head Latent Attention (MLA) Explained", section "Which
// Models Use MLA and What Is Next") names MXFP4 quantisation of the KV cache beside MLA; the
// element and scale formats are those of the OCP Microscaling Formats (MX) specification v1.0.
// A cached row of W = d_c + d_r numbers ([c_kv | rotated k_rope]) is cut into blocks of 32
// consecutive elements; a block stores one E8M0 scale byte (2^e, byte e + 127) and 32 element
// codes, E4M3 bytes (MXFP8) or E2M1 nibbles (MXFP4, element 2i in the low nibble of byte i).
// The dequantised element is 2^e * elem(code).
//
// Encoding choices (the pages give none): the block exponent is the smallest e with
// max|v| <= max_elem * 2^e, clamped to [-127, 127] (so no element of a block saturates; a zero
// block gets -127); codes round to nearest, ties to even, from the fp32 value v * 2^-e, which is
// exact because the scale is a power of two.  Decoding into bf16 is exact: every E4M3 or E2M1
// value times a power of two in the bf16 normal range is a bf16 number.
#pragma once

#include <cuda_fp16.h>

#include "mla_common.cuh"

namespace mla {

enum KvFormat { KV_PLAIN = 0, KV_MXFP8 = 1, KV_MXFP4 = 2 };
constexpr int MX_BLOCK = 32;

// Bytes of element codes per cached row, and scale bytes per row.
__host__ __device__ inline int mx_row_bytes(int fmt, int width) { return fmt == KV_MXFP4 ? width / 2 : width; }
__host__ __device__ inline int mx_scale_bytes(int width) { return width / MX_BLOCK; }

// 2^e as a float for e in [-127, 128] (2^-127 is a subnormal, 2^128 gives +inf)
__device__ __forceinline__ float exp2_int(int e) {
    return e >= -126 ? __uint_as_float((uint32_t)(e + 127) << 23) : __uint_as_float(0x00400000u);
}

// Block exponent from the block's largest magnitude (see the encoding choices above).
template <int FMT>
__device__ __forceinline__ int mx_block_exponent(float amax) {
    constexpr int EMAX = FMT == KV_MXFP8 ? 8 : 2;            // exponent of the top binade
    constexpr float MAXV = FMT == KV_MXFP8 ? 448.f : 6.f;    // largest finite element
    const uint32_t ef = (__float_as_uint(amax) >> 23) & 0xFFu;
    if (!(amax > 0.f) || ef == 0u) return -127;   // zero, or below 2^-126: the clamp decides
    int e = (int)ef - 127 - EMAX;                 // floor(log2 amax) - EMAX
    if (amax * exp2_int(-e) > MAXV) ++e;          // exact: the scaled maximum is in [2^EMAX, 2^(EMAX+1))
    return e < -127 ? -127 : (e > 127 ? 127 : e);
}

// Two fp32 values to E4M3 codes (round to nearest even, saturating): lo in the low byte.
__device__ __forceinline__ uint32_t e4m3x2_from_f32(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// Two fp32 values to E2M1 codes (round to nearest even, saturating): lo in the low nibble.
__device__ __forceinline__ uint32_t e2m1x2_from_f32(float lo, float hi) {
    uint16_t r;
    asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u16.u8 %0, t;\n\t}"
        : "=h"(r)
        : "f"(hi), "f"(lo));
    return r & 0xFFu;
}

// Two E4M3 codes (low byte first) to two floats, exact.
__device__ __forceinline__ float2 e4m3x2_to_f32(uint32_t codes2) {
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"((uint16_t)codes2));
    __half2_raw raw;
    raw.x = (unsigned short)(h2 & 0xFFFFu);
    raw.y = (unsigned short)(h2 >> 16);
    return __half22float2(__half2(raw));
}

// Two E2M1 codes (low nibble first) to two floats, exact.
__device__ __forceinline__ float2 e2m1x2_to_f32(uint32_t byte) {
    uint32_t h2;
    asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}" : "=r"(h2) : "r"(byte & 0xFFu));
    __half2_raw raw;
    raw.x = (unsigned short)(h2 & 0xFFFFu);
    raw.y = (unsigned short)(h2 >> 16);
    return __half22float2(__half2(raw));
}

// Dequantised element k of a cached row (portable path: one element at a time).
template <int FMT>
__device__ __forceinline__ float mx_load(const uint8_t* codes_row, const uint8_t* scales_row, int k) {
    const float s = exp2_int((int)scales_row[k / MX_BLOCK] - 127);
    if (FMT == KV_MXFP8) {
        const float2 v = e4m3x2_to_f32(codes_row[k]);
        return v.x * s;
    } else {
        const uint32_t b = codes_row[k >> 1];
        const float2 v = e2m1x2_to_f32(b);
        return ((k & 1) ? v.y : v.x) * s;
    }
}

// The 32 lanes of a warp hold one block of a row (lane l: element l of the block).  The warp
// finds the block exponent, codes every element and stores the block: 32 code bytes (MXFP8:
// lanes 0 and 16 write 16 bytes each) or 16 bytes of nibbles (MXFP4: lane 0), plus the scale
// byte (lane 0).  `codes` points at the block's first code byte, `scale` at its scale byte;
// `store` gates the writes (warp-uniform), every lane takes part in the shuffles.
template <int FMT>
__device__ __forceinline__ void mx_store_block(uint8_t* codes, uint8_t* scale, float v, int lane, bool store) {
    const float amax = warp_max(fabsf(v));
    const int e = mx_block_exponent<FMT>(amax);
    const float x = v * exp2_int(-e);
    const float nb = __shfl_down_sync(0xffffffffu, x, 1);
    uint32_t w;  // meaningful in lanes 4j: elements 4j..4j+3 packed
    if (FMT == KV_MXFP8) {
        const uint32_t pair = e4m3x2_from_f32(x, nb);              // even lanes: elements l, l+1
        const uint32_t up = __shfl_down_sync(0xffffffffu, pair, 2);
        w = pair | (up << 16);
        const uint32_t w1 = __shfl_down_sync(0xffffffffu, w, 4);
        const uint32_t w2 = __shfl_down_sync(0xffffffffu, w, 8);
        const uint32_t w3 = __shfl_down_sync(0xffffffffu, w, 12);
        if (store && (lane & 15) == 0) *reinterpret_cast<uint4*>(codes + lane) = make_uint4(w, w1, w2, w3);
    } else {
        const uint32_t byte = e2m1x2_from_f32(x, nb);              // even lanes: elements l, l+1
        const uint32_t b1 = __shfl_down_sync(0xffffffffu, byte, 2);
        const uint32_t b2 = __shfl_down_sync(0xffffffffu, byte, 4);
        const uint32_t b3 = __shfl_down_sync(0xffffffffu, byte, 6);
        w = byte | (b1 << 8) | (b2 << 16) | (b3 << 24);            // lanes 8j: elements 8j..8j+7
        const uint32_t w1 = __shfl_down_sync(0xffffffffu, w, 8);
        const uint32_t w2 = __shfl_down_sync(0xffffffffu, w, 16);
        const uint32_t w3 = __shfl_down_sync(0xffffffffu, w, 24);
        if (store && lane == 0) *reinterpret_cast<uint4*>(codes) = make_uint4(w, w1, w2, w3);
    }
    if (store && lane == 0) *scale = (uint8_t)(e + 127);
}

}  // namespace mla
