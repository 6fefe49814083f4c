// MX (OCP Microscaling) element conversions and block quantisation shared by the MX kernels
// and the GEMM epilogue that rounds the SwiGLU activation to MXFP8.
#pragma once

#include <cuda_fp16.h>

#include "moe_internal.cuh"

namespace rdg {

// floor(log2(a)) of a finite a > 0 from its bits (exact); -200 for a == 0.
__device__ __forceinline__ int floor_log2_f32(float a) {
    const uint32_t b = __float_as_uint(a);
    const int e = (int)((b >> 23) & 0xFF);
    if (e > 0) return e - 127;
    const uint32_t m = b & 0x7FFFFF;
    return m ? (31 - __clz((int)m)) - 149 : -200;
}

// 2^p as fp32 for p in [-149, 127] (exact).
__device__ __forceinline__ float pow2_f32(int p) {
    if (p >= -126) return __uint_as_float((uint32_t)(p + 127) << 23);
    return __uint_as_float(1u << (p + 149));
}

// Block scale exponent of a block whose largest magnitude is amax.
__device__ __forceinline__ int mx_scale_exp(float amax, int emax) {
    const int fl = floor_log2_f32(amax);
    int s = fl == -200 ? -127 : fl - emax;
    return s < -127 ? -127 : (s > 127 ? 127 : s);
}

// Two fp32 values to E4M3 codes, round to nearest even, saturating: (lo code of a, hi of b).
__device__ __forceinline__ uint32_t e4m3x2(float a, float b) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(b), "f"(a));
    return r;
}
// Two E4M3 codes (low byte first) to two fp32 values.
__device__ __forceinline__ float2 e4m3x2_to_f32(uint32_t codes) {
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"((uint16_t)codes));
    const __half2 h = *reinterpret_cast<const __half2*>(&h2);
    return __half22float2(h);
}
// Two fp32 values to one byte of E2M1 codes (a in the low nibble).
__device__ __forceinline__ uint32_t e2m1x2(float a, float b) {
    uint32_t r;
    asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u32.u8 %0, t;\n\t}"
        : "=r"(r)
        : "f"(b), "f"(a));
    return r;
}
// One byte of E2M1 codes to two fp32 values (low nibble first).
__device__ __forceinline__ float2 e2m1x2_to_f32(uint32_t byte) {
    uint32_t h2;
    asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}"
        : "=r"(h2)
        : "r"(byte));
    const __half2 h = *reinterpret_cast<const __half2*>(&h2);
    return __half22float2(h);
}

// Round 32 fp32 values (one MX block, n valid) to MXFP8 and back, in place.
__device__ __forceinline__ void mx_fakequant_e4m3_block(float (&v)[32], int n) {
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i)
        if (i < n) amax = fmaxf(amax, fabsf(v[i]));
    const int s = mx_scale_exp(amax, 8);
    const float inv = pow2_f32(-s), sc = pow2_f32(s);
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
        const float2 q = e4m3x2_to_f32(e4m3x2(v[i] * inv, v[i + 1] * inv));
        v[i] = q.x * sc;
        v[i + 1] = q.y * sc;
    }
}

// Column of the logical weight that column m of column block nb holds (-1: padding).
__device__ __forceinline__ int mx_block_col(const MxBlocks& b, int nb, int m) {
    if (b.half) {
        const int up = nb >= b.nbh;
        const int c = (nb - (up ? b.nbh : 0)) * 64 + m;
        return c < b.half ? c + (up ? b.half : 0) : -1;
    }
    const int c = nb * 64 + m;
    return c < b.cols ? c : -1;
}

}  // namespace rdg
