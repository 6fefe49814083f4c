// Pieces of the block-scaled (MX) tcgen05 GEMM (gemm_mx_tc.cu): the scale-atom copy into tensor
// memory, the kind::mxf8f6f4 MMA and its instruction descriptor, and the epilogue blocks (SwiGLU
// rounded to MXFP8; fp32 rows).
#pragma once

#include "mx.cuh"

namespace rdg {

constexpr int kAtom = 512;  // one scale atom: 32 rows of 16 bytes (see gemm_mx_tc.cu)

// 1D bulk copy global -> shared, completing on an mbarrier (both addresses 16-byte aligned,
// size a multiple of 16).
__device__ __forceinline__ void bulk_copy(uint32_t dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(dst),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Shared-memory descriptor without swizzle (a scale atom: 32 rows of 16 bytes, 8-row groups
// 128 bytes apart).
__device__ __forceinline__ uint64_t smem_desc_plain(uint32_t addr) {
    return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)(128u >> 4) << 16) |
           ((uint64_t)(128u >> 4) << 32) | (1ull << 46);
}
// 32 rows x 128 bits of shared memory into 4 TMEM columns of every lane quarter.
__device__ __forceinline__ void tmem_cp_atom(uint32_t taddr, uint64_t sdesc) {
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
                 : "memory");
}
// D[tmem] (+)= (A * scaleA) (B * scaleB): A E4M3, B E2M1, scales E8M0 from TMEM.
__device__ __forceinline__ void umma_mx(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                        uint32_t idesc, uint32_t sfa, uint32_t sfb,
                                        uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, "
        "[%4], [%5], p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
        : "memory");
}
// Instruction descriptor, kind::mxf8f6f4 with block scales: B scale-factor id (bits 4-5), A
// E4M3 (bits 7-9 = 0), B E2M1 (bits 10-12 = 5), both K-major (bits 15, 16 = 0), N >> 3 (bits
// 17-22), E8M0 scales (bit 23), M >> 4 (bits 24-28), A scale-factor id (bits 29-30).
__host__ __device__ constexpr uint32_t idesc_mx(int M, int N, uint32_t sf_id) {
    return (sf_id << 4) | (5u << 10) | ((uint32_t)(N >> 3) << 17) | (1u << 23) |
           ((uint32_t)(M >> 4) << 24) | (sf_id << 29);
}

// The same with the roles of the formats swapped: A E2M1 (bits 7-9 = 5), B E4M3 (bits 10-12 = 0),
// for products with the weights as the M side (the decode layer of decode_mx_tc.cu); the A and
// B scale-factor ids (which K block of their atoms' four) given separately.
__host__ __device__ constexpr uint32_t idesc_mx_w4a8(int M, int N, uint32_t sfa_id,
                                                     uint32_t sfb_id) {
    return (sfb_id << 4) | (5u << 7) | ((uint32_t)(N >> 3) << 17) | (1u << 23) |
           ((uint32_t)(M >> 4) << 24) | (sfa_id << 29);
}

// One MX block of h (32 columns from col0) from its gate and up accumulators: SwiGLU in
// fp32 (accumulators times the row scale s), rounded to MXFP8; stores the 32 codes of a valid
// row and returns the scale byte (127 for a block past the end of the columns).
__device__ __forceinline__ uint32_t h_block_mxfp8(const uint32_t (&g)[32], const uint32_t (&u)[32],
                                                  float s, int col0, int N, bool row_ok,
                                                  uint8_t* hrow) {
    if (col0 >= N) return 127u;
    float hv[32];
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        hv[i] = silu(__uint_as_float(g[i]) * s) * (__uint_as_float(u[i]) * s);
        amax = fmaxf(amax, fabsf(hv[i]));
    }
    const int se = mx_scale_exp(amax, 8);
    const float inv = pow2_f32(-se);
    uint32_t w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
        w[i] = e4m3x2(hv[4 * i] * inv, hv[4 * i + 1] * inv) |
               (e4m3x2(hv[4 * i + 2] * inv, hv[4 * i + 3] * inv) << 16);
    if (row_ok) {
        uint4* dst = reinterpret_cast<uint4*>(hrow + col0);
        dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
        dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
    }
    return (uint32_t)(se + 127);
}

// 32 fp32 accumulator columns from col0 of one output row (N a multiple of 32).
__device__ __forceinline__ void store_y_block(const uint32_t (&y)[32], int col0, int N,
                                              float* yrow) {
    if (col0 >= N) return;
    float4* dst = reinterpret_cast<float4*>(yrow + col0);
#pragma unroll
    for (int v = 0; v < 8; ++v)
        dst[v] = make_float4(__uint_as_float(y[4 * v]), __uint_as_float(y[4 * v + 1]),
                             __uint_as_float(y[4 * v + 2]), __uint_as_float(y[4 * v + 3]));
}

}  // namespace rdg
