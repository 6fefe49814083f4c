// Block-scaled low-precision experts (MX formats): 4-bit expert weights, 8-bit activations.
//
// Expert parallelism page, the Mega MoE paragraph: the fused expert kernel of the newest GPUs
// multiplies FP8 activations by FP4 weights with block scales. The formats follow the OCP
// Microscaling specification: 32 consecutive elements along the reduction axis K share one
// E8M0 scale 2^s, s = floor(log2(max |v|)) - emax (emax 2 for E2M1, 8 for E4M3), clamped to
// [-127, 127] (-127 for an all-zero block); each element is v / 2^s rounded to nearest even and
// saturated at the format's largest finite value (cvt.rn.satfinite does exactly that).
//
// Storage of MX weights (one kind; gate_up: K = d, columns 2I with the gate and up halves
// blocked separately; down: K = I, columns d), in blocks of 64 columns x 32 K rows:
//   block (e, nb, kb): 1 KB of E2M1 codes at ((e * NB + nb) * KB + kb) * 1024, as 256 words
//     [k-step ks (2)][16-column m-tile mt (4)][lane l (32)]; word byte b = hi + 2 kh, nibble
//     bit, holds column 16 mt + (l >> 2) + 8 hi and K row 32 kb + 16 ks + 2 (l & 3) + bit + 8 kh
//     of the block: lane l's A fragment of mma.m16n8k16 (weights as the M side, K along the
//     MMA's K) for that m-tile and k-step, one byte per A register;
//   its 64 E8M0 scales (one per column, s + 127) at scales_off + ((e * NB + nb) * KB + kb) * 64.
// NB = ceil(cols / 64) (gate_up: 2 ceil(I / 64), gate blocks first), KB = ceil(K / 32); padding
// columns and rows hold code 0. A decode consumer reads its whole A fragment with one 4-byte
// load; a run of K blocks of one column block is contiguous.
//   MXFP8 rows [R, K]: codes [R][K] (E4M3) and scales [R][ceil(K / 32)].
// Every MX value is exact in bf16 (E2M1 times 2^s for s in [-127, 125], and E4M3 times 2^s
// down to bf16's smallest subnormal), so the layer runs the bf16 tensor-core GEMMs on the
// dequantized values: weights dequantized into bf16 for the experts that received rows, x and
// the SwiGLU activation h rounded to MXFP8 and back (h in the gate_up GEMM's epilogue, from its
// fp32 value).
#include "mx.cuh"

namespace rdg {

namespace {

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// One thread per (group, column block, K block, column m of the block): 32 rows of one column.
__global__ void __launch_bounds__(256)
    mx_quant_weights_kernel(const __nv_bfloat16* __restrict__ w, int G, int K, int cols,
                            MxBlocks bl, uint8_t* __restrict__ codes,
                            uint8_t* __restrict__ scales) {
    griddep_wait();
    const long long total = (long long)G * bl.nb * bl.kb * 64;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const int m = (int)(i & 63);
        const long long blk = i >> 6;  // (g * NB + nb) * KB + kb
        const int kb = (int)(blk % bl.kb);
        const long long gn = blk / bl.kb;
        const int nb = (int)(gn % bl.nb), g = (int)(gn / bl.nb);
        const int col = mx_block_col(bl, nb, m);  // -1: padding
        const int k0 = kb * 32, nr = min(32, K - k0);
        float v[32];
        float amax = 0.0f;
#pragma unroll
        for (int r = 0; r < 32; ++r) {
            v[r] = (col >= 0 && r < nr)
                       ? __bfloat162float(w[((size_t)g * K + k0 + r) * cols + col])
                       : 0.0f;
            amax = fmaxf(amax, fabsf(v[r]));
        }
        const int s = mx_scale_exp(amax, 2);
        const float inv = pow2_f32(-s);
        uint8_t* cb = codes + blk * 1024;
        const int mt = m >> 4, r16 = m & 15, hi = r16 >> 3, lq = r16 & 7;
#pragma unroll
        for (int kk = 0; kk < 32; kk += 2) {
            // rows kk, kk + 1 of column m share a byte (even row in the low nibble)
            const int ks = kk >> 4, kx = kk & 15, kh = kx >> 3, l = lq * 4 + ((kx & 7) >> 1);
            cb[(((ks * 4 + mt) * 32 + l) << 2) + hi + 2 * kh] =
                (uint8_t)e2m1x2(v[kk] * inv, v[kk + 1] * inv);
        }
        scales[blk * 64 + m] = (uint8_t)(s + 127);
    }
}

// One block of 64 threads per (group, column block, K block); thread m dequantizes column m
// (16 code bytes, one scale) into 32 rows of bf16 [G, K, cols]. A group without rows (offsets)
// is skipped.
__global__ void __launch_bounds__(64)
    mx_dequant_weights_kernel(const uint8_t* __restrict__ codes,
                              const uint8_t* __restrict__ scales, int G, int K, int cols,
                              MxBlocks bl, const int32_t* __restrict__ offsets,
                              __nv_bfloat16* __restrict__ w) {
    griddep_wait();
    const long long nblk = (long long)G * bl.nb * bl.kb;
    const int m = threadIdx.x;
    for (long long blk = blockIdx.x; blk < nblk; blk += gridDim.x) {
        const int kb = (int)(blk % bl.kb);
        const long long gn = blk / bl.kb;
        const int nb = (int)(gn % bl.nb), g = (int)(gn / bl.nb);
        if (offsets && __ldg(offsets + g + 1) == __ldg(offsets + g)) continue;
        const int col = mx_block_col(bl, nb, m);
        if (col < 0) continue;
        const float sc = pow2_f32((int)__ldg(scales + blk * 64 + m) - 127);
        const uint8_t* cb = codes + blk * 1024;
        const int mt = m >> 4, r16 = m & 15, hi = r16 >> 3, lq = r16 & 7;
        const int k0 = kb * 32, nr = min(32, K - k0);
        __nv_bfloat16* dst = w + ((size_t)g * K + k0) * cols + col;
#pragma unroll
        for (int kk = 0; kk < 32; kk += 2) {
            const int ks = kk >> 4, kx = kk & 15, kh = kx >> 3, l = lq * 4 + ((kx & 7) >> 1);
            const float2 q = e2m1x2_to_f32(__ldg(cb + (((ks * 4 + mt) * 32 + l) << 2) + hi + 2 * kh));
            if (kk < nr) dst[(size_t)kk * cols] = __float2bfloat16_rn(q.x * sc);
            if (kk + 1 < nr) dst[(size_t)(kk + 1) * cols] = __float2bfloat16_rn(q.y * sc);
        }
    }
}

// One thread per (row, K block): 32 bf16 values rounded to MXFP8 and back into out (may be in;
// null: not written), and optionally the codes and scales.
__global__ void __launch_bounds__(256)
    mx_rows_kernel(const __nv_bfloat16* __restrict__ in, int R, int K,
                   __nv_bfloat16* __restrict__ out, uint8_t* __restrict__ codes,
                   uint8_t* __restrict__ scales) {
    griddep_wait();
    const int KB = (K + 31) / 32;
    const long long total = (long long)R * KB;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const int kb = (int)(i % KB);
        const long long row = i / KB;
        const int k0 = kb * 32, n = min(32, K - k0);  // n is a multiple of 8 (K is)
        const uint4* src = reinterpret_cast<const uint4*>(in + row * K + k0);
        float v[32];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint4 u = q * 8 < n ? src[q] : make_uint4(0u, 0u, 0u, 0u);
            const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                v[8 * q + 2 * h] = bf_lo(w4[h]);
                v[8 * q + 2 * h + 1] = bf_hi(w4[h]);
            }
        }
        float amax = 0.0f;
#pragma unroll
        for (int t = 0; t < 32; ++t) amax = fmaxf(amax, fabsf(v[t]));
        const int s = mx_scale_exp(amax, 8);
        const float inv = pow2_f32(-s), sc = pow2_f32(s);
        uint32_t cw[8], ow[16];
#pragma unroll
        for (int t = 0; t < 32; t += 2) {
            const uint32_t c = e4m3x2(v[t] * inv, v[t + 1] * inv);
            const float2 q = e4m3x2_to_f32(c);
            ow[t / 2] = pack_bf16x2(q.x * sc, q.y * sc);
            if ((t & 2) == 0)
                cw[t / 4] = c;
            else
                cw[t / 4] |= c << 16;
        }
        if (out) {
            uint4* dst = reinterpret_cast<uint4*>(out + row * K + k0);
#pragma unroll
            for (int q = 0; q < 4; ++q)
                if (q * 8 < n)
                    dst[q] = make_uint4(ow[4 * q], ow[4 * q + 1], ow[4 * q + 2], ow[4 * q + 3]);
        }
        if (codes) {
            uint8_t* cd = codes + row * K + k0;
            for (int t = 0; t < n; ++t) cd[t] = (uint8_t)(cw[t / 4] >> (8 * (t & 3)));
            scales[row * KB + kb] = (uint8_t)(s + 127);
        }
    }
}

int grid_for(long long work) {
    const long long cap = (long long)device_sm_count() * 8;
    long long g = (work + 255) / 256;
    if (g > cap) g = cap;
    return (int)(g < 1 ? 1 : g);
}

}  // namespace

MxBlocks mx_blocks(bool gate_up, int K, int N) {
    MxBlocks b;
    b.half = gate_up ? N : 0;
    b.nbh = gate_up ? (N + 63) / 64 : (N + 63) / 64;
    b.nb = gate_up ? 2 * b.nbh : b.nbh;
    b.kb = (K + 31) / 32;
    b.cols = gate_up ? 2 * N : N;
    return b;
}

MxGeom mx_geom(bool gate_up, int K, int N, int G) {
    const MxBlocks b = mx_blocks(gate_up, K, N);
    MxGeom m;
    m.blocks = b;
    m.codes = (size_t)G * b.nb * b.kb * 1024;
    m.scales_off = m.codes;  // a multiple of 1024
    m.total = m.codes + (size_t)G * b.nb * b.kb * 64;
    return m;
}

cudaError_t launch_mx_quant_weights(bool gate_up, const void* w, int G, int K, int N, void* mx,
                                    cudaStream_t s) {
    const MxGeom m = mx_geom(gate_up, K, N, G);
    uint8_t* base = static_cast<uint8_t*>(mx);
    const long long work = (long long)G * m.blocks.nb * m.blocks.kb * 64;
    return launch_kernel(mx_quant_weights_kernel, dim3(grid_for(work)), dim3(256), 0, s,
                         static_cast<const __nv_bfloat16*>(w), G, K, m.blocks.cols, m.blocks,
                         base, base + m.scales_off);
}

cudaError_t launch_mx_dequant_weights(bool gate_up, const void* mx, int G, int K, int N,
                                      const int32_t* offsets, void* w, cudaStream_t s) {
    const MxGeom m = mx_geom(gate_up, K, N, G);
    const uint8_t* base = static_cast<const uint8_t*>(mx);
    const long long blocks = (long long)G * m.blocks.nb * m.blocks.kb;
    const long long cap = (long long)device_sm_count() * 32;
    return launch_kernel(mx_dequant_weights_kernel, dim3((unsigned)(blocks < cap ? blocks : cap)),
                         dim3(64), 0, s, base, base + m.scales_off, G, K, m.blocks.cols,
                         m.blocks, offsets, static_cast<__nv_bfloat16*>(w));
}

cudaError_t launch_mx_rows(const void* in, int R, int K, void* out, void* codes, void* scales,
                           cudaStream_t s) {
    const long long work = (long long)R * ((K + 31) / 32);
    return launch_kernel(mx_rows_kernel, dim3(grid_for(work)), dim3(256), 0, s,
                         static_cast<const __nv_bfloat16*>(in), R, K,
                         static_cast<__nv_bfloat16*>(out), static_cast<uint8_t*>(codes),
                         static_cast<uint8_t*>(scales));
}

}  // namespace rdg
