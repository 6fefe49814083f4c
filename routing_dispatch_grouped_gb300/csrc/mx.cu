// Block-scaled low-precision experts (MX formats): 4-bit expert weights, 8-bit activations.
//
// Expert parallelism page, the Mega MoE paragraph: the fused expert kernel of the newest GPUs
// multiplies FP8 activations by FP4 weights with block scales. The formats follow the OCP
// Microscaling specification: 32 consecutive elements along the reduction axis K share one
// E8M0 scale 2^s, s = floor(log2(max |v|)) - emax (emax 2 for E2M1, 8 for E4M3), clamped to
// [-127, 127] (-127 for an all-zero block); each element is v / 2^s rounded to nearest even and
// saturated at the format's largest finite value (cvt.rn.satfinite does exactly that).
//
// Storage:
//   MX weights of one kind (gate_up: K = d, N = 2I; down: K = I, N = d), [E, K, N] logically:
//     codes  [E][K][N / 2] bytes, byte j of row k holding column 2j (low nibble) and 2j + 1
//     scales [E][ceil(K / 32)][N] bytes (E8M0: s + 127), after the codes at a 256-byte boundary.
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

// One thread per (group, K block, column pair): 32 rows of columns 2j, 2j + 1.
__global__ void __launch_bounds__(256)
    mx_quant_weights_kernel(const uint32_t* __restrict__ w, int G, int K, int N,
                            uint8_t* __restrict__ codes, uint8_t* __restrict__ scales) {
    griddep_wait();
    const int NP = N / 2, KB = (K + 31) / 32;
    const long long total = (long long)G * KB * NP;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const int j = (int)(i % NP);
        const long long gk = i / NP;
        const int kb = (int)(gk % KB), g = (int)(gk / KB);
        const int k0 = kb * 32, n = min(32, K - k0);
        const uint32_t* src = w + ((size_t)g * K + k0) * NP + j;
        float a[32], b[32];
        float ma = 0.0f, mb = 0.0f;
#pragma unroll
        for (int r = 0; r < 32; ++r) {
            const uint32_t v = r < n ? __ldg(src + (size_t)r * NP) : 0u;
            a[r] = bf_lo(v);
            b[r] = bf_hi(v);
            ma = fmaxf(ma, fabsf(a[r]));
            mb = fmaxf(mb, fabsf(b[r]));
        }
        const int sa = mx_scale_exp(ma, 2), sb = mx_scale_exp(mb, 2);
        const float ia = pow2_f32(-sa), ib = pow2_f32(-sb);
        uint8_t* dst = codes + ((size_t)g * K + k0) * NP + j;
#pragma unroll
        for (int r = 0; r < 32; ++r)
            if (r < n) dst[(size_t)r * NP] = (uint8_t)e2m1x2(a[r] * ia, b[r] * ib);
        uint8_t* sc = scales + ((size_t)g * KB + kb) * N + 2 * j;
        sc[0] = (uint8_t)(sa + 127);
        sc[1] = (uint8_t)(sb + 127);
    }
}

// One block per (group, 32-row K block); a group without rows (offsets) leaves at once. Thread
// t takes 8-column chunks t, t + blockDim, ...: its 8 scales once, then 4 code bytes and 16
// bytes of bf16 per row (aligned for any N that is a multiple of 8).
__global__ void __launch_bounds__(256)
    mx_dequant_weights_kernel(const uint8_t* __restrict__ codes,
                              const uint8_t* __restrict__ scales, int G, int K, int N,
                              const int32_t* __restrict__ offsets, __nv_bfloat16* __restrict__ w) {
    griddep_wait();
    const int NP = N / 2, KB = (K + 31) / 32, chunks = N / 8;
    for (int bid = blockIdx.x; bid < G * KB; bid += gridDim.x) {
        const int g = bid / KB, kb = bid - g * KB;
        if (offsets && __ldg(offsets + g + 1) == __ldg(offsets + g)) continue;
        const int k0 = kb * 32, nr = min(32, K - k0);
        for (int c = threadIdx.x; c < chunks; c += blockDim.x) {
            const uint2 sv = __ldg(reinterpret_cast<const uint2*>(
                scales + ((size_t)g * KB + kb) * N + 8 * c));
            float sc[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
                sc[i] = pow2_f32((int)(((i < 4 ? sv.x : sv.y) >> (8 * (i % 4))) & 0xFF) - 127);
            const uint8_t* src = codes + ((size_t)g * K + k0) * NP + 4 * c;
            __nv_bfloat16* dst = w + ((size_t)g * K + k0) * N + 8 * c;
            for (int r = 0; r < nr; ++r) {
                const uint32_t cw = __ldg(reinterpret_cast<const uint32_t*>(src + (size_t)r * NP));
                uint32_t o[4];
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    const float2 q = e2m1x2_to_f32((cw >> (8 * b)) & 0xFF);
                    o[b] = pack_bf16x2(q.x * sc[2 * b], q.y * sc[2 * b + 1]);
                }
                *reinterpret_cast<uint4*>(dst + (size_t)r * N) = make_uint4(o[0], o[1], o[2], o[3]);
            }
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

MxGeom mx_geom(int K, int N, int G) {
    MxGeom m;
    m.codes = (size_t)G * K * (N / 2);
    m.scales_off = (m.codes + 255) / 256 * 256;
    m.total = m.scales_off + (size_t)G * ((K + 31) / 32) * N;
    return m;
}

cudaError_t launch_mx_quant_weights(const void* w, int G, int K, int N, void* mx,
                                    cudaStream_t s) {
    const MxGeom m = mx_geom(K, N, G);
    uint8_t* base = static_cast<uint8_t*>(mx);
    const long long work = (long long)G * ((K + 31) / 32) * (N / 2);
    return launch_kernel(mx_quant_weights_kernel, dim3(grid_for(work)), dim3(256), 0, s,
                         static_cast<const uint32_t*>(w), G, K, N, base, base + m.scales_off);
}

cudaError_t launch_mx_dequant_weights(const void* mx, int G, int K, int N,
                                      const int32_t* offsets, void* w, cudaStream_t s) {
    const MxGeom m = mx_geom(K, N, G);
    const uint8_t* base = static_cast<const uint8_t*>(mx);
    const long long blocks = (long long)G * ((K + 31) / 32);
    const long long cap = (long long)device_sm_count() * 16;
    return launch_kernel(mx_dequant_weights_kernel, dim3((unsigned)(blocks < cap ? blocks : cap)),
                         dim3(256), 0, s, base, base + m.scales_off, G, K, N, offsets,
                         static_cast<__nv_bfloat16*>(w));
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
