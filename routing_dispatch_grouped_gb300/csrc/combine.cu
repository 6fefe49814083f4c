// Combine: weighted return of the expert outputs to token order.
//
// Expert parallelism page, "Token dispatch": the expert results come back and are combined with
// the routing weights; "Adding an implementation": the call returns the weighted expert output
// for each token. Each thread owns 4 columns of one token: the k fp32 values are gathered with
// 16-byte loads, summed in slot order in fp32, the shared-expert value (if any) is added, and the
// sum is rounded once to the output dtype.
#include "moe_internal.cuh"

namespace rdg {
namespace {

__device__ __forceinline__ void store4(float* out, size_t idx4, float4 v) {
    reinterpret_cast<float4*>(out)[idx4] = v;
}
__device__ __forceinline__ void store4(__nv_bfloat16* out, size_t idx4, float4 v) {
    __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y);
    __nv_bfloat162 b = __floats2bfloat162_rn(v.z, v.w);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t*>(&a);
    u.y = *reinterpret_cast<uint32_t*>(&b);
    reinterpret_cast<uint2*>(out)[idx4] = u;
}

// Grid: x over 4-column groups of the row (256 per block), y over tokens (grid-stride). Every
// thread issues its k independent 16-byte loads before summing, so a batch of one token still
// spreads over d/1024 blocks.
template <typename OutT>
__global__ void __launch_bounds__(256) combine_kernel(const float4* __restrict__ y, int T, int d4,
                                                      int k,
                                                      const int32_t* __restrict__ slot_to_sorted,
                                                      const float* __restrict__ weights,
                                                      const float4* __restrict__ y_shared,
                                                      OutT* __restrict__ out) {
    __shared__ int pos_s[kMaxK];
    __shared__ float w_s[kMaxK];
    griddep_wait();
    const int c = blockIdx.x * blockDim.x + threadIdx.x;
    for (int t = blockIdx.y; t < T; t += gridDim.y) {
        __syncthreads();
        if (threadIdx.x < k) {
            pos_s[threadIdx.x] = __ldg(slot_to_sorted + (size_t)t * k + threadIdx.x);
            w_s[threadIdx.x] = weights ? __ldg(weights + (size_t)t * k + threadIdx.x) : 1.0f;
        }
        __syncthreads();
        if (c >= d4) continue;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int j = 0; j < k; ++j) {
            const int p = pos_s[j];
            if (p >= 0) {
                const float w = w_s[j];
                const float4 v = __ldg(y + (size_t)p * d4 + c);
                acc.x = fmaf(w, v.x, acc.x);
                acc.y = fmaf(w, v.y, acc.y);
                acc.z = fmaf(w, v.z, acc.z);
                acc.w = fmaf(w, v.w, acc.w);
            }
        }
        if (y_shared) {
            const float4 v = __ldg(y_shared + (size_t)t * d4 + c);
            acc.x += v.x;
            acc.y += v.y;
            acc.z += v.z;
            acc.w += v.w;
        }
        store4(out, (size_t)t * d4 + c, acc);
    }
}

}  // namespace

cudaError_t launch_combine(const float* y_sorted, const int32_t* slot_to_sorted,
                           const float* weights, const float* y_shared, int T, int d, int k,
                           bool out_bf16, void* out, cudaStream_t s) {
    const int d4 = d / 4;
    const int bx = (d4 + 255) / 256;
    const int by = T < 65535 ? T : 65535;
    const dim3 grid(bx, by);
    const float4* y = reinterpret_cast<const float4*>(y_sorted);
    const float4* ys = reinterpret_cast<const float4*>(y_shared);
    if (out_bf16)
        return launch_kernel(combine_kernel<__nv_bfloat16>, grid, dim3(256), 0, s, y, T, d4, k,
                             slot_to_sorted, weights, ys, static_cast<__nv_bfloat16*>(out));
    return launch_kernel(combine_kernel<float>, grid, dim3(256), 0, s, y, T, d4, k,
                         slot_to_sorted, weights, ys, static_cast<float*>(out));
}

}  // namespace rdg
