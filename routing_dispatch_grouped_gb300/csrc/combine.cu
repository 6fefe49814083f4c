// Combine: weighted return of the expert outputs to token order.
//
// Expert parallelism page, "Token dispatch": the expert results come back and are combined with
// the routing weights; "Adding an implementation": the call returns the weighted expert output
// for each token. One warp per token: the k fp32 rows are gathered with 16-byte loads, summed in
// slot order in fp32, the shared-expert row (if any) is added, and the sum is rounded once to
// the output dtype.
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

template <typename OutT>
__global__ void __launch_bounds__(256) combine_kernel(const float4* __restrict__ y, int T, int d4,
                                                      int k,
                                                      const int32_t* __restrict__ slot_to_sorted,
                                                      const float* __restrict__ weights,
                                                      const float4* __restrict__ y_shared,
                                                      OutT* __restrict__ out) {
    const int lane = threadIdx.x & 31;
    const int warps_total = gridDim.x * (blockDim.x >> 5);
    for (int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); t < T; t += warps_total) {
        int my_pos = -1;
        float my_w = 0.0f;
        if (lane < k) {
            my_pos = __ldg(slot_to_sorted + (size_t)t * k + lane);
            my_w = weights ? __ldg(weights + (size_t)t * k + lane) : 1.0f;
        }
        // uniform trip count: every lane takes part in each shuffle
        for (int base = 0; base < d4; base += 32) {
            const int c = base + lane;
            const bool in = c < d4;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int j = 0; j < k; ++j) {
                const int p = __shfl_sync(0xFFFFFFFFu, my_pos, j);
                const float w = __shfl_sync(0xFFFFFFFFu, my_w, j);
                if (in && p >= 0) {
                    const float4 v = __ldg(y + (size_t)p * d4 + c);
                    acc.x = fmaf(w, v.x, acc.x);
                    acc.y = fmaf(w, v.y, acc.y);
                    acc.z = fmaf(w, v.z, acc.z);
                    acc.w = fmaf(w, v.w, acc.w);
                }
            }
            if (!in) continue;
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
}

}  // namespace

cudaError_t launch_combine(const float* y_sorted, const int32_t* slot_to_sorted,
                           const float* weights, const float* y_shared, int T, int d, int k,
                           bool out_bf16, void* out, cudaStream_t s) {
    const int warps = 8;
    int blocks = (T + warps - 1) / warps;
    const int max_blocks = device_sm_count() * 8;
    if (blocks > max_blocks) blocks = max_blocks;
    const int d4 = d / 4;
    const float4* y = reinterpret_cast<const float4*>(y_sorted);
    const float4* ys = reinterpret_cast<const float4*>(y_shared);
    if (out_bf16)
        combine_kernel<__nv_bfloat16><<<blocks, 32 * warps, 0, s>>>(
            y, T, d4, k, slot_to_sorted, weights, ys, static_cast<__nv_bfloat16*>(out));
    else
        combine_kernel<float><<<blocks, 32 * warps, 0, s>>>(y, T, d4, k, slot_to_sorted, weights,
                                                            ys, static_cast<float*>(out));
    return cudaGetLastError();
}

}  // namespace rdg
