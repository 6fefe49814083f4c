// Router top-k gating: one warp per token.
//
// Expert parallelism page, "Adding an implementation": the router's outputs are top_k_index and
// top_k_weights [T, k]. The score function, tie order and NaN order are this library's reading
// (descending fp32 logit, ties to the lower expert index, -0 == +0, NaN below -inf).
//
// Lane l holds experts l, l+32, l+64, ... (coalesced 128-byte loads per step). Each of the k
// rounds takes a warp-wide maximum of a 32-bit order key (redux.sync), then the lowest expert
// index among lanes holding that key, and removes the winner. The weights are computed in fp32
// from the selected logits, summed in slot order.
#include "route_warp.cuh"

namespace rdg {
namespace {

template <int VPL>
__global__ void __launch_bounds__(256) route_kernel(const float* __restrict__ logits, int T, int E,
                                                    int k, int score_fn, int renorm,
                                                    int32_t* __restrict__ ids,
                                                    float* __restrict__ weights) {
    griddep_wait();
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t >= T) return;  // whole warp leaves together
    int id;
    float w;
    route_token_warp<VPL>(logits + (size_t)t * E, E, k, score_fn, renorm, lane, &id, &w);
    if (lane < k) {
        ids[(size_t)t * k + lane] = id;
        weights[(size_t)t * k + lane] = w;
    }
}

}  // namespace

cudaError_t launch_route(const float* logits, int T, int E, int k, int score_fn, bool renorm,
                         int32_t* ids, float* weights, cudaStream_t s) {
    const int warps = 8;
    const dim3 grid((T + warps - 1) / warps), block(32 * warps);
    const int rn = renorm ? 1 : 0;
    auto kern = E <= 32 ? route_kernel<1> : E <= 64 ? route_kernel<2>
              : E <= 128 ? route_kernel<4> : route_kernel<8>;
    return launch_kernel(kern, grid, block, 0, s, logits, T, E, k, score_fn, rn, ids, weights);
}

}  // namespace rdg
