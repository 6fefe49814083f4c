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
#include "moe_internal.cuh"

namespace rdg {
namespace {

// Monotone map from fp32 to uint32 for "larger logit first": NaN -> 1, -inf -> 0x007FFFFF,
// +inf -> 0xFF800000; -0.0 is folded onto +0.0. Key 0 marks an empty or already-taken entry.
__device__ __forceinline__ uint32_t order_key(float v) {
    if (v != v) return 1u;
    if (v == 0.0f) v = 0.0f;
    const uint32_t u = __float_as_uint(v);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

template <int VPL>
__global__ void __launch_bounds__(256) route_kernel(const float* __restrict__ logits, int T, int E,
                                                    int k, int score_fn, int renorm,
                                                    int32_t* __restrict__ ids,
                                                    float* __restrict__ weights) {
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t >= T) return;  // whole warp leaves together
    const float* row = logits + (size_t)t * E;

    float v[VPL];
    uint32_t key[VPL];
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
        const int e = lane + 32 * i;
        v[i] = (e < E) ? __ldg(row + e) : -INFINITY;
        key[i] = (e < E) ? order_key(v[i]) : 0u;
    }

    int my_id = 0;
    float my_val = 0.0f;
    for (int r = 0; r < k; ++r) {
        // best entry of this lane: largest key, first (= lowest index) among equals
        uint32_t bk = 0u;
        int bi = 0x7FFFFFFF;
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
            if (key[i] > bk) {
                bk = key[i];
                bi = lane + 32 * i;
            }
        }
        const uint32_t wk = __reduce_max_sync(0xFFFFFFFFu, bk);
        const int cand = (bk == wk) ? bi : 0x7FFFFFFF;
        const int win = (int)__reduce_min_sync(0xFFFFFFFFu, (uint32_t)cand);
        float wv = 0.0f;
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
            if (lane + 32 * i == win) {
                key[i] = 0u;
                wv = v[i];
            }
        }
        wv = __shfl_sync(0xFFFFFFFFu, wv, win & 31);
        if (lane == r) {
            my_id = win;
            my_val = wv;
        }
    }

    // weights
    float w = 0.0f;
    if (score_fn == 0) {  // softmax
        const float m = __shfl_sync(0xFFFFFFFFu, my_val, 0);  // slot 0 holds the maximum
        const float ex = (lane < k) ? expf(my_val - m) : 0.0f;
        float denom = 0.0f;
        if (renorm) {
            for (int j = 0; j < k; ++j) denom += __shfl_sync(0xFFFFFFFFu, ex, j);
        } else {
            float part = 0.0f;
#pragma unroll
            for (int i = 0; i < VPL; ++i) {
                const int e = lane + 32 * i;
                if (e < E && !(v[i] != v[i])) part += expf(v[i] - m);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xFFFFFFFFu, part, o);
            denom = part;
        }
        w = ex / denom;
    } else {  // sigmoid
        const float sg = (lane < k) ? 1.0f / (1.0f + expf(-my_val)) : 0.0f;
        w = sg;
        if (renorm) {
            float denom = 0.0f;
            for (int j = 0; j < k; ++j) denom += __shfl_sync(0xFFFFFFFFu, sg, j);
            w = sg / denom;
        }
    }
    if (lane < k) {
        ids[(size_t)t * k + lane] = my_id;
        weights[(size_t)t * k + lane] = w;
    }
}

}  // namespace

cudaError_t launch_route(const float* logits, int T, int E, int k, int score_fn, bool renorm,
                         int32_t* ids, float* weights, cudaStream_t s) {
    const int warps = 8;
    const dim3 grid((T + warps - 1) / warps), block(32 * warps);
    const int rn = renorm ? 1 : 0;
    if (E <= 32)
        route_kernel<1><<<grid, block, 0, s>>>(logits, T, E, k, score_fn, rn, ids, weights);
    else if (E <= 64)
        route_kernel<2><<<grid, block, 0, s>>>(logits, T, E, k, score_fn, rn, ids, weights);
    else if (E <= 128)
        route_kernel<4><<<grid, block, 0, s>>>(logits, T, E, k, score_fn, rn, ids, weights);
    else
        route_kernel<8><<<grid, block, 0, s>>>(logits, T, E, k, score_fn, rn, ids, weights);
    return cudaGetLastError();
}

}  // namespace rdg
