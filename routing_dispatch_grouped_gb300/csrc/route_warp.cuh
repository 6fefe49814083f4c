// Router top-k for one token by one warp, shared by the router kernel and the fused small-batch
// route+dispatch kernel.
//
// Expert parallelism page, "Adding an implementation": the router's outputs are top_k_index and
// top_k_weights. Reading: descending fp32 logit, ties to the lower expert index, -0 == +0, NaN
// below -inf; softmax (optionally renormalised over the k selected) or sigmoid weights.
#pragma once

#include "moe_internal.cuh"

namespace rdg {

// Monotone map from fp32 to uint32 for "larger logit first": NaN -> 1, -inf -> 0x007FFFFF,
// +inf -> 0xFF800000; -0.0 is folded onto +0.0. Key 0 marks an empty or already-taken entry.
__device__ __forceinline__ uint32_t route_order_key(float v) {
    if (v != v) return 1u;
    if (v == 0.0f) v = 0.0f;
    const uint32_t u = __float_as_uint(v);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Lane l holds experts l, l+32, ... (VPL = ceil(E/32) values; entries at or past E are
// ignored). After the call lane j < k holds slot j: *id = the expert, *w = its weight. All 32
// lanes must call it together.
template <int VPL>
__device__ __forceinline__ void route_select_warp(const float (&v)[VPL], int E, int k,
                                                  int score_fn, int renorm, int lane, int* id,
                                                  float* wt) {
    uint32_t key[VPL];
#pragma unroll
    for (int i = 0; i < VPL; ++i) key[i] = (lane + 32 * i < E) ? route_order_key(v[i]) : 0u;
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
    *id = my_id;
    *wt = w;
}

// Router top-k of one token from its logits row in global memory.
template <int VPL>
__device__ __forceinline__ void route_token_warp(const float* __restrict__ row, int E, int k,
                                                 int score_fn, int renorm, int lane, int* id,
                                                 float* wt) {
    float v[VPL];
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
        const int e = lane + 32 * i;
        v[i] = (e < E) ? __ldg(row + e) : -INFINITY;
    }
    route_select_warp<VPL>(v, E, k, score_fn, renorm, lane, id, wt);
}

}  // namespace rdg
