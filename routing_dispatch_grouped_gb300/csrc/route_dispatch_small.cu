// Fused router + dispatch indices for small batches (T*k <= 1024), in one block of 1024 threads.
//
// Expert parallelism page, "Choosing an implementation": at decode the layer should need no host
// synchronisation and be capturable in a CUDA graph; with a handful of tokens the cost is launch
// latency, so the five launches of route + histogram + scan + rank collapse into one. The result
// is the same definition as the multi-kernel path (Expert parallelism page, "Token dispatch";
// rows of an expert in ascending slot order), computed in shared memory:
//   1. warp w routes tokens w, w+32, ... (the same per-token warp routine as the router kernel);
//   2. warp w counts the experts of slots [32w, 32w+32) with a warp match;
//   3. thread e turns the 32 per-warp counts of expert e into per-warp bases and a total;
//   4. warp 0 scans the totals into offsets;
//   5. every slot's position = offset + base of its warp + earlier equal slots in its warp.
// The row copy into x_sorted stays a separate, grid-wide kernel.
#include "route_warp.cuh"

namespace rdg {
namespace {

constexpr int kWarps = 32;

template <int VPL>
__global__ void __launch_bounds__(1024) route_dispatch_small_kernel(
    const float* __restrict__ logits, int T, int E, int k, int score_fn, int renorm,
    int32_t* __restrict__ ids, float* __restrict__ weights, int32_t* __restrict__ counts,
    int32_t* __restrict__ offsets, int32_t* __restrict__ sorted_to_slot,
    int32_t* __restrict__ slot_to_sorted) {
    __shared__ int ids_s[kSmallDispatchMaxSlots];
    __shared__ int cnt[kWarps][kMaxE];  // per-warp counts, then per-warp bases
    __shared__ int tot[kMaxE];
    __shared__ int off_s[kMaxE + 1];
    griddep_wait();
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int R = T * k;

    for (int t = w; t < T; t += kWarps) {
        int id;
        float wt;
        route_token_warp<VPL>(logits + (size_t)t * E, E, k, score_fn, renorm, lane, &id, &wt);
        if (lane < k) {
            ids[(size_t)t * k + lane] = id;
            weights[(size_t)t * k + lane] = wt;
            ids_s[t * k + lane] = id;
        }
    }
    for (int i = threadIdx.x; i < kWarps * kMaxE; i += blockDim.x) (&cnt[0][0])[i] = 0;
    __syncthreads();

    const int s = w * 32 + lane;
    const int e = (s < R) ? ids_s[s] : -1;
    const unsigned peers = __match_any_sync(0xFFFFFFFFu, e);
    if (e >= 0 && lane == __ffs(peers) - 1) cnt[w][e] = __popc(peers);
    __syncthreads();

    if (threadIdx.x < E) {
        int run = 0;
        for (int ww = 0; ww < kWarps; ++ww) {
            const int v = cnt[ww][threadIdx.x];
            cnt[ww][threadIdx.x] = run;
            run += v;
        }
        tot[threadIdx.x] = run;
    }
    __syncthreads();
    if (w == 0) {
        const int per = (E + 31) / 32;
        const int e0 = min(E, lane * per), e1 = min(E, e0 + per);
        int run = 0;
        for (int x = e0; x < e1; ++x) run += tot[x];
        int incl = run;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            if (lane >= o) incl += y;
        }
        int base = incl - run;
        for (int x = e0; x < e1; ++x) {
            off_s[x] = base;
            counts[x] = tot[x];
            offsets[x] = base;
            base += tot[x];
        }
        if (lane == 31) {
            off_s[E] = incl;
            offsets[E] = incl;
        }
    }
    __syncthreads();

    if (e >= 0) {
        const int pos = off_s[e] + cnt[w][e] + __popc(peers & ((1u << lane) - 1u));
        sorted_to_slot[pos] = s;
        slot_to_sorted[s] = pos;
    }
}

}  // namespace

cudaError_t launch_route_dispatch_small(const float* logits, int T, int E, int k, int score_fn,
                                        bool renorm, int32_t* ids, float* weights,
                                        int32_t* counts, int32_t* offsets,
                                        int32_t* sorted_to_slot, int32_t* slot_to_sorted,
                                        cudaStream_t s) {
    const int rn = renorm ? 1 : 0;
    auto kern = E <= 32 ? route_dispatch_small_kernel<1> : E <= 64 ? route_dispatch_small_kernel<2>
              : E <= 128 ? route_dispatch_small_kernel<4> : route_dispatch_small_kernel<8>;
    return launch_kernel(kern, dim3(1), dim3(1024), 0, s, logits, T, E, k, score_fn, rn, ids,
                         weights, counts, offsets, sorted_to_slot, slot_to_sorted);
}

}  // namespace rdg
