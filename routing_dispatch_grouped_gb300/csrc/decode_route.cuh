// Router top-k and dispatch indices of a decode batch, computed by every block of a one-kernel
// decode layer in its own shared memory (decode_fused.cu, decode_mx_tc.cu).
//
// Same definitions as the stand-alone kernels (Expert parallelism page, "Adding an
// implementation": the router gives top_k_index and top_k_weights; "Token dispatch": the rows
// of an expert in ascending slot order): the warp router of route_kernel, and the counting sort
// of route_dispatch_small_kernel, so ids, weights and the sorted order agree bit for bit. With at
// most 32 slots one warp builds the same indices by votes instead.
#pragma once

#include "moe_internal.cuh"
#include "route_warp.cuh"

namespace rdg {

struct DecodeRouteIO {
    const float* logits;  // [T, E]
    int T, E, k, R, score_fn, renorm;
    // written by the writer block only
    int32_t* topk_ids;
    float* topk_w;
    int32_t* counts;
    int32_t* offsets;
    int32_t* s2p;  // sorted row -> slot
    int32_t* p2s;  // slot -> sorted row
};

// The lists the dispatch leaves in shared memory, and its scratch (free again once
// decode_dispatch has returned).
struct DecodeRouteSmem {
    // lists: per touched expert q (ascending expert id) its id, row count and first sorted row;
    // per sorted row its token and routing weight; per slot its sorted row (optional)
    int* eq;
    int* tq;
    int* offq;
    int* tok;
    float* wrow;
    int* pos;
    volatile int* nq;  // number of touched experts
    // scratch
    int* ids;
    float* w;
    int* rank;
    int* cnt;
    int* off;
    int* chunk;  // [chunk of 32 slots][E]: counts, then bases
};

// Carves the scratch out of `base` (kDecodeFusedMaxRows * 12 + kMaxE * 8 + 128 bytes plus
// ceil(R / 32) * E ints).
__device__ __forceinline__ void decode_route_scratch(DecodeRouteSmem& sm, void* base) {
    sm.ids = reinterpret_cast<int*>(base);
    sm.w = reinterpret_cast<float*>(sm.ids + kDecodeFusedMaxRows);
    sm.rank = reinterpret_cast<int*>(sm.w + kDecodeFusedMaxRows);
    sm.cnt = sm.rank + kDecodeFusedMaxRows;
    sm.off = sm.cnt + kMaxE;
    sm.chunk = sm.off + kMaxE + 32;
}

// Warp w of NWARPS routes tokens w, w + NWARPS, ... (the logits load heads the critical path);
// `vpl` = logits per lane (E <= 32 vpl). The block's set-up can run beside it; the chunk
// counters are cleared here, and a block barrier must follow before decode_dispatch.
template <int NWARPS>
__device__ __forceinline__ void decode_route_tokens(const DecodeRouteIO& io,
                                                    const DecodeRouteSmem& sm, int vpl) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int t = warp; t < io.T; t += NWARPS) {
        const float* row = io.logits + (size_t)t * io.E;
        int id;
        float wt;
        switch (vpl) {
            case 1: route_token_warp<1>(row, io.E, io.k, io.score_fn, io.renorm, lane, &id, &wt); break;
            case 2: route_token_warp<2>(row, io.E, io.k, io.score_fn, io.renorm, lane, &id, &wt); break;
            case 4: route_token_warp<4>(row, io.E, io.k, io.score_fn, io.renorm, lane, &id, &wt); break;
            default: route_token_warp<8>(row, io.E, io.k, io.score_fn, io.renorm, lane, &id, &wt); break;
        }
        if (lane < io.k) {
            sm.ids[t * io.k + lane] = id;
            sm.w[t * io.k + lane] = wt;
        }
    }
    const int nch = (io.R + 31) / 32;
    for (int i = threadIdx.x; i < nch * io.E; i += blockDim.x) sm.chunk[i] = 0;
}

// The dispatch indices from the routed ids (block-wide; call after the barrier that follows
// decode_route_tokens). Returns the number of touched experts; the writer block also stores
// ids, weights, counts, offsets and both permutations.
__device__ __forceinline__ int decode_dispatch(const DecodeRouteIO& io, const DecodeRouteSmem& sm,
                                               bool writer) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int R = io.R, E = io.E, nch = (R + 31) / 32;
    if (R <= 32) {
        // at most 32 slots: warp 0 alone, by votes. Slot s's sorted row is the number of slots
        // routed to a lower expert plus those of its own expert with a lower slot index (the
        // counting sort's order), and the touched experts come out in ascending id order.
        if (warp == 0) {
            const bool act = lane < R;
            const int e = act ? sm.ids[lane] : -1;
            const unsigned peers = __match_any_sync(0xFFFFFFFFu, e);
            const int lead = (act && lane == __ffs(peers) - 1) ? 1 : 0;
            int off = 0, qi = 0;
            for (int j = 0; j < R; ++j) {
                const int ej = __shfl_sync(0xFFFFFFFFu, e, j);
                const int lj = __shfl_sync(0xFFFFFFFFu, lead, j);
                off += ej < e ? 1 : 0;
                qi += (lj && ej < e) ? 1 : 0;
            }
            if (act) {
                const int pos = off + __popc(peers & ((1u << lane) - 1u));
                sm.tok[pos] = lane / io.k;
                sm.wrow[pos] = sm.w[lane];
                if (sm.pos) sm.pos[lane] = pos;
                if (writer) {
                    io.topk_ids[lane] = e;
                    io.topk_w[lane] = sm.w[lane];
                    io.s2p[pos] = lane;
                    io.p2s[lane] = pos;
                }
            }
            if (lead) {
                sm.eq[qi] = e;
                sm.tq[qi] = __popc(peers);
                sm.offq[qi] = off;
            }
            const unsigned lm = __ballot_sync(0xFFFFFFFFu, lead != 0);
            if (lane == 0) *sm.nq = __popc(lm);
        }
        if (writer) {
            for (int e = threadIdx.x; e <= E; e += blockDim.x) {
                int cnt = 0, below = 0;
                for (int s = 0; s < R; ++s) {
                    const int v = sm.ids[s];
                    cnt += v == e ? 1 : 0;
                    below += v < e ? 1 : 0;
                }
                if (e < E) io.counts[e] = cnt;
                io.offsets[e] = below;
            }
        }
        __syncthreads();
        return *sm.nq;
    }
    const int nwarps = blockDim.x >> 5;
    for (int ch = warp; ch < nch; ch += nwarps) {
        const int s = ch * 32 + lane;
        const int e = s < R ? sm.ids[s] : -1;
        const unsigned peers = __match_any_sync(0xFFFFFFFFu, e);
        if (e >= 0) {
            sm.rank[s] = __popc(peers & ((1u << lane) - 1u));
            if (lane == __ffs(peers) - 1) sm.chunk[ch * E + e] = __popc(peers);
        }
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int run = 0;
        for (int ch = 0; ch < nch; ++ch) {
            const int v = sm.chunk[ch * E + e];
            sm.chunk[ch * E + e] = run;
            run += v;
        }
        sm.cnt[e] = run;
    }
    __syncthreads();
    if (warp == 0) {
        // exclusive scan of the counts, and the touched experts in ascending id order
        const int per = (E + 31) / 32;
        const int e0 = min(E, lane * per), e1 = min(E, e0 + per);
        int run = 0;
        for (int e = e0; e < e1; ++e) run += sm.cnt[e];
        int incl = run;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            if (lane >= o) incl += y;
        }
        int base = incl - run;
        for (int e = e0; e < e1; ++e) {
            sm.off[e] = base;
            base += sm.cnt[e];
        }
        if (lane == 31) sm.off[E] = incl;
        int nt = 0;
        for (int eb = 0; eb < E; eb += 32) {
            const int e = eb + lane;
            const int cnt = e < E ? sm.cnt[e] : 0;
            const unsigned m = __ballot_sync(0xFFFFFFFFu, cnt > 0);
            if (cnt > 0) {
                const int q = nt + __popc(m & ((1u << lane) - 1u));
                sm.eq[q] = e;
                sm.tq[q] = cnt;
            }
            nt += __popc(m);
        }
        if (lane == 0) *sm.nq = nt;
    }
    __syncthreads();
    const int nq = *sm.nq;
    for (int q = threadIdx.x; q < nq; q += blockDim.x) sm.offq[q] = sm.off[sm.eq[q]];
    for (int s = threadIdx.x; s < R; s += blockDim.x) {
        const int e = sm.ids[s];
        const int pos = sm.off[e] + sm.chunk[(s >> 5) * E + e] + sm.rank[s];
        sm.tok[pos] = s / io.k;
        sm.wrow[pos] = sm.w[s];
        if (sm.pos) sm.pos[s] = pos;
        if (writer) {
            io.topk_ids[s] = e;
            io.topk_w[s] = sm.w[s];
            io.s2p[pos] = s;
            io.p2s[s] = pos;
        }
    }
    if (writer) {
        for (int e = threadIdx.x; e <= E; e += blockDim.x) {
            if (e < E) io.counts[e] = sm.cnt[e];
            io.offsets[e] = sm.off[e];
        }
    }
    __syncthreads();
    return nq;
}

}  // namespace rdg
