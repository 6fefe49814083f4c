// Dispatch: group the R = T*k routed slots by expert and copy each token's row to the sorted
// positions of its slots.
//
// Expert parallelism page, "Token dispatch": each (token, expert) pair is sent to the rank that
// owns the expert. On one GPU that exchange is this local permutation. Row order inside an
// expert is ascending slot order, fixed without atomics so the permutation is bit-reproducible.
//
// Four kernels:
//   1. hist   - one warp per chunk of 256 slots: per-chunk expert counts (warp match + popc).
//   2. scan   - one block: counts[E], offsets[E+1] and, per (chunk, expert), the first sorted
//               position that chunk writes for that expert.
//   3. rank   - one warp per chunk: walks its slots in order, 32 at a time; a slot's position
//               is the chunk base for its expert plus the number of earlier slots of the chunk
//               routed to the same expert.
//   4. copy   - one warp per token: reads the token's row once (16-byte vectors) and writes it
//               to the k sorted positions.
#include "moe_internal.cuh"

namespace rdg {
namespace {

constexpr int kWarpsPerBlock = 8;

__device__ __forceinline__ bool valid_id(int e, int E) { return e >= 0 && e < E; }

__global__ void __launch_bounds__(256) dispatch_hist_kernel(const int32_t* __restrict__ ids,
                                                            int R, int E, int nchunks,
                                                            int32_t* __restrict__ chunk_counts,
                                                            int* status) {
    __shared__ int cnt[kWarpsPerBlock][kMaxE];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int c = blockIdx.x * kWarpsPerBlock + w;
    if (c >= nchunks) return;
    for (int e = lane; e < E; e += 32) cnt[w][e] = 0;
    __syncwarp();
    bool bad = false;
    for (int r = 0; r < kDispatchChunk / 32; ++r) {
        const int s = c * kDispatchChunk + r * 32 + lane;
        int e = -1;
        if (s < R) {
            e = __ldg(ids + s);
            if (!valid_id(e, E)) {
                bad = true;
                e = -1;
            }
        }
        const unsigned peers = __match_any_sync(0xFFFFFFFFu, e);
        if (e >= 0 && lane == __ffs(peers) - 1) cnt[w][e] += __popc(peers);
        __syncwarp();
    }
    if (bad) set_status(status, MOE_ERR_DEVICE_BOUNDS);
    for (int e = lane; e < E; e += 32) chunk_counts[(size_t)c * E + e] = cnt[w][e];
}

// One block of 1024 threads. Thread (g, e) with g < G = 1024 / E owns chunks
// [g*L, min(nchunks, (g+1)*L)) of expert e. chunk_counts is overwritten in place by the chunk
// bases.
__global__ void __launch_bounds__(1024) dispatch_scan_kernel(int32_t* __restrict__ chunk,
                                                             int nchunks, int E,
                                                             int32_t* __restrict__ counts,
                                                             int32_t* __restrict__ offsets) {
    __shared__ int part[1024];
    __shared__ int tot[kMaxE];
    __shared__ int off[kMaxE + 1];
    const int tid = threadIdx.x;
    const int G = blockDim.x / E;
    const int L = (nchunks + G - 1) / G;
    const int e = tid % E, g = tid / E;
    const bool active = g < G;
    int c0 = 0, c1 = 0;
    if (active) {
        c0 = min(nchunks, g * L);
        c1 = min(nchunks, c0 + L);
        int sum = 0;
        for (int c = c0; c < c1; ++c) sum += chunk[(size_t)c * E + e];
        part[g * E + e] = sum;
    }
    __syncthreads();
    if (tid < E) {
        int run = 0;
        for (int gg = 0; gg < G; ++gg) {
            const int v = part[gg * E + tid];
            part[gg * E + tid] = run;
            run += v;
        }
        tot[tid] = run;
    }
    __syncthreads();
    if (tid < 32) {
        // exclusive scan over experts: lane handles a contiguous run of experts
        const int per = (E + 31) / 32;
        const int e0 = min(E, tid * per), e1 = min(E, e0 + per);
        int run = 0;
        for (int x = e0; x < e1; ++x) run += tot[x];
        int incl = run;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            if (tid >= o) incl += y;
        }
        int base = incl - run;
        for (int x = e0; x < e1; ++x) {
            off[x] = base;
            base += tot[x];
        }
        if (tid == 31) off[E] = incl;
    }
    __syncthreads();
    if (tid < E) counts[tid] = tot[tid];
    if (tid <= E) offsets[tid] = off[tid];
    if (active) {
        int base = off[e] + part[g * E + e];
        for (int c = c0; c < c1; ++c) {
            const int v = chunk[(size_t)c * E + e];
            chunk[(size_t)c * E + e] = base;
            base += v;
        }
    }
}

__global__ void __launch_bounds__(256) dispatch_rank_kernel(const int32_t* __restrict__ ids,
                                                            int R, int E, int nchunks,
                                                            const int32_t* __restrict__ chunk_base,
                                                            int32_t* __restrict__ sorted_to_slot,
                                                            int32_t* __restrict__ slot_to_sorted) {
    __shared__ int run[kWarpsPerBlock][kMaxE];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int c = blockIdx.x * kWarpsPerBlock + w;
    if (c >= nchunks) return;
    for (int e = lane; e < E; e += 32) run[w][e] = chunk_base[(size_t)c * E + e];
    __syncwarp();
    const unsigned lt = (1u << lane) - 1u;
    for (int r = 0; r < kDispatchChunk / 32; ++r) {
        const int s = c * kDispatchChunk + r * 32 + lane;
        int e = -1;
        if (s < R) {
            e = __ldg(ids + s);
            if (!valid_id(e, E)) e = -1;
        }
        const unsigned peers = __match_any_sync(0xFFFFFFFFu, e);
        if (e >= 0) {
            const int pos = run[w][e] + __popc(peers & lt);
            sorted_to_slot[pos] = s;
            slot_to_sorted[s] = pos;
        } else if (s < R) {
            slot_to_sorted[s] = -1;
        }
        __syncwarp();
        if (e >= 0 && lane == 31 - __clz(peers)) run[w][e] += __popc(peers);
        __syncwarp();
    }
}

// One warp per token (grid-stride). Rows are moved as 16-byte vectors.
__global__ void __launch_bounds__(256) dispatch_copy_kernel(const uint4* __restrict__ x,
                                                            int T, int k, int vec_per_row,
                                                            const int32_t* __restrict__ slot_to_sorted,
                                                            uint4* __restrict__ x_sorted) {
    const int lane = threadIdx.x & 31;
    const int warps_total = gridDim.x * (blockDim.x >> 5);
    for (int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); t < T; t += warps_total) {
        const int my_pos = (lane < k) ? __ldg(slot_to_sorted + (size_t)t * k + lane) : -1;
        const uint4* src = x + (size_t)t * vec_per_row;
        // uniform trip count: every lane takes part in each shuffle
        for (int base = 0; base < vec_per_row; base += 32) {
            const int v = base + lane;
            const bool in = v < vec_per_row;
            const uint4 val = in ? __ldg(src + v) : make_uint4(0u, 0u, 0u, 0u);
            for (int j = 0; j < k; ++j) {
                const int p = __shfl_sync(0xFFFFFFFFu, my_pos, j);
                if (in && p >= 0) x_sorted[(size_t)p * vec_per_row + v] = val;
            }
        }
    }
}

}  // namespace

size_t dispatch_scratch_bytes(int R, int E) {
    const size_t nchunks = ((size_t)R + kDispatchChunk - 1) / kDispatchChunk;
    return nchunks * (size_t)E * sizeof(int32_t);
}

int dispatch_kernel_count(bool copy_rows) { return copy_rows ? 4 : 3; }

cudaError_t launch_dispatch(const int32_t* ids, const void* x, size_t row_bytes, int T, int E,
                            int k, int32_t* counts, int32_t* offsets, int32_t* sorted_to_slot,
                            int32_t* slot_to_sorted, void* x_sorted, int32_t* chunk_scratch,
                            int* status, cudaStream_t s) {
    const int R = T * k;
    const int nchunks = (R + kDispatchChunk - 1) / kDispatchChunk;
    const int blocks = (nchunks + kWarpsPerBlock - 1) / kWarpsPerBlock;
    // With no slots only the scan runs: it writes zero counts and offsets.
    if (blocks > 0)
        dispatch_hist_kernel<<<blocks, 32 * kWarpsPerBlock, 0, s>>>(ids, R, E, nchunks,
                                                                    chunk_scratch, status);
    dispatch_scan_kernel<<<1, 1024, 0, s>>>(chunk_scratch, nchunks, E, counts, offsets);
    if (blocks > 0)
        dispatch_rank_kernel<<<blocks, 32 * kWarpsPerBlock, 0, s>>>(
            ids, R, E, nchunks, chunk_scratch, sorted_to_slot, slot_to_sorted);
    if (T > 0 && x != nullptr && x_sorted != nullptr) {
        const int vec = (int)(row_bytes / 16);
        const int max_blocks = device_sm_count() * 8;
        int cblocks = (T + kWarpsPerBlock - 1) / kWarpsPerBlock;
        if (cblocks > max_blocks) cblocks = max_blocks;
        dispatch_copy_kernel<<<cblocks, 32 * kWarpsPerBlock, 0, s>>>(
            static_cast<const uint4*>(x), T, k, vec, slot_to_sorted, static_cast<uint4*>(x_sorted));
    }
    return cudaGetLastError();
}

}  // namespace rdg
