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
//   4. copy   - one thread per 16-byte vector of a token's row: reads it once and writes it to
//               the token's k sorted positions.
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
    griddep_wait();
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
    griddep_wait();
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
    griddep_wait();
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

// Grid: x over 16-byte vectors of the row (256 per block), y over tokens (grid-stride). Each
// thread reads its vector of x once and writes it to the token's k sorted rows.
__global__ void __launch_bounds__(256) dispatch_copy_kernel(const uint4* __restrict__ x,
                                                            int T, int k, int vec_per_row,
                                                            const int32_t* __restrict__ slot_to_sorted,
                                                            uint4* __restrict__ x_sorted) {
    __shared__ int pos_s[kMaxK];
    griddep_wait();
    const int v = blockIdx.x * blockDim.x + threadIdx.x;
    for (int t = blockIdx.y; t < T; t += gridDim.y) {
        __syncthreads();
        if (threadIdx.x < k) pos_s[threadIdx.x] = __ldg(slot_to_sorted + (size_t)t * k + threadIdx.x);
        __syncthreads();
        if (v >= vec_per_row) continue;
        const uint4 val = __ldg(x + (size_t)t * vec_per_row + v);
        for (int j = 0; j < k; ++j) {
            const int p = pos_s[j];
            if (p >= 0) x_sorted[(size_t)p * vec_per_row + v] = val;
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
    cudaError_t e = cudaSuccess;
    if (blocks > 0 &&
        (e = launch_kernel(dispatch_hist_kernel, dim3(blocks), dim3(32 * kWarpsPerBlock), 0, s,
                           ids, R, E, nchunks, chunk_scratch, status)) != cudaSuccess)
        return e;
    if ((e = launch_kernel(dispatch_scan_kernel, dim3(1), dim3(1024), 0, s, chunk_scratch,
                           nchunks, E, counts, offsets)) != cudaSuccess)
        return e;
    if (blocks > 0 &&
        (e = launch_kernel(dispatch_rank_kernel, dim3(blocks), dim3(32 * kWarpsPerBlock), 0, s,
                           ids, R, E, nchunks, (const int32_t*)chunk_scratch, sorted_to_slot,
                           slot_to_sorted)) != cudaSuccess)
        return e;
    if (T > 0 && x != nullptr && x_sorted != nullptr)
        return launch_dispatch_copy(x, row_bytes, T, k, slot_to_sorted, x_sorted, s);
    return cudaGetLastError();
}

cudaError_t launch_dispatch_copy(const void* x, size_t row_bytes, int T, int k,
                                 const int32_t* slot_to_sorted, void* x_sorted, cudaStream_t s) {
    const int vec = (int)(row_bytes / 16);
    const dim3 grid((vec + 255) / 256, T < 65535 ? T : 65535);
    return launch_kernel(dispatch_copy_kernel, grid, dim3(256), 0, s,
                         static_cast<const uint4*>(x), T, k, vec, slot_to_sorted,
                         static_cast<uint4*>(x_sorted));
}

}  // namespace rdg
