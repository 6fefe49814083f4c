// Router from hidden states: logits = x . W_r (+ b) in fp32, then the router top-k, in one
// kernel.
//
// Expert parallelism page, introduction: a router sends each token to its experts; the
// workloads define the router's logits as the hidden states times a router weight [d, E]
// (plus a per-expert bias on two of them). This is the step right before the routing kernel;
// fusing it saves writing the [T, E] logits and reading them back, and gives decode one launch
// less. The top-k and weights are the warp router of route.cu (route_select_warp), fed from
// registers, so for the same logits the ids and weights are bit-identical to moe_route.
//
// More than 1024 tokens of bf16 x run on the tensor pipe (route_hidden_mma_kernel below);
// otherwise on the FP32 pipes. FP32-pipe layout: a block has 8 warps; lane l accumulates
// experts l, l+32, ... of 8 tokens (the register layout the warp router reads). K is walked
// in chunks of 64 rows staged in shared memory (x as fp32, W_r); the loads of chunk c + 1 are
// issued into registers before chunk c is multiplied, so their latency hides behind the FMAs.
//   - large batches (KS = 1): warp w owns tokens 8w .. 8w+7 of the block's 64 and sums each
//     logit over K in ascending order;
//   - small batches (KS = 8): a cluster of 8 blocks shares 8 tokens; block r of the cluster
//     takes K rows [r D, r D + D) (D = d/8 rounded up to the chunk), its 8 warps split each
//     chunk's rows (warp w takes rows w, w+8, ...) and add their sums in warp order; block 0
//     then adds the 8 blocks' sums in rank order from their shared memory (distributed shared
//     memory within the cluster) and selects.
// Either way every logit's summation order is fixed by the sizes, so results do not depend on
// timing.

#include "route_warp.cuh"

namespace rdg {
namespace {

constexpr int kWarps = 8;
constexpr int kTokPerWarp = 8;
constexpr int kChunk = 64;  // K rows per shared-memory step
constexpr int kCluster = 8; // blocks per cluster on the small-batch path

__device__ __forceinline__ uint32_t cta_rank_in_cluster() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
                 ::: "memory");
}
__device__ __forceinline__ float ld_cluster_f32(const float* local, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
                 : "=r"(remote)
                 : "r"(smem_u32(local)), "r"(rank));
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
    return v;
}

template <int VPL, int KS>
struct RhShape {
    static constexpr int kTok = kWarps / KS * kTokPerWarp;               // tokens per block
    static constexpr int kXPer = kTok * kChunk / (kWarps * 32);           // x values per thread
    static constexpr int kWPer = kChunk * VPL * 32 / (kWarps * 32);       // W values per thread
    static constexpr size_t kSmem = (size_t)(kTok * (kChunk + 1) + kChunk * VPL * 32) * 4 +
                                    (KS > 1 ? (size_t)kWarps * kTokPerWarp * VPL * 32 * 4 : 0);
};

template <int VPL, bool kBf16, int KS>
__global__ void __launch_bounds__(kWarps * 32)
route_hidden_kernel(const void* __restrict__ x_raw, const float* __restrict__ w_router,
                    const float* __restrict__ bias, int T, int d, int E, int k, int score_fn,
                    int renorm, float* __restrict__ logits, int32_t* __restrict__ ids,
                    float* __restrict__ weights) {
    using S = RhShape<VPL, KS>;
    extern __shared__ float rh_smem[];
    float* xs = rh_smem;                          // [kTok][kChunk + 1]
    float* ws = xs + S::kTok * (kChunk + 1);      // [kChunk][VPL * 32]
    float* red = ws + kChunk * VPL * 32;          // [kWarps][8][VPL * 32] (KS > 1)
    griddep_wait();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    // KS = 1: one block per 64 tokens, all of K. KS > 1: a cluster per 8 tokens, block r of
    // it taking K rows [k_lo, k_hi)
    const int crank = (KS == 1) ? 0 : (int)cta_rank_in_cluster();
    const int t0 = (KS == 1 ? blockIdx.x : blockIdx.x / kCluster) * S::kTok;
    const int k_span = (KS == 1) ? d : ((d + kCluster * kChunk - 1) / (kCluster * kChunk)) * kChunk;
    const int k_lo = crank * k_span, k_hi = min(d, k_lo + k_span);
    const int tg = (KS == 1) ? warp : 0;          // this warp's 8 tokens within the block
    const int ks = (KS == 1) ? 0 : warp;          // this warp's rows: ks, ks + KS, ...

    float acc[kTokPerWarp][VPL];
#pragma unroll
    for (int t = 0; t < kTokPerWarp; ++t)
#pragma unroll
        for (int j = 0; j < VPL; ++j) acc[t][j] = 0.0f;

    // thread i of the block loads x element (i + 256 m) and W element (i + 256 m) of a chunk
    float xr[S::kXPer], wr[S::kWPer];
    auto load_chunk = [&](int k0) {
#pragma unroll
        for (int m = 0; m < S::kXPer; ++m) {
            const int i = threadIdx.x + m * kWarps * 32;
            const int t = i / kChunk, kk = i % kChunk;
            const int tok = t0 + t, col = k0 + kk;
            float v = 0.0f;
            if (tok < T && col < k_hi) {
                if (kBf16)
                    v = __bfloat162float(
                        static_cast<const __nv_bfloat16*>(x_raw)[(size_t)tok * d + col]);
                else
                    v = static_cast<const float*>(x_raw)[(size_t)tok * d + col];
            }
            xr[m] = v;
        }
#pragma unroll
        for (int m = 0; m < S::kWPer; ++m) {
            const int i = threadIdx.x + m * kWarps * 32;
            const int kk = i / (VPL * 32), e = i % (VPL * 32);
            const int row = k0 + kk;
            wr[m] = (row < k_hi && e < E) ? __ldg(w_router + (size_t)row * E + e) : 0.0f;
        }
    };
    auto store_chunk = [&]() {
#pragma unroll
        for (int m = 0; m < S::kXPer; ++m) {
            const int i = threadIdx.x + m * kWarps * 32;
            xs[(i / kChunk) * (kChunk + 1) + i % kChunk] = xr[m];
        }
#pragma unroll
        for (int m = 0; m < S::kWPer; ++m) ws[threadIdx.x + m * kWarps * 32] = wr[m];
    };

    if (k_lo < k_hi) load_chunk(k_lo);
    for (int k0 = k_lo; k0 < k_hi; k0 += kChunk) {
        store_chunk();
        __syncthreads();
        if (k0 + kChunk < k_hi) load_chunk(k0 + kChunk);  // in flight during the FMAs below
#pragma unroll 4
        for (int kk = ks; kk < kChunk; kk += KS) {
            float w[VPL];
#pragma unroll
            for (int j = 0; j < VPL; ++j) w[j] = ws[kk * VPL * 32 + lane + 32 * j];
#pragma unroll
            for (int t = 0; t < kTokPerWarp; ++t) {
                const float xv = xs[(tg * kTokPerWarp + t) * (kChunk + 1) + kk];
#pragma unroll
                for (int j = 0; j < VPL; ++j) acc[t][j] = fmaf(xv, w[j], acc[t][j]);
            }
        }
        __syncthreads();
    }

    if (KS > 1) {
        // add the warps' partial sums in warp order (warp 0 keeps the block's sum in red
        // slot 0), then the blocks' sums in rank order (block 0, through distributed shared
        // memory); every block stays until block 0 has read its sum
#pragma unroll
        for (int t = 0; t < kTokPerWarp; ++t)
#pragma unroll
            for (int j = 0; j < VPL; ++j)
                red[((warp * kTokPerWarp) + t) * VPL * 32 + lane + 32 * j] = acc[t][j];
        __syncthreads();
        if (warp == 0) {
#pragma unroll
            for (int t = 0; t < kTokPerWarp; ++t)
#pragma unroll
                for (int j = 0; j < VPL; ++j) {
                    float s = 0.0f;
                    for (int w = 0; w < kWarps; ++w)
                        s += red[((w * kTokPerWarp) + t) * VPL * 32 + lane + 32 * j];
                    acc[t][j] = s;
                }
        }
        __syncthreads();  // every warp has read red before warp 0 overwrites slot 0
        if (warp == 0) {
#pragma unroll
            for (int t = 0; t < kTokPerWarp; ++t)
#pragma unroll
                for (int j = 0; j < VPL; ++j) red[t * VPL * 32 + lane + 32 * j] = acc[t][j];
        }
        cluster_sync_all();
        if (crank == 0 && warp == 0) {
#pragma unroll
            for (int t = 0; t < kTokPerWarp; ++t)
#pragma unroll
                for (int j = 0; j < VPL; ++j) {
                    float s = 0.0f;
                    for (int r = 0; r < kCluster; ++r)
                        s += ld_cluster_f32(red + t * VPL * 32 + lane + 32 * j, (uint32_t)r);
                    acc[t][j] = s;
                }
        }
        cluster_sync_all();
        if (crank != 0 || warp != 0) return;
    }

#pragma unroll
    for (int t = 0; t < kTokPerWarp; ++t) {
        const int tok = t0 + tg * kTokPerWarp + t;
        if (tok >= T) break;  // uniform across the warp
        float v[VPL];
#pragma unroll
        for (int j = 0; j < VPL; ++j) {
            const int e = lane + 32 * j;
            v[j] = -INFINITY;
            if (e < E) {
                v[j] = bias ? acc[t][j] + __ldg(bias + e) : acc[t][j];
                if (logits) logits[(size_t)tok * E + e] = v[j];
            }
        }
        int id;
        float wt;
        route_select_warp<VPL>(v, E, k, score_fn, renorm, lane, &id, &wt);
        if (lane < k) {
            ids[(size_t)tok * k + lane] = id;
            weights[(size_t)tok * k + lane] = wt;
        }
    }
}

// ---- large batches of bf16 x on the tensor pipe ----
// logits[64 tokens][EPAD experts] of a block = x (bf16, exact) times W_r split into three bf16
// terms hi + mid + lo (together about 24 significant bits), each product on mma.sync
// m16n8k16 with fp32 accumulation; K in chunks of 64 (the next chunk's loads in flight during
// the MMAs). Warp w: tokens 16 (w % 4) .. +15, experts EPAD/2 * (w / 4) .. +EPAD/2. Then the
// logits go through shared memory to the warp router's register layout (8 tokens per warp).
template <int EPAD>
struct MmaShape {
    static constexpr int kNT = EPAD / 16;                 // n-tiles of 8 experts per warp
    static constexpr int kXStride = kChunk * 2 + 16;      // bytes per x row (padded)
    static constexpr int kWStride = EPAD * 2 + 16;        // bytes per W row of one plane
    static constexpr int kXBytes = 64 * kXStride;
    static constexpr int kPlaneBytes = kChunk * kWStride;
    static constexpr int kWPer = kChunk * EPAD / 256;     // W values per thread per chunk
    static constexpr size_t kSmem = (size_t)kXBytes + 3 * kPlaneBytes;
    static_assert(3 * kPlaneBytes >= 64 * EPAD * 4, "logits must fit in the W planes");
};

template <int EPAD>
__global__ void __launch_bounds__(256)
route_hidden_mma_kernel(const __nv_bfloat16* __restrict__ x, const float* __restrict__ w_router,
                        const float* __restrict__ bias, int T, int d, int E, int k,
                        int score_fn, int renorm, float* __restrict__ logits,
                        int32_t* __restrict__ ids, float* __restrict__ weights) {
    using S = MmaShape<EPAD>;
    extern __shared__ __align__(16) uint8_t rm_smem[];
    uint8_t* xs = rm_smem;
    uint8_t* wp = rm_smem + S::kXBytes;  // planes hi, mid, lo
    griddep_wait();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int t0 = blockIdx.x * 64;
    const int m0 = 16 * (warp & 3), n_base = (EPAD / 2) * (warp >> 2);

    float acc[S::kNT][4];
#pragma unroll
    for (int n = 0; n < S::kNT; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.0f;

    uint4 xr[2];
    float wr[S::kWPer];
    auto load_chunk = [&](int k0) {
#pragma unroll
        for (int m = 0; m < 2; ++m) {  // 64 rows x 8 vectors of 8 bf16
            const int i = threadIdx.x + 256 * m, r = i >> 3, c = (i & 7) * 8;
            const int tok = t0 + r, col = k0 + c;
            xr[m] = (tok < T && col < d)
                        ? __ldg(reinterpret_cast<const uint4*>(x + (size_t)tok * d + col))
                        : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int m = 0; m < S::kWPer; ++m) {
            const int i = threadIdx.x + 256 * m, r = i / EPAD, e = i % EPAD;
            const int row = k0 + r;
            wr[m] = (row < d && e < E) ? __ldg(w_router + (size_t)row * E + e) : 0.0f;
        }
    };
    auto store_chunk = [&]() {
#pragma unroll
        for (int m = 0; m < 2; ++m) {
            const int i = threadIdx.x + 256 * m, r = i >> 3, c = (i & 7) * 8;
            *reinterpret_cast<uint4*>(xs + r * S::kXStride + c * 2) = xr[m];
        }
#pragma unroll
        for (int m = 0; m < S::kWPer; ++m) {
            const int i = threadIdx.x + 256 * m, r = i / EPAD, e = i % EPAD;
            const float w = wr[m];
            const __nv_bfloat16 hi = __float2bfloat16_rn(w);
            const float r1 = w - __bfloat162float(hi);
            const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
            const __nv_bfloat16 lo = __float2bfloat16_rn(r1 - __bfloat162float(mid));
            const int off = r * S::kWStride + e * 2;
            *reinterpret_cast<__nv_bfloat16*>(wp + off) = hi;
            *reinterpret_cast<__nv_bfloat16*>(wp + S::kPlaneBytes + off) = mid;
            *reinterpret_cast<__nv_bfloat16*>(wp + 2 * S::kPlaneBytes + off) = lo;
        }
    };

    load_chunk(0);
    for (int k0 = 0; k0 < d; k0 += kChunk) {
        store_chunk();
        __syncthreads();
        if (k0 + kChunk < d) load_chunk(k0 + kChunk);
#pragma unroll
        for (int ks = 0; ks < kChunk / 16; ++ks) {
            // A: rows m0 + (l & 15), columns 16 ks + 8 (l >> 4) (ldmatrix.x4)
            uint32_t a0, a1, a2, a3;
            const uint32_t a_addr = smem_u32(xs + (m0 + (lane & 15)) * S::kXStride +
                                             (16 * ks + 8 * (lane >> 4)) * 2);
            asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                         : "=r"(a0), "=r"(a1), "=r"(a2), "=r"(a3)
                         : "r"(a_addr));
#pragma unroll
            for (int np = 0; np < S::kNT / 2; ++np) {
                // B of two n-tiles: rows 16 ks + (l & 7) + 8 ((l >> 3) & 1), columns
                // n_base + 16 np + 8 (l >> 4) (ldmatrix.x4.trans from the [k][e] plane)
                const int brow = 16 * ks + (lane & 7) + 8 * ((lane >> 3) & 1);
                const int bcol = n_base + 16 * np + 8 * (lane >> 4);
#pragma unroll
                for (int pl = 0; pl < 3; ++pl) {
                    uint32_t b0, b1, b2, b3;
                    const uint32_t b_addr =
                        smem_u32(wp + pl * S::kPlaneBytes + brow * S::kWStride + bcol * 2);
                    asm volatile(
                        "ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                        : "=r"(b0), "=r"(b1), "=r"(b2), "=r"(b3)
                        : "r"(b_addr));
                    asm volatile(
                        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
                        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
                        : "+f"(acc[2 * np][0]), "+f"(acc[2 * np][1]), "+f"(acc[2 * np][2]),
                          "+f"(acc[2 * np][3])
                        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
                    asm volatile(
                        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
                        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
                        : "+f"(acc[2 * np + 1][0]), "+f"(acc[2 * np + 1][1]),
                          "+f"(acc[2 * np + 1][2]), "+f"(acc[2 * np + 1][3])
                        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b2), "r"(b3));
                }
            }
        }
        __syncthreads();
    }

    // C fragments (token m0 + l/4 [+8], expert 2 (l%4) [+1]) -> logits in shared memory
    float* ls = reinterpret_cast<float*>(wp);  // [64][EPAD]
#pragma unroll
    for (int n = 0; n < S::kNT; ++n) {
        const int e = n_base + 8 * n + 2 * (lane & 3), r = m0 + (lane >> 2);
        ls[r * EPAD + e] = acc[n][0];
        ls[r * EPAD + e + 1] = acc[n][1];
        ls[(r + 8) * EPAD + e] = acc[n][2];
        ls[(r + 8) * EPAD + e + 1] = acc[n][3];
    }
    __syncthreads();
    constexpr int VPL = EPAD / 32;
#pragma unroll 1
    for (int t = 0; t < 8; ++t) {
        const int r = 8 * warp + t, tok = t0 + r;
        if (tok >= T) break;  // uniform across the warp
        float v[VPL];
#pragma unroll
        for (int j = 0; j < VPL; ++j) {
            const int e = lane + 32 * j;
            v[j] = -INFINITY;
            if (e < E) {
                v[j] = bias ? ls[r * EPAD + e] + __ldg(bias + e) : ls[r * EPAD + e];
                if (logits) logits[(size_t)tok * E + e] = v[j];
            }
        }
        int id;
        float wt;
        route_select_warp<VPL>(v, E, k, score_fn, renorm, lane, &id, &wt);
        if (lane < k) {
            ids[(size_t)tok * k + lane] = id;
            weights[(size_t)tok * k + lane] = wt;
        }
    }
}

template <int EPAD>
cudaError_t launch_mma(const void* x, const float* w_router, const float* bias, int T, int d,
                       int E, int k, int score_fn, int renorm, float* logits, int32_t* ids,
                       float* weights, cudaStream_t s) {
    using S = MmaShape<EPAD>;
    {
        const cudaError_t e = ensure_max_dynamic_smem(route_hidden_mma_kernel<EPAD>, (int)S::kSmem);
        if (e != cudaSuccess) return e;
    }
    return launch_kernel(route_hidden_mma_kernel<EPAD>, dim3((T + 63) / 64), dim3(256), S::kSmem,
                         s, static_cast<const __nv_bfloat16*>(x), w_router, bias, T, d, E, k,
                         score_fn, renorm, logits, ids, weights);
}

template <int VPL, int KS>
cudaError_t launch_shape(const void* x, bool bf16, const float* w_router, const float* bias,
                         int T, int d, int E, int k, int score_fn, int renorm, float* logits,
                         int32_t* ids, float* weights, cudaStream_t s) {
    using S = RhShape<VPL, KS>;
    auto kern = bf16 ? route_hidden_kernel<VPL, true, KS> : route_hidden_kernel<VPL, false, KS>;
    if (S::kSmem > 48 * 1024) {
        const cudaError_t e = ensure_max_dynamic_smem(kern, (int)S::kSmem);
        if (e != cudaSuccess) return e;
    }
    const int groups = (T + S::kTok - 1) / S::kTok;
    const int cl = KS > 1 ? kCluster : 1;
    return launch_kernel_ex(kern, dim3((unsigned)(groups * cl)), dim3(kWarps * 32), S::kSmem, s,
                            cl, x, w_router, bias, T, d, E, k, score_fn, renorm, logits, ids,
                            weights);
}

template <int VPL>
cudaError_t launch_vpl(const void* x, bool bf16, const float* w_router, const float* bias, int T,
                       int d, int E, int k, int score_fn, int renorm, float* logits,
                       int32_t* ids, float* weights, cudaStream_t s) {
    // up to 1024 tokens: a cluster of 8 blocks per 8 tokens, K split over blocks and warps
    // (many blocks, short dependent chains); beyond: 64 tokens per block
    if (T <= 1024)
        return launch_shape<VPL, 8>(x, bf16, w_router, bias, T, d, E, k, score_fn, renorm,
                                    logits, ids, weights, s);
    return launch_shape<VPL, 1>(x, bf16, w_router, bias, T, d, E, k, score_fn, renorm, logits,
                                ids, weights, s);
}

}  // namespace

cudaError_t launch_route_hidden(const void* x, bool bf16, const float* w_router,
                                const float* bias, int T, int d, int E, int k, int score_fn,
                                bool renorm, float* logits, int32_t* ids, float* weights,
                                cudaStream_t s) {
    const int rn = renorm ? 1 : 0;
    // more than 1024 tokens of bf16 x (and d a multiple of 8): the tensor-pipe kernel
    if (bf16 && T > 1024 && d % 8 == 0) {
        if (E <= 64) return launch_mma<64>(x, w_router, bias, T, d, E, k, score_fn, rn, logits, ids, weights, s);
        if (E <= 128) return launch_mma<128>(x, w_router, bias, T, d, E, k, score_fn, rn, logits, ids, weights, s);
        return launch_mma<256>(x, w_router, bias, T, d, E, k, score_fn, rn, logits, ids, weights, s);
    }
    if (E <= 32) return launch_vpl<1>(x, bf16, w_router, bias, T, d, E, k, score_fn, rn, logits, ids, weights, s);
    if (E <= 64) return launch_vpl<2>(x, bf16, w_router, bias, T, d, E, k, score_fn, rn, logits, ids, weights, s);
    if (E <= 128) return launch_vpl<4>(x, bf16, w_router, bias, T, d, E, k, score_fn, rn, logits, ids, weights, s);
    return launch_vpl<8>(x, bf16, w_router, bias, T, d, E, k, score_fn, rn, logits, ids, weights, s);
}

}  // namespace rdg
