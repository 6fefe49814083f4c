// Backward pass of the expert layer: the small kernels and the fp32-layer GEMMs.
//
// The routing weights multiply the expert outputs (Expert parallelism page, introduction and
// "Token dispatch": the results are combined with the routing weights), so the loss reaches
// them and, through the router's score function, the logits:
//   combine backward: dy[p] = w[t, j] dout[t] for p = slot_to_sorted[t k + j] (rounded to the
//     layer dtype) and d w[t, j] = dout[t] . y_sorted[p] (fp32, a fixed-order block sum);
//   scale gradient (the score scales the expert input): d w[slot of p] = the sum of the SwiGLU
//     backward's per-tile partials of row p, in tile order;
//   router backward: the Jacobian of the routing weights with respect to the logits, the
//     selected experts held fixed (softmax over all experts or over the selected ones, sigmoid
//     with or without renormalisation);
//   fp32 layers: the dgrad and wgrad GEMMs on the FFMA pipes (no TF32), same contracts as the
//     tensor-core kernels.
#include "moe_internal.cuh"

namespace rdg {
namespace {

__device__ __forceinline__ float4 load4(const float* p, size_t i4) {
    return __ldg(reinterpret_cast<const float4*>(p) + i4);
}
__device__ __forceinline__ float4 load4(const __nv_bfloat16* p, size_t i4) {
    const uint2 u = __ldg(reinterpret_cast<const uint2*>(p) + i4);
    return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u),
                       __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xFFFF0000u));
}
__device__ __forceinline__ void store4(float* p, size_t i4, float4 v) {
    reinterpret_cast<float4*>(p)[i4] = v;
}
__device__ __forceinline__ void store4(__nv_bfloat16* p, size_t i4, float4 v) {
    reinterpret_cast<uint2*>(p)[i4] = make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
}

// Sum of one value per thread of a 256-thread block, in a fixed order (warp trees, then the
// eight warp sums in warp order); the result is valid in thread 0.
__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    const int warp = threadIdx.x >> 5;
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[warp] = v;
    __syncthreads();
    float s = 0.0f;
    if (threadIdx.x == 0)
        for (int w = 0; w < 8; ++w) s += red[w];
    return s;
}

// One block per token (grid-stride). Thread i owns the 4-column groups i, i + 256, ...
template <typename T>
__global__ void __launch_bounds__(256)
    combine_backward_kernel(const T* __restrict__ dout, const float* __restrict__ y, int tokens,
                            int d4, int k, const int32_t* __restrict__ slot_to_sorted,
                            const float* __restrict__ weights, T* __restrict__ dy,
                            float* __restrict__ dw) {
    __shared__ int pos_s[kMaxK];
    __shared__ float w_s[kMaxK];
    __shared__ float red[8];
    griddep_wait();
    for (int t = blockIdx.x; t < tokens; t += gridDim.x) {
        __syncthreads();
        if (threadIdx.x < k) {
            pos_s[threadIdx.x] = __ldg(slot_to_sorted + (size_t)t * k + threadIdx.x);
            w_s[threadIdx.x] = weights ? __ldg(weights + (size_t)t * k + threadIdx.x) : 1.0f;
        }
        __syncthreads();
        for (int j = 0; j < k; ++j) {
            const int p = pos_s[j];
            const float w = w_s[j];
            float part = 0.0f;
            if (p >= 0) {
                for (int c = threadIdx.x; c < d4; c += 256) {
                    const float4 g = load4(dout, (size_t)t * d4 + c);
                    store4(dy, (size_t)p * d4 + c, make_float4(w * g.x, w * g.y, w * g.z, w * g.w));
                    if (dw) {
                        const float4 v = load4(y, (size_t)p * d4 + c);
                        part = fmaf(g.x, v.x, fmaf(g.y, v.y, fmaf(g.z, v.z, fmaf(g.w, v.w, part))));
                    }
                }
            }
            if (dw) {
                const float s = block_sum(part, red);
                if (threadIdx.x == 0) dw[(size_t)t * k + j] = p >= 0 ? s : 0.0f;
            }
        }
    }
}

// d w[slot] = sum over tiles of scale_part[p][tile], one thread per sorted row p.
__global__ void __launch_bounds__(256)
    scale_grad_kernel(const float* __restrict__ part, int R, int n_tiles,
                      const int32_t* __restrict__ sorted_to_slot, float* __restrict__ dw) {
    griddep_wait();
    const int p = blockIdx.x * blockDim.x + threadIdx.x;
    if (p >= R) return;
    float s = 0.0f;
    for (int i = 0; i < n_tiles; ++i) s += __ldg(part + (size_t)p * n_tiles + i);
    dw[__ldg(sorted_to_slot + p)] = s;
}

// One warp per token; lane l handles experts l, l + 32, ...
__global__ void __launch_bounds__(256)
    route_backward_kernel(const float* __restrict__ logits, const int32_t* __restrict__ ids,
                          const float* __restrict__ weights, const float* __restrict__ d_weights,
                          int T, int E, int k, int score_fn, int renorm,
                          float* __restrict__ d_logits) {
    griddep_wait();
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t >= T) return;
    const float* row = logits + (size_t)t * E;
    // slot j lives in lane j (k <= 32)
    const int id = lane < k ? __ldg(ids + (size_t)t * k + lane) : -1;
    const float w = lane < k ? __ldg(weights + (size_t)t * k + lane) : 0.0f;
    const float g = lane < k ? __ldg(d_weights + (size_t)t * k + lane) : 0.0f;
    float inner = w * g;  // sum_j w_j g_j
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) inner += __shfl_xor_sync(0xFFFFFFFFu, inner, o);
    float sig_sum = 0.0f, mx = -INFINITY, denom = 0.0f;
    if (score_fn == MOE_SCORE_SIGMOID && renorm) {
        float sg = lane < k ? 1.0f / (1.0f + expf(-__ldg(row + id))) : 0.0f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sg += __shfl_xor_sync(0xFFFFFFFFu, sg, o);
        sig_sum = sg;
    }
    if (score_fn == MOE_SCORE_SOFTMAX && !renorm) {
        for (int m = lane; m < E; m += 32) mx = fmaxf(mx, __ldg(row + m));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
        for (int m = lane; m < E; m += 32) denom += expf(__ldg(row + m) - mx);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) denom += __shfl_xor_sync(0xFFFFFFFFu, denom, o);
    }
    for (int m0 = 0; m0 < E; m0 += 32) {
        const int m = m0 + lane;
        // the slot holding expert m, if any (the k ids of a token are distinct)
        int slot = -1;
        for (int j = 0; j < k; ++j)
            if (__shfl_sync(0xFFFFFFFFu, id, j) == m) slot = j;
        float wj = 0.0f, gj = 0.0f;
        for (int j = 0; j < k; ++j) {
            const float wv = __shfl_sync(0xFFFFFFFFu, w, j);
            const float gv = __shfl_sync(0xFFFFFFFFu, g, j);
            if (j == slot) {
                wj = wv;
                gj = gv;
            }
        }
        if (m >= E) continue;
        float dl = 0.0f;
        if (score_fn == MOE_SCORE_SOFTMAX) {
            if (renorm) {
                if (slot >= 0) dl = wj * (gj - inner);
            } else {
                const float pm = expf(__ldg(row + m) - mx) / denom;
                dl = pm * ((slot >= 0 ? gj : 0.0f) - inner);
            }
        } else if (slot >= 0) {
            if (renorm) {
                const float sg = 1.0f / (1.0f + expf(-__ldg(row + m)));
                dl = (gj - inner) / sig_sum * sg * (1.0f - sg);
            } else {
                dl = gj * wj * (1.0f - wj);  // the weight is the sigmoid itself
            }
        }
        d_logits[(size_t)t * E + m] = dl;
    }
}

// ---- fp32 layers: dgrad and wgrad on the FFMA pipes (tiles of 32 x 32, K step 32) ----
constexpr int BM = 32, BN = 32, BK = 32;

// out[row][n] = sum_k a[row][k] w[e][n][k]; block (n tile, row tile over the experts' row
// blocks). kDgradDown: SwiGLU backward epilogue and per-(row, 32-column tile) scale partials.
template <bool kDown>
__global__ void __launch_bounds__(256) simt_dgrad(DgradArgs p, int K, int N) {
    __shared__ float As[BM][BK + 1];
    __shared__ float Bs[BN][BK + 1];
    __shared__ float red[BM][17];
    __shared__ int s_e, s_m0, s_end;
    griddep_wait();
    const int tid = threadIdx.x;
    if (tid == 0) {
        int e_found = -1, m0 = 0, end = 0, mt = blockIdx.y;
        const int groups = p.offsets ? p.E : 1;
        for (int e = 0; e < groups; ++e) {
            const int lo = p.offsets ? p.offsets[e] : 0;
            const int hi = p.offsets ? p.offsets[e + 1] : p.R;
            const int tiles = (hi - lo + BM - 1) / BM;
            if (mt < tiles) {
                e_found = e;
                m0 = lo + mt * BM;
                end = hi;
                break;
            }
            mt -= tiles;
        }
        s_e = e_found;
        s_m0 = m0;
        s_end = end;
    }
    __syncthreads();
    const int e = s_e;
    if (e < 0) return;
    const int m0 = s_m0, end = s_end, n0 = blockIdx.x * BN;
    const float* A = static_cast<const float*>(p.a);
    const float* W = static_cast<const float*>(p.w) + (size_t)e * N * K;
    const int tx = tid & 15, ty = tid >> 4;
    float acc[2][2] = {};
    for (int k0 = 0; k0 < K; k0 += BK) {
        for (int i = tid; i < BM * BK; i += 256) {
            const int r = i / BK, c = i % BK, row = m0 + r, kk = k0 + c;
            As[r][c] = (row < end && kk < K) ? A[(size_t)row * K + kk] : 0.0f;
            const int n = n0 + r;
            Bs[r][c] = (n < N && kk < K) ? W[(size_t)n * K + kk] : 0.0f;
        }
        __syncthreads();
#pragma unroll 8
        for (int kk = 0; kk < BK; ++kk) {
            const float a0 = As[ty * 2][kk], a1 = As[ty * 2 + 1][kk];
            const float b0 = Bs[tx * 2][kk], b1 = Bs[tx * 2 + 1][kk];
            acc[0][0] = fmaf(a0, b0, acc[0][0]);
            acc[0][1] = fmaf(a0, b1, acc[0][1]);
            acc[1][0] = fmaf(a1, b0, acc[1][0]);
            acc[1][1] = fmaf(a1, b1, acc[1][1]);
        }
        __syncthreads();
    }
    float* out = static_cast<float*>(p.out);
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int r = ty * 2 + i, row = m0 + r;
        float ds = 0.0f;
        if (row < end) {
            if (kDown) {
                const float* ab = static_cast<const float*>(p.ab) + (size_t)row * 2 * p.I;
                float s = 1.0f;
                if (p.scale_rows) s = p.topk_weights[p.sorted_to_slot[row]];
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int col = n0 + tx * 2 + j;
                    if (col >= N) continue;
                    const float a = ab[col], b = ab[p.I + col], dh = acc[i][j];
                    const float g = s * a, u = s * b;
                    const float sig = 1.0f / (1.0f + expf(-g));
                    const float dg = dh * u * sig * (1.0f + g * (1.0f - sig));
                    const float du = dh * g * sig;
                    ds = fmaf(dg, a, fmaf(du, b, ds));
                    out[(size_t)row * 2 * p.I + col] = s * dg;
                    out[(size_t)row * 2 * p.I + p.I + col] = s * du;
                }
            } else {
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int col = n0 + tx * 2 + j;
                    if (col < N) out[(size_t)row * N + col] = acc[i][j];
                }
            }
        }
        if (kDown) red[r][tx] = ds;
    }
    if (kDown && p.scale_rows) {
        __syncthreads();
        if (tid < BM && m0 + tid < end) {
            float s = 0.0f;
            for (int x = 0; x < 16; ++x) s += red[tid][x];
            p.scale_part[(size_t)(m0 + tid) * gridDim.x + blockIdx.x] = s;
        }
    }
}

// dw[e][m][n] = sum over rows r of expert e of a[r][m] b[r][n]; grid (n tiles, m tiles, E).
__global__ void __launch_bounds__(256) simt_wgrad(WgradArgs p) {
    __shared__ float As[BK][BM + 1];
    __shared__ float Bs[BK][BN + 1];
    griddep_wait();
    const int e = blockIdx.z;
    const int lo = p.offsets ? p.offsets[e] : 0;
    const int hi = p.offsets ? p.offsets[e + 1] : p.R;
    const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN, tid = threadIdx.x;
    const int tx = tid & 15, ty = tid >> 4;
    const float* A = static_cast<const float*>(p.a);
    const float* B = static_cast<const float*>(p.b);
    float acc[2][2] = {};
    for (int r0 = lo; r0 < hi; r0 += BK) {
        for (int i = tid; i < BK * BM; i += 256) {
            const int kk = i / BM, c = i % BM, r = r0 + kk;
            As[kk][c] = (r < hi && m0 + c < p.M) ? A[(size_t)r * p.M + m0 + c] : 0.0f;
            Bs[kk][c] = (r < hi && n0 + c < p.N) ? B[(size_t)r * p.N + n0 + c] : 0.0f;
        }
        __syncthreads();
#pragma unroll 8
        for (int kk = 0; kk < BK; ++kk) {
            const float a0 = As[kk][ty * 2], a1 = As[kk][ty * 2 + 1];
            const float b0 = Bs[kk][tx * 2], b1 = Bs[kk][tx * 2 + 1];
            acc[0][0] = fmaf(a0, b0, acc[0][0]);
            acc[0][1] = fmaf(a0, b1, acc[0][1]);
            acc[1][0] = fmaf(a1, b0, acc[1][0]);
            acc[1][1] = fmaf(a1, b1, acc[1][1]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int m = m0 + ty * 2 + i, n = n0 + tx * 2 + j;
            if (m < p.M && n < p.N)
                static_cast<float*>(p.dw)[((size_t)e * p.M + m) * p.N + n] = acc[i][j];
        }
}

}  // namespace

cudaError_t launch_combine_backward(const void* dout, bool bf16, const float* y_sorted,
                                    const int32_t* slot_to_sorted, const float* weights, int T,
                                    int d, int k, void* dy_sorted, float* d_weights,
                                    cudaStream_t s) {
    const int grid = T < 65536 ? T : 65536;
    if (bf16)
        return launch_kernel(combine_backward_kernel<__nv_bfloat16>, dim3(grid), dim3(256), 0, s,
                             static_cast<const __nv_bfloat16*>(dout), y_sorted, T, d / 4, k,
                             slot_to_sorted, weights, static_cast<__nv_bfloat16*>(dy_sorted),
                             d_weights);
    return launch_kernel(combine_backward_kernel<float>, dim3(grid), dim3(256), 0, s,
                         static_cast<const float*>(dout), y_sorted, T, d / 4, k, slot_to_sorted,
                         weights, static_cast<float*>(dy_sorted), d_weights);
}

cudaError_t launch_scale_grad(const float* scale_part, int R, int n_tiles,
                              const int32_t* sorted_to_slot, float* d_weights, cudaStream_t s) {
    return launch_kernel(scale_grad_kernel, dim3((R + 255) / 256), dim3(256), 0, s, scale_part, R,
                         n_tiles, sorted_to_slot, d_weights);
}

cudaError_t launch_route_backward(const float* logits, const int32_t* ids, const float* weights,
                                  const float* d_weights, int T, int E, int k, int score_fn,
                                  bool renorm, float* d_logits, cudaStream_t s) {
    return launch_kernel(route_backward_kernel, dim3((T + 7) / 8), dim3(256), 0, s, logits, ids,
                         weights, d_weights, T, E, k, score_fn, renorm ? 1 : 0, d_logits);
}

cudaError_t launch_dgrad_f32(const DgradArgs& a, cudaStream_t s) {
    const bool down = a.kind == kDgradDown;
    const int K = down ? a.d : 2 * a.I, N = down ? a.I : a.d;
    const int groups = a.offsets ? a.E : 1;
    const dim3 grid((N + BN - 1) / BN, (a.R + BM - 1) / BM + groups);
    return launch_kernel(down ? simt_dgrad<true> : simt_dgrad<false>, grid, dim3(256), 0, s, a, K,
                         N);
}

cudaError_t launch_wgrad_f32(const WgradArgs& a, cudaStream_t s) {
    const int groups = a.offsets ? a.E : 1;
    const dim3 grid((a.N + BN - 1) / BN, (a.M + BM - 1) / BM, groups);
    return launch_kernel(simt_wgrad, grid, dim3(256), 0, s, a);
}

}  // namespace rdg
