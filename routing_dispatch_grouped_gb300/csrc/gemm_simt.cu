// fp32 grouped GEMM on the FFMA pipes, for fp32 layers.
//
// Same contract as the tensor-core path (gate_up with SwiGLU fused into the epilogue, or down
// with fp32 output), written as a plain shared-memory tiled kernel: TF32 tensor cores would not
// hold a 1e-4 relative error, and fp32 layers are small. Tile 32 x 32, K step 32, 256 threads,
// 2 x 2 outputs per thread (per accumulator). Block (n-tile, m-tile); the m-tile index runs over
// the concatenation of every expert's row blocks, looked up from the device offsets.
#include "moe_internal.cuh"

namespace rdg {
namespace {

constexpr int BM = 32, BN = 32, BK = 32;

template <bool kGU>
__global__ void __launch_bounds__(256) simt_grouped_gemm(GroupedGemmArgs p) {
    __shared__ float As[BM][BK + 1];
    __shared__ float Bs[2][BK][BN + 1];
    __shared__ int s_e, s_m0, s_end;
    griddep_wait();
    const int tid = threadIdx.x;
    if (tid == 0) {
        int e_found = -1, m0 = 0, end = 0;
        int mt = blockIdx.y;
        for (int e = 0; e < p.E; ++e) {
            const int a = p.offsets ? p.offsets[e] : 0;
            const int b = p.offsets ? p.offsets[e + 1] : p.R;
            const int tiles = (b - a + BM - 1) / BM;
            if (mt < tiles) {
                e_found = e;
                m0 = a + mt * BM;
                end = b;
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
    const int m0 = s_m0, end = s_end;
    const int n0 = blockIdx.x * BN;
    const int K = p.K, N = p.N;
    const int ldb = kGU ? 2 * N : N;
    const float* A = static_cast<const float*>(p.a);
    const float* B = static_cast<const float*>(p.b) + (size_t)e * K * ldb;
    const int tx = tid & 15, ty = tid >> 4;

    float acc[2][2][2] = {};  // [gate/up][i][j]
    for (int k0 = 0; k0 < K; k0 += BK) {
        for (int i = tid; i < BM * BK; i += 256) {
            const int r = i / BK, c = i % BK;
            const int row = m0 + r, kk = k0 + c;
            As[r][c] = (row < end && kk < K) ? A[(size_t)row * K + kk] : 0.0f;
        }
        for (int i = tid; i < BK * BN; i += 256) {
            const int r = i / BN, c = i % BN;
            const int kk = k0 + r, col = n0 + c;
            const bool ok = kk < K && col < N;
            Bs[0][r][c] = ok ? B[(size_t)kk * ldb + col] : 0.0f;
            if (kGU) Bs[1][r][c] = ok ? B[(size_t)kk * ldb + N + col] : 0.0f;
        }
        __syncthreads();
#pragma unroll 8
        for (int kk = 0; kk < BK; ++kk) {
            const float a0 = As[ty * 2][kk], a1 = As[ty * 2 + 1][kk];
#pragma unroll
            for (int g = 0; g < (kGU ? 2 : 1); ++g) {
                const float b0 = Bs[g][kk][tx * 2], b1 = Bs[g][kk][tx * 2 + 1];
                acc[g][0][0] = fmaf(a0, b0, acc[g][0][0]);
                acc[g][0][1] = fmaf(a0, b1, acc[g][0][1]);
                acc[g][1][0] = fmaf(a1, b0, acc[g][1][0]);
                acc[g][1][1] = fmaf(a1, b1, acc[g][1][1]);
            }
        }
        __syncthreads();
    }
    float* out = static_cast<float*>(p.out);
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int row = m0 + ty * 2 + i;
        if (row >= end) continue;
        float s = 1.0f;
        if ((kGU && p.scale_rows) || (!kGU && p.weight_rows))
            s = p.topk_weights[p.sorted_to_slot[row]];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int col = n0 + tx * 2 + j;
            if (col >= N) continue;
            if (kGU) {
                if (p.ab) {  // the unscaled accumulators, kept for the backward pass
                    float* ab = static_cast<float*>(p.ab) + (size_t)row * 2 * N;
                    ab[col] = acc[0][i][j];
                    ab[N + col] = acc[1][i][j];
                }
                const float g = acc[0][i][j] * s, u = acc[1][i][j] * s;
                out[(size_t)row * N + col] = g / (1.0f + expf(-g)) * u;
            } else {
                out[(size_t)row * N + col] = acc[0][i][j] * s;
            }
        }
    }
}

}  // namespace

cudaError_t launch_grouped_gemm_f32(const GroupedGemmArgs& a, cudaStream_t s) {
    const int groups = a.offsets ? a.E : 1;
    const dim3 grid((a.N + BN - 1) / BN, (a.R + BM - 1) / BM + groups);
    return launch_kernel(a.kind == kGateUp ? simt_grouped_gemm<true> : simt_grouped_gemm<false>,
                         grid, dim3(256), 0, s, a);
}

}  // namespace rdg
