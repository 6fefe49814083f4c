// Grouped expert GEMM on the sm_103a tensor cores with the weights as the MMA M operand.
//
// Same computation as gemm_tc.cu (Tensor parallelism page, "Packed strategies": packed
// [E, hidden, 2*expert_dim] gate|up weight, gate first; Expert parallelism page, "Adding an
// implementation": each expert runs on the rows routed to it), with the roles of the operands
// swapped so that ragged expert row counts cost at most 15 padded rows instead of 127:
//
//   D^T[w_cols, tokens] = W^T[w_cols, K] . X^T[K, tokens]
//
// - A = 128 weight rows of the MMA x 64 K, read by TMA straight from the pages' [K, N]-contiguous
//   weight layout as an MN-major operand (two 64-column blocks, 128-byte swizzle). For gate_up
//   the two blocks are 64 gate columns and the 64 up columns of the same h columns; for down
//   they are 128 consecutive output columns.
// - B = up to 256 token rows x 64 K of x_sorted / h, K-major, fetched with the smallest of four
//   token boxes (256/128/64/32 rows) that covers the tile's tokens, so a tile holding the last
//   40 rows of an expert moves 4 KB of tokens per k-block instead of 32 KB.
// - MMA: M = 128, N = the tile's token count rounded up to 16 (at most 256), K = 16: one MMA
//   per K step reads 12 KB of shared memory per 128 cycles, inside its bandwidth.
// - TMEM: two tile buffers of 256 columns (512 total): the epilogue of one tile overlaps the
//   MMAs of the next.
// - Epilogue: thread = one accumulator row (weight column), loop over the tile's tokens. In
//   gate_up, TMEM lanes 64..127 (up) are read by two warps that pass their values through a
//   double-buffered 16 KB shared-memory exchange to the two warps holding lanes 0..63 (gate),
//   which compute SiLU(gate) * up. Each warp store covers 32 consecutive columns of one token
//   row (64 B for bf16 h, 128 B for fp32 y).
// Tiles are enumerated on the device from the offsets: expert, then weight-column block, then
// token block, so CTAs running together share weight blocks through L2. Waits are bounded as
// in gemm_tc.cu.

#include "moe_internal.cuh"

namespace rdg {
namespace {

constexpr int kThreads = 192;
constexpr int kWM = 128;                 // MMA M: weight rows of the accumulator
constexpr int kWBlock = 64 * kTileK * 2; // one 64-column x 64-k MN-major block: 8 KB
constexpr int kABytes = 2 * kWBlock;     // 16 KB of weights per stage
constexpr int kXchFloats = 32 * 64;      // one exchange buffer: 32 tokens x 64 columns fp32
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// Token-tile size and pipeline depth. Large batches: 256-token tiles, 4 stages of 48 KB. Small
// batches (decode): 32-token tiles, 10 stages of 20 KB, so more weight bytes are in flight and no
// 256-row token box is fetched for a handful of tokens.
template <int TOK, int STAGES>
struct Cfg {
    static constexpr int kTok = TOK;
    static constexpr int kStages = STAGES;
    static constexpr int kBBytes = TOK * kTileK * 2;
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr uint32_t kAccCols = TOK;                 // one accumulator: TOK fp32 columns
    static constexpr uint32_t kTmemCols = 2 * TOK < 32 ? 32 : 2 * TOK;  // two buffers, pow2
    static_assert(kStageBytes % 1024 == 0, "stages must keep 1024-byte alignment");
};
using CfgLarge = Cfg<256, 4>;
using CfgSmall = Cfg<32, 10>;

// Output columns covered by one tile: 64 h columns (gate_up) or 128 y columns (down).
template <int KIND>
struct Shape {
    static constexpr int kCols = (KIND == kGateUp) ? 64 : 128;
};

struct SwapParams {
    const int32_t* offsets;
    const int32_t* sorted_to_slot;
    const float* topk_weights;
    void* out;
    int* status;
    int R, K, N, E;
    int n_tiles;   // ceil(N / 128) weight-column blocks
    int k_blocks;  // ceil(K / 64)
    int row_scale;
    int packed;    // weights in the packed layout (pack.cu)
    int nb, nbh, kpad;
};

template <int STAGES>
struct __align__(8) SmemTail {
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
    int total_tiles;
    int prefix[kMaxE + 1];
    int off[kMaxE + 1];
    int mt[kMaxE];
};

template <class C>
constexpr size_t smem_bytes() {
    return 1024 + (size_t)C::kStages * C::kStageBytes + 2 * kXchFloats * 4 +
           sizeof(SmemTail<C::kStages>);
}

struct Tile {
    int e, row0, row_end, n0;
};

template <int KIND, int TOK, class ST>
__device__ __forceinline__ Tile decode(const ST& st, int E, int tile) {
    int lo = 0, hi = E - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (st.prefix[mid] <= tile)
            lo = mid;
        else
            hi = mid - 1;
    }
    const int local = tile - st.prefix[lo];
    const int m = st.mt[lo];
    const int nb = local / m, mb = local - nb * m;
    Tile t;
    t.e = lo;
    t.row0 = st.off[lo] + mb * TOK;
    t.row_end = st.off[lo + 1];
    t.n0 = nb * Shape<KIND>::kCols;
    return t;
}

__device__ __forceinline__ uint32_t idesc_swap(int n_tok) {
    // fp32 accumulator, bf16 A and B, A MN-major (bit 15), B K-major, N >> 3, M = 128 >> 4
    return (1u << 4) | (1u << 7) | (1u << 10) | (1u << 15) | ((uint32_t)(n_tok >> 3) << 17) |
           ((uint32_t)(kWM >> 4) << 24);
}


// Token box i has max(16, TOK >> i) rows; pick the smallest that holds n_tok rows.
template <int TOK>
__device__ __forceinline__ int token_box(int n_tok) {
    int i = 0;
    while (i < 3 && (TOK >> (i + 1)) >= 16 && (TOK >> (i + 1)) >= n_tok) ++i;
    return i;
}

template <int KIND, class C>
__global__ void __launch_bounds__(kThreads, 1)
    tc_grouped_gemm_swap(const __grid_constant__ CUtensorMap tmW,
                         const __grid_constant__ CUtensorMap tmX0,
                         const __grid_constant__ CUtensorMap tmX1,
                         const __grid_constant__ CUtensorMap tmX2,
                         const __grid_constant__ CUtensorMap tmX3, const SwapParams p) {
    constexpr int kStages = C::kStages;
    constexpr int kStageBytes = C::kStageBytes;
    constexpr int kTok = C::kTok;
    constexpr uint32_t kTmemCols = C::kTmemCols;
    constexpr uint32_t kAcc = C::kAccCols;
    using ST = SmemTail<kStages>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    float* xch = reinterpret_cast<float*>(smem + (size_t)kStages * kStageBytes);
    ST& st = *reinterpret_cast<ST*>(smem + (size_t)kStages * kStageBytes + 2 * kXchFloats * 4);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int E = p.E;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&st.full[s], 1);
            mbar_init(&st.empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&st.tfull[a], 1);
            mbar_init(&st.tempty[a], 4);
        }
        mbar_init(&st.drain, 1);
        st.abort = 0;
        fence_barrier_init();
        fence_proxy_async_smem();
    }
    if (warp == 1) tmem_alloc(&st.tmem_base, kTmemCols);
    // everything above is independent of the previous kernel; its outputs are read from here on
    griddep_wait();
    if (warp == 2) {
        for (int e = lane; e <= E; e += 32)
            st.off[e] = p.offsets ? __ldg(p.offsets + e) : (e == 0 ? 0 : p.R);
        __syncwarp();
        if (lane == 0) {
            int acc = 0;
            for (int e = 0; e < E; ++e) {
                int rows = st.off[e + 1] - st.off[e];
                if (rows < 0) rows = 0;
                const int m = (rows + kTok - 1) / kTok;
                st.mt[e] = m > 0 ? m : 1;
                st.prefix[e] = acc;
                acc += m * p.n_tiles;
            }
            st.prefix[E] = acc;
            st.total_tiles = acc;
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = st.tmem_base;
    const int total = st.total_tiles;
    volatile int* abort_flag = &st.abort;

    if (warp == 0) {
        // ================= TMA producer =================
        if (lane == 0) {
            tma_prefetch_desc(&tmW);
            tma_prefetch_desc(&tmX0);
            tma_prefetch_desc(&tmX1);
            tma_prefetch_desc(&tmX2);
            tma_prefetch_desc(&tmX3);
            // Small batches stream weights that nothing re-reads past the few column tiles of a
            // token box, while every weight tile re-reads the tokens: evict-first / evict-last
            // hints (measured: decode T=64 gate_up 147 -> 135 us). Large batches load without
            // hints (measured slower with them on every prefill workload).
            constexpr bool kHint = kTok <= 32;
            auto load_w = [&](uint32_t dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1,
                              int c2, uint64_t pol) {
                if (kHint)
                    tma_load_3d_hint(dst, map, bar, c0, c1, c2, pol);
                else
                    tma_load_3d(dst, map, bar, c0, c1, c2);
            };
            const uint64_t pol_w = kHint ? l2_evict_first() : 0, pol_x = kHint ? l2_evict_last() : 0;
            uint32_t stage = 0, phase = 0;
            uint32_t armed_phase[kStages];
            bool armed[kStages];
#pragma unroll
            for (int s = 0; s < kStages; ++s) {
                armed[s] = false;
                armed_phase[s] = 0;
            }
            bool ok = true;
            for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
                const Tile t = decode<KIND, kTok>(st, E, tile);
                int n_tok = t.row_end - t.row0;
                if (n_tok > kTok) n_tok = kTok;
                const int bi = token_box<kTok>((n_tok + 15) & ~15);
                const int box_rows = (kTok >> bi) < 16 ? 16 : (kTok >> bi);
                const CUtensorMap* tmX = bi == 0 ? &tmX0 : bi == 1 ? &tmX1 : bi == 2 ? &tmX2 : &tmX3;
                const uint32_t stage_bytes = kABytes + (uint32_t)box_rows * kTileK * 2;
                for (int kb = 0; kb < p.k_blocks; ++kb) {
                    if (!mbar_wait(&st.empty[stage], phase ^ 1u, abort_flag, kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&st.full[stage], stage_bytes);
                    armed[stage] = true;
                    armed_phase[stage] = phase;
                    const uint32_t a_dst = smem_u32(smem + (size_t)stage * kStageBytes);
                    const int kc = kb * kTileK;
                    if (p.packed) {
                        // packed blocks of one expert are adjacent along the third dimension:
                        // down reads blocks n0/64 and n0/64 + 1 in one copy; gate_up reads the
                        // gate block and the up block of the same columns (two copies)
                        const int b0 = t.e * p.nb + (t.n0 >> 6);
                        load_w(a_dst, &tmW, &st.full[stage], 0, kc, b0, pol_w);
                        if (KIND == kGateUp)
                            load_w(a_dst + kWBlock, &tmW, &st.full[stage], 0, kc, b0 + p.nbh,
                                   pol_w);
                    } else {
                        load_w(a_dst, &tmW, &st.full[stage], t.n0, kc, t.e, pol_w);
                        // gate_up: the up columns of the same h columns; down: the next 64
                        load_w(a_dst + kWBlock, &tmW, &st.full[stage],
                               (KIND == kGateUp) ? p.N + t.n0 : t.n0 + 64, kc, t.e, pol_w);
                    }
                    if (kHint)
                        tma_load_2d_hint(a_dst + kABytes, tmX, &st.full[stage], kc, t.row0,
                                         pol_x);
                    else
                        tma_load_2d(a_dst + kABytes, tmX, &st.full[stage], kc, t.row0);
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {
                st.abort = 1;
                set_status(p.status, MOE_ERR_TIMEOUT);
            }
            // let every copy this thread started land before shared memory is released (after
            // an abort elsewhere nothing else waits for them)
            for (int s = 0; s < kStages; ++s)
                if (armed[s]) mbar_wait(&st.full[s], armed_phase[s], nullptr, kWaitLimitNs);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ================= MMA issuer =================
        if (lane == 0) {
            uint32_t stage = 0, phase = 0, it = 0;
            bool ok = true, issued = false;
            for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x, ++it) {
                const Tile t = decode<KIND, kTok>(st, E, tile);
                int n_tok = t.row_end - t.row0;
                if (n_tok > kTok) n_tok = kTok;
                n_tok = (n_tok + 15) & ~15;
                const uint32_t idesc = idesc_swap(n_tok);
                const uint32_t acc = it & 1u;
                if (!mbar_wait(&st.tempty[acc], ((it >> 1) & 1u) ^ 1u, abort_flag, kWaitLimitNs)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d0 = tmem_base + acc * kAcc;
                for (int kb = 0; kb < p.k_blocks; ++kb) {
                    if (!mbar_wait(&st.full[stage], phase, abort_flag, kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(smem + (size_t)stage * kStageBytes);
                    const uint32_t b_addr = a_addr + kABytes;
#pragma unroll
                    for (int kk = 0; kk < kTileK / 16; ++kk) {
                        // A: MN-major weight blocks (64 columns, 8 KB apart), 8-row K groups 1 KB
                        //    apart, +2 KB per K=16 step. B: K-major tokens, +32 B per K=16 step.
                        umma_bf16(d0, smem_desc(a_addr + kk * 2048, kWBlock, 1024),
                                  smem_desc(b_addr + kk * 32, 16, 1024), idesc,
                                  (kb | kk) != 0 ? 1u : 0u);
                    }
                    issued = true;
                    umma_commit(&st.empty[stage]);
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (ok) umma_commit(&st.tfull[acc]);
            }
            if (!ok) {
                st.abort = 1;
                set_status(p.status, MOE_ERR_TIMEOUT);
            }
            if (*abort_flag && issued) {
                umma_commit(&st.drain);
                mbar_wait(&st.drain, 0, nullptr, kWaitLimitNs);
            }
        }
        __syncwarp();
    } else {
        // ================= epilogue (warps 2..5) =================
        const int q = warp & 3;  // TMEM lane quarter: rows 32q .. 32q+31 of the accumulator
        uint32_t it = 0, xbuf = 0;
        for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++it) {
            const Tile t = decode<KIND, kTok>(st, E, tile);
            const uint32_t acc = it & 1u;
            const bool ok = mbar_wait(&st.tfull[acc], (it >> 1) & 1u, abort_flag, kWaitLimitNs);
            if (!ok && lane == 0) {
                st.abort = 1;
                set_status(p.status, MOE_ERR_TIMEOUT);
            }
            // the four epilogue warps leave together, so none is left at a named barrier
            if (epilogue_any(!ok || *abort_flag != 0)) break;
            tc_fence_after();
            int n_valid = t.row_end - t.row0;
            if (n_valid > kTok) n_valid = kTok;
            const int chunks = (n_valid + 31) >> 5;
            const uint32_t tbase = tmem_base + acc * kAcc + ((uint32_t)(q * 32) << 16);
            if (KIND == kGateUp) {
                // lanes 0..63: gate of h columns n0 .. n0+63; lanes 64..127: up of the same
                const bool is_gate = q < 2;
                const int hc = (q & 1) * 32 + lane;  // h column within the tile
                const int col = t.n0 + hc;
                const bool col_ok = col < p.N;
                __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out);
#pragma unroll 1
                for (int c = 0; c < chunks; ++c, xbuf ^= 1u) {
                    const int tok0 = t.row0 + c * 32;
                    uint32_t v[32];
                    tmem_ld_32x32b_x32(tbase + c * 32, v);
                    tmem_ld_wait();
                    float* xb = xch + xbuf * kXchFloats;
                    if (!is_gate) {
#pragma unroll
                        for (int j = 0; j < 32; ++j) xb[j * 64 + hc] = __uint_as_float(v[j]);
                    }
                    float my_s = 1.0f;
                    if (p.row_scale && tok0 + lane < t.row_end)
                        my_s = __ldg(p.topk_weights + __ldg(p.sorted_to_slot + tok0 + lane));
                    epilogue_sync();
                    if (is_gate) {
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            const float s = __shfl_sync(0xFFFFFFFFu, my_s, j);
                            const float g = __uint_as_float(v[j]) * s;
                            const float u = xb[j * 64 + hc] * s;
                            if (tok0 + j < t.row_end && col_ok)
                                out[(size_t)(tok0 + j) * p.N + col] =
                                    __float2bfloat16_rn(silu(g) * u);
                        }
                    }
                }
            } else {
                const int col = t.n0 + q * 32 + lane;
                const bool col_ok = col < p.N;
                float* out = static_cast<float*>(p.out);
#pragma unroll 1
                for (int c = 0; c < chunks; ++c) {
                    const int tok0 = t.row0 + c * 32;
                    float my_s = 1.0f;
                    if (p.row_scale && tok0 + lane < t.row_end)
                        my_s = __ldg(p.topk_weights + __ldg(p.sorted_to_slot + tok0 + lane));
                    uint32_t y[32];
                    tmem_ld_32x32b_x32(tbase + c * 32, y);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const float s = __shfl_sync(0xFFFFFFFFu, my_s, j);
                        if (tok0 + j < t.row_end && col_ok)
                            out[(size_t)(tok0 + j) * p.N + col] = __uint_as_float(y[j]) * s;
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&st.tempty[acc]);
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, kTmemCols);
}

template <int KIND, class C>
cudaError_t launch_swap_kind(const GroupedGemmArgs& a, cudaStream_t s) {
    constexpr int kTok = C::kTok;
    constexpr size_t kSmemBytes = smem_bytes<C>();
    {
        const cudaError_t e =
            ensure_max_dynamic_smem(tc_grouped_gemm_swap<KIND, C>, (int)kSmemBytes);
        if (e != cudaSuccess) return e;
    }

    const int groups = a.offsets ? a.E : 1;
    CUtensorMap tmW, tmX;
    const cuuint64_t wn = (KIND == kGateUp) ? 2 * (cuuint64_t)a.N : (cuuint64_t)a.N;
    const cuuint64_t w_dims[3] = {wn, (cuuint64_t)a.K, (cuuint64_t)groups};
    const cuuint64_t w_str[2] = {wn * 2, wn * 2 * (cuuint64_t)a.K};
    const cuuint32_t w_box[3] = {64, kTileK, 1};
    const cuuint64_t x_dims[2] = {(cuuint64_t)a.K, (cuuint64_t)a.R};
    const cuuint64_t x_str[1] = {(cuuint64_t)a.K * 2};
    CUtensorMap tmX1, tmX2, tmX3;
    const PackedGeom g = packed_geom(KIND, a.K, a.N);
    const cuuint64_t pk_dims[3] = {64, (cuuint64_t)g.kpad, (cuuint64_t)groups * g.nb};
    const cuuint64_t pk_str[2] = {128, (cuuint64_t)g.kpad * 128};
    const cuuint32_t pk_box[3] = {64, kTileK, (KIND == kGateUp) ? 1u : 2u};
    if (!(a.packed ? encode_tensor_map_bf16(&tmW, a.b, 3, pk_dims, pk_str, pk_box)
                   : encode_tensor_map_bf16(&tmW, a.b, 3, w_dims, w_str, w_box)))
        return cudaErrorInvalidValue;
    // token boxes of max(16, kTok >> i) rows (token_box picks one per tile)
    CUtensorMap* xm[4] = {&tmX, &tmX1, &tmX2, &tmX3};
    for (int i = 0; i < 4; ++i) {
        const int rows = (kTok >> i) < 16 ? 16 : (kTok >> i);
        const cuuint32_t x_box[2] = {kTileK, (cuuint32_t)rows};
        if (!encode_tensor_map_bf16(xm[i], a.a, 2, x_dims, x_str, x_box))
            return cudaErrorInvalidValue;
    }

    SwapParams p;
    p.offsets = a.offsets;
    p.sorted_to_slot = a.sorted_to_slot;
    p.topk_weights = a.topk_weights;
    p.out = a.out;
    p.status = a.status;
    p.R = a.R;
    p.K = a.K;
    p.N = a.N;
    p.E = groups;
    p.n_tiles = (a.N + Shape<KIND>::kCols - 1) / Shape<KIND>::kCols;
    p.k_blocks = (a.K + kTileK - 1) / kTileK;
    p.row_scale = (KIND == kGateUp) ? (a.scale_rows ? 1 : 0) : (a.weight_rows ? 1 : 0);
    p.packed = a.packed ? 1 : 0;
    p.nb = g.nb;
    p.nbh = g.nbh;
    p.kpad = g.kpad;

    const long long m_ub = (long long)(a.R + kTok - 1) / kTok + groups;
    const long long tiles_ub = m_ub * p.n_tiles;
    int grid = device_sm_count();
    if (tiles_ub < grid) grid = (int)tiles_ub;
    if (grid < 1) grid = 1;
    return launch_kernel(tc_grouped_gemm_swap<KIND, C>, dim3(grid), dim3(kThreads), kSmemBytes, s,
                         tmW, tmX, tmX1, tmX2, tmX3, p);
}

}  // namespace

cudaError_t launch_grouped_gemm_bf16_swap(const GroupedGemmArgs& a, cudaStream_t s) {
    if (a.R <= kSmallBatchRows)
        return a.kind == kGateUp ? launch_swap_kind<kGateUp, CfgSmall>(a, s)
                                 : launch_swap_kind<kDown, CfgSmall>(a, s);
    return a.kind == kGateUp ? launch_swap_kind<kGateUp, CfgLarge>(a, s)
                             : launch_swap_kind<kDown, CfgLarge>(a, s);
}

// Large batches: gate_up runs on the 128-row kernel, where each epilogue thread holds gate and
// up of its h columns (this kernel's gate_up passes the up half between warps and leaves the
// SiLU work to two of the four epilogue warps, which measured slower on every prefill
// workload). Small batches (at most kSmallBatchRows routed rows): both run here with 32-token
// tiles, which stream weights without fetching 128- or 256-row token tiles.
// CTA pairs take the rest of the large batches:
//   - gate_up: 256-row tiles (gemm_tc_2sm.cu), an expert's tail of at most 128 rows run with
//     the weights as M; measured in one process against the 128-row kernel: Mixtral 1.15 ms vs
//     1.18, Scout routed 1.65 vs 1.66-1.70, gpt-oss 0.961 vs 0.970 (before the swapped tails
//     the 256-row padding made gpt-oss slower, 1.03 vs 0.98);
//   - down of a single dense group: 256-row tiles (gemm_tc_2sm.cu), faster than the weights-
//     as-M pair on Scout's shared expert (0.76-0.81 ms against 0.93);
//   - routed down: weights as the M = 256 side, tokens as N padded to 16 (gemm_tc_swap_pair.cu),
//     measured faster than both 256-row tiles and this kernel on gpt-oss (0.52-0.53 ms against
//     0.58 and 0.56), Mixtral (0.59-0.60 against 0.61-0.62 and 0.65) and Scout's routed
//     experts (0.82-0.84 against 0.85-0.87 and 1.01).
// Small batches (at most kSmallBatchRows routed rows) run here.
GemmPick pick_grouped_gemm_bf16(GemmKind kind, int R, int groups, bool special_epilogue) {
    // training (saved accumulators) and MX layers (h rounded to MXFP8) use the 128-row kernel
    if (kind == kGateUp && special_epilogue) return kPickRows;
    if (R > kSmallBatchRows) {
        if (groups == 1) return kPick2sm;
        return kind == kDown ? kPickSwapPair : kPick2sm;
    }
    return kPickSwap;
}

cudaError_t launch_grouped_gemm_bf16(const GroupedGemmArgs& a, cudaStream_t s) {
    switch (pick_grouped_gemm_bf16(a.kind, a.R, a.offsets ? a.E : 1, a.ab || a.mx_h)) {
        case kPickRows: return launch_grouped_gemm_bf16_rows(a, s);
        case kPick2sm: return launch_grouped_gemm_bf16_2sm(a, s);
        case kPickSwapPair: return launch_grouped_gemm_bf16_swap_pair(a, s);
        default: return launch_grouped_gemm_bf16_swap(a, s);
    }
}

}  // namespace rdg
