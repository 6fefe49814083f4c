// Grouped expert GEMM on CTA pairs with the weights as the MMA M side:
//
//   D^T[w_cols, tokens] = W^T[w_cols, K] . X^T[K, tokens]
//
// Same computation as gemm_tc.cu (Tensor parallelism page, "Packed strategies": packed
// [E, hidden, 2*expert_dim] gate|up weight, gate first; Expert parallelism page, "Adding an
// implementation": each expert runs on the rows routed to it). It joins the two ideas of
// gemm_tc_swap.cu (tokens as the MMA N side, so a ragged expert pads at most 15 tokens) and
// gemm_tc_2sm.cu (one tcgen05.mma.cta_group::2 per K step, so each SM stages half of one
// operand). A cluster of two CTAs computes 256 weight columns x up to 256 tokens:
//   - CTA r holds 128 weight columns (A: two MN-major 64-column blocks, 16 KB per k-block): for
//     gate_up the gate columns and the up columns of h columns n0 + 64 r .. + 63, for down the
//     output columns n0 + 128 r .. + 127;
//   - and half of the tile's tokens (B, K-major): with n = the tile's token count rounded up to
//     16, CTA r holds tokens row0 + r n/2 .. row0 + (r + 1) n/2 - 1, fetched with the smallest
//     of five token boxes (128/64/32/16/8 rows) that covers n/2;
//   - the leader issues one M = 256, N = n, K = 16 MMA per step; the tensor memory of each CTA
//     receives its own 128 weight columns x all n tokens.
// Each SM then moves 32 KB of shared memory per k-block of a full tile (128 x 256 x 64 MACs)
// where the one-CTA kernels move 48 KB, and six stages fit. The epilogue is gemm_tc_swap.cu's:
// thread = weight column, loop over the tokens; in gate_up the up lanes (64..127) pass their
// values through shared memory to the gate lanes (0..63). Synchronisation is gemm_tc_2sm.cu's:
// both CTAs' copies complete on the leader's stage barrier, the leader's commits are multicast
// to both CTAs, both CTAs' epilogue warps release an accumulator on the leader's barrier, and
// every wait is bounded in time.

#include <atomic>

#include "pair.cuh"

namespace rdg {
namespace {

constexpr int kThreads = 192;
constexpr int kWBlock = 64 * kTileK * 2;          // one 64-column x 64-k MN-major block: 8 KB
constexpr int kABytes = 2 * kWBlock;              // 16 KB of weights per CTA and stage
constexpr int kXchFloats = 32 * 64;               // one exchange buffer: 32 tokens x 64 columns
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// Token tile and ring depth: HALF tokens per CTA at most (a pair tile of 2 HALF), STAGES stages
// of 16 KB of weights + HALF token rows.
template <int HALF, int STAGES>
struct PairCfg {
    static constexpr int kHalfTok = HALF;
    static constexpr int kPairTok = 2 * HALF;
    static constexpr int kStages = STAGES;
    static constexpr int kBBytes = HALF * kTileK * 2;
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr int kBoxes = HALF == 128 ? 5 : 4;   // token boxes of HALF >> i rows, >= 8
    static constexpr uint32_t kAccCols = 2 * HALF;        // one accumulator: the tile's tokens
    static constexpr uint32_t kTmemCols = 4 * HALF;       // two accumulators (a power of 2)
    static_assert(kStageBytes % 1024 == 0, "stages keep 1024-byte alignment");
    static_assert((HALF >> (kBoxes - 1)) == 8, "smallest token box: one 8-row swizzle atom");
};
// 256-token tiles, six stages. 128-token tiles with eight 24 KB stages (more weight bytes in
// flight, but the weights staged twice as often) measured slower: gpt-oss down 0.74 ms against
// 0.53, Mixtral 1.01 against 0.59.
using PairWide = PairCfg<128, 6>;

// Output columns of one pair tile: 128 h columns (gate_up) or 256 y columns (down).
template <int KIND>
struct Shape {
    static constexpr int kCols = (KIND == kGateUp) ? 128 : 256;
};

struct Params {
    const int32_t* offsets;
    const int32_t* sorted_to_slot;
    const float* topk_weights;
    void* out;
    int* status;
    int R, K, N, E;
    int n_tiles;   // weight-column blocks of Shape::kCols
    int k_blocks;  // ceil(K / 64)
    int row_scale;
    int packed;    // weights in the packed layout (pack.cu)
    int nb, nbh, kpad;
};

template <int STAGES>
struct __align__(8) SmemTail {
    uint64_t full[STAGES];    // used in the leader: both CTAs' copies complete here
    uint64_t empty[STAGES];   // in both CTAs: released by the leader's commits
    uint64_t tfull[2];        // in both CTAs
    uint64_t tempty[2];       // used in the leader: 4 epilogue warps of each CTA
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
    int total_tiles;
    int prefix[kMaxE + 1];
    int off[kMaxE + 1];
    int mt[kMaxE];  // 256-token blocks of each expert
};

template <class C>
constexpr size_t smem_bytes() {
    return 1024 + (size_t)C::kStages * C::kStageBytes + 2 * kXchFloats * 4 +
           sizeof(SmemTail<C::kStages>);
}

struct Tile {
    int e, row0, row_end, n0;
};

// Tiles run expert by expert, then weight-column block, then token block, so the pairs running
// together share each weight block through L2.
template <int KIND, int PAIR_TOK, class ST>
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
    t.row0 = st.off[lo] + mb * PAIR_TOK;
    t.row_end = st.off[lo + 1];
    t.n0 = nb * Shape<KIND>::kCols;
    return t;
}

// The MMA's N: the tile's tokens (at most a pair tile) rounded up to 16, so each CTA's half is
// a whole number of 8-row swizzle atoms.
template <class C>
__device__ __forceinline__ int tile_n(const Tile& t) {
    int n = t.row_end - t.row0;
    if (n > C::kPairTok) n = C::kPairTok;
    if (n < 1) n = 1;
    return (n + 15) & ~15;
}

// Token box i has kHalfTok >> i rows; the smallest that holds `half` rows.
template <class C>
__device__ __forceinline__ int box_index(int half) {
    int i = 0;
    while (i < C::kBoxes - 1 && (C::kHalfTok >> (i + 1)) >= half) ++i;
    return i;
}

template <int KIND, class C>
__global__ void __launch_bounds__(kThreads, 1)
    tc_grouped_gemm_swap_pair(const __grid_constant__ CUtensorMap tmW,
                              const __grid_constant__ CUtensorMap tmX0,
                              const __grid_constant__ CUtensorMap tmX1,
                              const __grid_constant__ CUtensorMap tmX2,
                              const __grid_constant__ CUtensorMap tmX3,
                              const __grid_constant__ CUtensorMap tmX4, const Params p) {
    constexpr int kStages = C::kStages;
    constexpr int kStageBytes = C::kStageBytes;
    constexpr int kHalfTok = C::kHalfTok;
    constexpr int kPairTok = C::kPairTok;
    constexpr uint32_t kAccCols = C::kAccCols;
    constexpr uint32_t kTmemCols = C::kTmemCols;
    using ST = SmemTail<kStages>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    float* xch = reinterpret_cast<float*>(smem + (size_t)kStages * kStageBytes);
    ST& st = *reinterpret_cast<ST*>(smem + (size_t)kStages * kStageBytes + 2 * kXchFloats * 4);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int E = p.E;
    const uint32_t rank = cta_rank();
    const bool leader = rank == 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&st.full[s], 1);   // the leader's producer arms it for both CTAs
            mbar_init(&st.empty[s], 1);  // one multicast commit from the leader
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&st.tfull[a], 1);
            mbar_init(&st.tempty[a], 8);  // 4 epilogue warps in each CTA
        }
        mbar_init(&st.drain, 1);
        st.abort = 0;
        fence_barrier_init();
        fence_proxy_async_smem();
    }
    if (warp == 1) tmem_alloc_2sm(&st.tmem_base, kTmemCols);
    // the peer's barriers exist before any copy, commit or arrive reaches them
    cluster_sync_all();
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
                const int m = (rows + kPairTok - 1) / kPairTok;
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
    const int pair0 = (int)cluster_idx(), npairs = (int)cluster_cnt();
    volatile int* abort_flag = &st.abort;

    if (warp == 0) {
        // ================= TMA producer (both CTAs) =================
        if (lane == 0) {
            tma_prefetch_desc(&tmW);
            tma_prefetch_desc(&tmX0);
            tma_prefetch_desc(&tmX1);
            tma_prefetch_desc(&tmX2);
            tma_prefetch_desc(&tmX3);
            tma_prefetch_desc(&tmX4);
            uint32_t stage = 0, phase = 0;
            bool ok = true;
            uint32_t armed_mask = 0, armed_par = 0;  // leader: stages armed, their phase
            // this CTA's weight blocks at (tile, kb): coordinates of their copies
            auto weight_blocks = [&](const Tile& t, int kc, auto&& op) {
                if (p.packed) {
                    if (KIND == kGateUp) {
                        // the gate block and the up block of h columns n0 + 64 rank .. + 63
                        const int b0 = t.e * p.nb + (t.n0 >> 6) + (int)rank;
                        op(0, 0, kc, b0);
                        op(1, 0, kc, b0 + p.nbh);
                    } else {
                        // output blocks n0/64 + 2 rank and the next: one two-block copy
                        op(0, 0, kc, t.e * p.nb + (t.n0 >> 6) + 2 * (int)rank);
                    }
                } else {
                    const int c0 =
                        (KIND == kGateUp) ? t.n0 + 64 * (int)rank : t.n0 + 128 * (int)rank;
                    op(0, c0, kc, t.e);
                    // gate_up: the up columns of the same h columns; down: the next 64
                    op(1, (KIND == kGateUp) ? p.N + c0 : c0 + 64, kc, t.e);
                }
            };
            for (int tile = pair0; tile < total && ok; tile += npairs) {
                const Tile t = decode<KIND, kPairTok>(st, E, tile);
                const int half = tile_n<C>(t) >> 1;
                const int bi = box_index<C>(half);
                const CUtensorMap* tmX = bi == 0   ? &tmX0
                                         : bi == 1 ? &tmX1
                                         : bi == 2 ? &tmX2
                                         : bi == 3 ? &tmX3
                                                   : &tmX4;  // (only with five boxes)
                const uint32_t stage_bytes = kABytes + (uint32_t)(kHalfTok >> bi) * kTileK * 2;
                const int tok0 = t.row0 + (int)rank * half;
                for (int kb = 0; kb < p.k_blocks; ++kb) {
                    if (!mbar_wait(&st.empty[stage], phase ^ 1u, abort_flag, kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    // the leader's stage barrier counts the bytes of both CTAs (same boxes)
                    if (leader) {
                        mbar_arrive_expect_tx(&st.full[stage], 2 * stage_bytes);
                        armed_mask |= 1u << stage;
                        armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
                    }
                    const uint32_t bar = mapa(smem_u32(&st.full[stage]), 0);
                    const uint32_t a_dst = smem_u32(smem + (size_t)stage * kStageBytes);
                    weight_blocks(t, kb * kTileK, [&](int j, int c0, int c1, int c2) {
                        tma_load_3d_pair(a_dst + j * kWBlock, &tmW, bar, c0, c1, c2);
                    });
                    tma_load_2d_pair(a_dst + kABytes, tmX, bar, kb * kTileK, tok0);
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
            // the leader's stage barriers count both CTAs' copies: let every armed stage land
            // before shared memory is released (after an abort nothing else waits for them;
            // on the normal path they have landed already)
            if (leader)
                for (int s = 0; s < kStages; ++s)
                    if ((armed_mask >> s) & 1u)
                        mbar_wait(&st.full[s], (armed_par >> s) & 1u, nullptr, kWaitLimitNs);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ================= MMA issuer (leader only) =================
        if (lane == 0 && leader) {
            uint32_t stage = 0, phase = 0, it = 0;
            bool ok = true, issued = false;
            for (int tile = pair0; tile < total && ok; tile += npairs, ++it) {
                const Tile t = decode<KIND, kPairTok>(st, E, tile);
                // M = 256 across the pair, N = the tile's tokens, A MN-major, B K-major
                const uint32_t idesc = idesc_bf16_f32_ab(2 * 128, tile_n<C>(t), true, false);
                const uint32_t acc = it & 1u;
                if (!mbar_wait(&st.tempty[acc], ((it >> 1) & 1u) ^ 1u, abort_flag, kWaitLimitNs)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * kAccCols;
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
                        // each CTA's operands at these offsets of its own shared memory:
                        // A MN-major weight blocks (64 columns, 8 KB apart), 8-row K groups 1 KB
                        // apart, +2 KB per K=16 step; B K-major tokens, +32 B per K=16 step
                        umma_bf16_2sm(d_tmem, smem_desc(a_addr + kk * 2048, kWBlock, 1024),
                                      smem_desc(b_addr + kk * 32, 16, 1024), idesc,
                                      (kb | kk) != 0 ? 1u : 0u);
                    }
                    issued = true;
                    umma_commit_2sm(&st.empty[stage]);
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (ok) umma_commit_2sm(&st.tfull[acc]);
            }
            if (!ok) {
                st.abort = 1;
                set_status(p.status, MOE_ERR_TIMEOUT);
            }
            if (*abort_flag && issued) {
                umma_commit_2sm(&st.drain);  // tracks the pair MMAs issued above
                mbar_wait(&st.drain, 0, nullptr, kWaitLimitNs);
            }
        }
        __syncwarp();
    } else {
        // ================= epilogue (warps 2..5, both CTAs) =================
        const int q = warp & 3;  // TMEM lane quarter: weight columns 32q .. 32q+31 of this CTA
        uint32_t it = 0, xbuf = 0;
        const uint32_t tempty_leader0 = mapa(smem_u32(&st.tempty[0]), 0);
        const uint32_t tempty_leader1 = mapa(smem_u32(&st.tempty[1]), 0);
        for (int tile = pair0; tile < total; tile += npairs, ++it) {
            const Tile t = decode<KIND, kPairTok>(st, E, tile);
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
            if (n_valid > kPairTok) n_valid = kPairTok;
            const int chunks = (n_valid + 31) >> 5;
            const uint32_t tbase = tmem_base + acc * kAccCols + ((uint32_t)(q * 32) << 16);
            if (KIND == kGateUp) {
                // lanes 0..63: gate of h columns n0 + 64 rank .. + 63; lanes 64..127: their up
                const bool is_gate = q < 2;
                const int hc = (q & 1) * 32 + lane;
                const int col = t.n0 + 64 * (int)rank + hc;
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
                const int col = t.n0 + 128 * (int)rank + q * 32 + lane;
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
            if (lane == 0) mbar_arrive_cluster(acc ? tempty_leader1 : tempty_leader0);
        }
    }

    // ---- teardown ----
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // nothing of the peer reaches this CTA's shared memory or tensor memory after this point
    cluster_sync_all();
    if (warp == 1) tmem_dealloc_2sm(tmem_base, kTmemCols);
}

template <int KIND, class C>
cudaError_t launch_swap_pair_kind(const GroupedGemmArgs& a, cudaStream_t s) {
    constexpr size_t kSmemBytes = smem_bytes<C>();
    constexpr int kBoxes = C::kBoxes;
    {
        const cudaError_t e =
            ensure_max_dynamic_smem(tc_grouped_gemm_swap_pair<KIND, C>, (int)kSmemBytes);
        if (e != cudaSuccess) return e;
    }

    const int groups = a.offsets ? a.E : 1;
    CUtensorMap tmW;
    const cuuint64_t wn = (KIND == kGateUp) ? 2 * (cuuint64_t)a.N : (cuuint64_t)a.N;
    const cuuint64_t w_dims[3] = {wn, (cuuint64_t)a.K, (cuuint64_t)groups};
    const cuuint64_t w_str[2] = {wn * 2, wn * 2 * (cuuint64_t)a.K};
    const cuuint32_t w_box[3] = {64, kTileK, 1};
    const PackedGeom g = packed_geom(KIND, a.K, a.N);
    const cuuint64_t pk_dims[3] = {64, (cuuint64_t)g.kpad, (cuuint64_t)groups * g.nb};
    const cuuint64_t pk_str[2] = {128, (cuuint64_t)g.kpad * 128};
    const cuuint32_t pk_box[3] = {64, kTileK, (KIND == kGateUp) ? 1u : 2u};
    if (!(a.packed ? encode_tensor_map_bf16(&tmW, a.b, 3, pk_dims, pk_str, pk_box)
                   : encode_tensor_map_bf16(&tmW, a.b, 3, w_dims, w_str, w_box)))
        return cudaErrorInvalidValue;
    CUtensorMap tmX[5];
    const cuuint64_t x_dims[2] = {(cuuint64_t)a.K, (cuuint64_t)a.R};
    const cuuint64_t x_str[1] = {(cuuint64_t)a.K * 2};
    for (int i = 0; i < kBoxes; ++i) {
        const cuuint32_t x_box[2] = {kTileK, (cuuint32_t)(C::kHalfTok >> i)};
        if (!encode_tensor_map_bf16(&tmX[i], a.a, 2, x_dims, x_str, x_box))
            return cudaErrorInvalidValue;
    }
    for (int i = kBoxes; i < 5; ++i) tmX[i] = tmX[kBoxes - 1];  // not selected

    Params p;
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

    static std::atomic<int> max_clusters[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) dev = 0;
    int mc = max_clusters[dev].load(std::memory_order_relaxed);
    if (mc == 0) {
        mc = max_pair_clusters(tc_grouped_gemm_swap_pair<KIND, C>, kThreads, kSmemBytes);
        max_clusters[dev].store(mc, std::memory_order_relaxed);
    }
    const long long tiles_ub =
        ((long long)(a.R + C::kPairTok - 1) / C::kPairTok + groups) * p.n_tiles;
    long long clusters = mc;
    if (tiles_ub < clusters) clusters = tiles_ub;
    if (clusters < 1) clusters = 1;
    return launch_kernel_ex(tc_grouped_gemm_swap_pair<KIND, C>, dim3((unsigned)(2 * clusters)),
                            dim3(kThreads), kSmemBytes, s, 2, tmW, tmX[0], tmX[1], tmX[2], tmX[3],
                            tmX[4], p);
}

}  // namespace

cudaError_t launch_grouped_gemm_bf16_swap_pair(const GroupedGemmArgs& a, cudaStream_t s) {
    return a.kind == kGateUp ? launch_swap_pair_kind<kGateUp, PairWide>(a, s)
                             : launch_swap_pair_kind<kDown, PairWide>(a, s);
}

}  // namespace rdg
