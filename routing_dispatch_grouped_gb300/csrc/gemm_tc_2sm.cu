// Grouped expert GEMM on CTA pairs: tcgen05.mma.cta_group::2 (the 2-SM form of the sm_100-family
// tensor core instruction), bf16 in, fp32 accumulate.
//
// Same computation as gemm_tc.cu (Tensor parallelism page, "Packed strategies": packed
// [E, hidden, 2*expert_dim] gate|up weight, gate first; Expert parallelism page, "Adding an
// implementation": each expert runs on the rows routed to it), for experts with many rows. A
// cluster of two CTAs computes one 256-row x 256-column tile:
//   - CTA r holds rows [m0 + 128 r, m0 + 128 r + 128) of the token tile (A, 16 KB per k-block)
//     and half of the weight tile (B, 16 KB per k-block): for gate_up CTA 0 holds the 128 gate
//     columns and CTA 1 the 128 up columns of the same h columns; for down the two halves of the
//     256 output columns.
//   - The leader (rank 0) issues one M=256, N=256, K=16 MMA per step; each CTA's tensor memory
//     receives its own 128 rows x all 256 columns, so the epilogue of each CTA is the 1-SM one.
//   - A stage is 32 KB per CTA instead of 48 KB, so six stages fit in shared memory and the
//     loads in flight cover about half as much again of MMA time.
// gate_up tails: an expert's last tile of at most 128 rows would leave most of an M = 256 MMA
// empty. It runs instead with the operands' roles swapped (as gemm_tc_swap_pair.cu does): the
// weights are the M = 256 side (CTA r: the gate and up columns of h columns n0 + 64 r .. + 63,
// in the stage's weight half) and the tail's tokens the N side (rounded up to 16, half in each
// CTA, fetched with an 8- to 64-row box into the stage's token half); the up half of the
// accumulator reaches the gate lanes through shared memory in the epilogue.
// Synchronisation: both CTAs' copies complete on the leader's stage barrier (armed by the leader
// for the bytes of both), the leader's commits arrive on the stage and accumulator barriers of
// both CTAs, and the epilogue warps of both CTAs release an accumulator on the leader's barrier.
// Every mbarrier wait is bounded in time as in the 1-SM kernels.

#include <atomic>

#include "pair.cuh"

namespace rdg {
namespace {

constexpr int kStages = 6;
constexpr int kABytes = kTileM * kTileK * 2;     // 16 KB: this CTA's 128 rows
constexpr int kBBlockBytes = 64 * kTileK * 2;    // 8 KB
constexpr int kBBytes = 2 * kBBlockBytes;        // 16 KB: this CTA's half of the 256 columns
constexpr int kStageBytes = kABytes + kBBytes;   // 32 KB
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 512;
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr int kPairRows = 2 * kTileM;            // 256 rows per pair tile
constexpr int kBandTiles = 8;                    // row tiles per band of the tile order
constexpr int kTailRows = 128;                   // gate_up tails of at most this many rows swap
constexpr int kTailBoxes = 4;                    // token boxes of 64 >> i rows for swapped tails
constexpr int kXchFloats = 32 * 64;              // one exchange buffer: 32 tokens x 64 columns

struct PairParams {
    const int32_t* offsets;
    const int32_t* sorted_to_slot;
    const float* topk_weights;
    void* out;
    int* status;
    int R, K, N, E;
    int n_tile;    // output columns per pair tile: 128 h columns (gate_up) or 256 (down)
    int n_tiles;
    int k_blocks;
    int row_scale;
    int packed, nb, nbh, kpad;
    int band_m;    // groups of at least this many row tiles run in bands (see decode_pair)
    int swap_tails;  // gate_up: run tails of <= kTailRows rows with the weights as M
};

struct __align__(8) SmemTail {
    uint64_t full[kStages];   // used in the leader: both CTAs' copies complete here
    uint64_t empty[kStages];  // in both CTAs: released by the leader's commits
    uint64_t tfull[2];        // in both CTAs
    uint64_t tempty[2];       // used in the leader: 4 epilogue warps of each CTA
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
    int total_tiles;
    int prefix[kMaxE + 1];
    int off[kMaxE + 1];
    int mt[kMaxE];  // 256-row blocks of each expert
};

constexpr size_t kSmemBytes =
    1024 + (size_t)kStages * kStageBytes + 2 * kXchFloats * 4 + sizeof(SmemTail);

struct PairTile {
    int e, row0, row_end, n0;  // row0: this CTA's first row
    int tile_row0;             // the pair tile's first row
    int tail_n;                // > 0: a swapped tail of tail_n tokens (rounded up to 16)
};

__device__ __forceinline__ PairTile decode_pair(const SmemTail& st, int E, int n_tile,
                                                int n_tiles, int band_m, int tile,
                                                uint32_t rank, int swap_tails) {
    int lo = 0, hi = E - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (st.prefix[mid] <= tile)
            lo = mid;
        else
            hi = mid - 1;
    }
    // A group's tiles run column block by column block, each over all the group's row tiles,
    // so CTAs running together share each weight block through L2 and the weights stream once.
    // A group whose rows outnumber its weight columns and whose row panel exceeds a share of L2
    // (band_m row tiles or more: a dense shared expert) runs instead in bands of kBandTiles row
    // tiles, every column block of a band before the next band: the band's rows stay in L2
    // and the (smaller) weights stream once per band.
    const int local = tile - st.prefix[lo];
    const int m = st.mt[lo];
    const int band_w = m >= band_m ? kBandTiles : m;
    const int band = local / (band_w * n_tiles);
    const int first_m = band * band_w;
    const int bm = min(band_w, m - first_m);
    const int r = local - band * kBandTiles * n_tiles;
    const int nb = r / bm, mb = first_m + (r - (r / bm) * bm);
    PairTile t;
    t.e = lo;
    t.tile_row0 = st.off[lo] + mb * kPairRows;
    t.row0 = t.tile_row0 + (int)rank * kTileM;
    t.row_end = st.off[lo + 1];
    t.n0 = nb * n_tile;
    const int rows = t.row_end - t.tile_row0;
    t.tail_n = (swap_tails && rows <= kTailRows) ? ((rows + 15) & ~15) : 0;
    return t;
}


template <int KIND>
__global__ void __launch_bounds__(kThreads, 1)
    tc_grouped_gemm_2sm(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmW1,
                        const __grid_constant__ CUtensorMap tmX0,
                        const __grid_constant__ CUtensorMap tmX1,
                        const __grid_constant__ CUtensorMap tmX2,
                        const __grid_constant__ CUtensorMap tmX3, const PairParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    float* xch = reinterpret_cast<float*>(smem + (size_t)kStages * kStageBytes);
    SmemTail& st = *reinterpret_cast<SmemTail*>(smem + (size_t)kStages * kStageBytes +
                                                2 * kXchFloats * 4);
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
                const int m = (rows + kPairRows - 1) / kPairRows;
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
            tma_prefetch_desc(&tmA);
            tma_prefetch_desc(&tmB);
            if (p.swap_tails) {
                tma_prefetch_desc(&tmW1);
                tma_prefetch_desc(&tmX0);
                tma_prefetch_desc(&tmX1);
                tma_prefetch_desc(&tmX2);
                tma_prefetch_desc(&tmX3);
            }
            uint32_t stage = 0, phase = 0;
            bool ok = true;
            uint32_t armed_mask = 0, armed_par = 0;  // leader: stages armed, their phase
            for (int tile = pair0; tile < total && ok; tile += npairs) {
                const PairTile t =
                    decode_pair(st, E, p.n_tile, p.n_tiles, p.band_m, tile, rank, p.swap_tails);
                // a swapped tail: this CTA's half of the tail's tokens through the smallest of
                // the 64/32/16/8-row boxes that holds it (both CTAs pick the same box)
                uint32_t stage_bytes = kStageBytes;
                const CUtensorMap* tmT = &tmX0;
                int tok0 = 0;
                if (t.tail_n) {
                    const int half = t.tail_n >> 1;
                    int bi = 0;
                    while (bi < kTailBoxes - 1 && (64 >> (bi + 1)) >= half) ++bi;
                    tmT = bi == 0 ? &tmX0 : bi == 1 ? &tmX1 : bi == 2 ? &tmX2 : &tmX3;
                    stage_bytes = kBBytes + (uint32_t)(64 >> bi) * kTileK * 2;
                    tok0 = t.tile_row0 + (int)rank * half;
                }
                for (int kb = 0; kb < p.k_blocks; ++kb) {
                    if (!mbar_wait(&st.empty[stage], phase ^ 1u, abort_flag, kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    // the leader's stage barrier counts the bytes of both CTAs
                    if (leader) {
                        mbar_arrive_expect_tx(&st.full[stage], 2 * stage_bytes);
                        armed_mask |= 1u << stage;
                        armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
                    }
                    const uint32_t bar = mapa(smem_u32(&st.full[stage]), 0);
                    const uint32_t a_dst = smem_u32(smem + (size_t)stage * kStageBytes);
                    const uint32_t b_dst = a_dst + kABytes;
                    const int kc = kb * kTileK;
                    if (t.tail_n) {
                        tma_load_2d_pair(a_dst, tmT, bar, kc, tok0);
                        // the gate block and the up block of h columns n0 + 64 rank .. + 63
                        if (p.packed) {
                            const int g = t.e * p.nb + (t.n0 >> 6) + (int)rank;
                            tma_load_3d_pair(b_dst, &tmW1, bar, 0, kc, g);
                            tma_load_3d_pair(b_dst + kBBlockBytes, &tmW1, bar, 0, kc, g + p.nbh);
                        } else {
                            const int c0 = t.n0 + 64 * (int)rank;
                            tma_load_3d_pair(b_dst, &tmB, bar, c0, kc, t.e);
                            tma_load_3d_pair(b_dst + kBBlockBytes, &tmB, bar, p.N + c0, kc, t.e);
                        }
                        if (++stage == kStages) {
                            stage = 0;
                            phase ^= 1u;
                        }
                        continue;
                    }
                    tma_load_2d_pair(a_dst, &tmA, bar, kc, t.row0);
                    // this CTA's two 64-column weight blocks: gate_up = gate (rank 0) or up
                    // (rank 1) of h columns n0 .. n0+127; down = output columns
                    // n0 + 128 rank .. + 127
                    if (p.packed) {
                        const int blk = t.e * p.nb + ((KIND == kGateUp)
                                                          ? (int)rank * p.nbh + (t.n0 >> 6)
                                                          : (t.n0 >> 6) + 2 * (int)rank);
                        tma_load_3d_pair(b_dst, &tmB, bar, 0, kc, blk);
                    } else {
                        const int c0 = (KIND == kGateUp) ? (int)rank * p.N + t.n0
                                                         : t.n0 + 128 * (int)rank;
                        tma_load_3d_pair(b_dst, &tmB, bar, c0, kc, t.e);
                        tma_load_3d_pair(b_dst + kBBlockBytes, &tmB, bar, c0 + 64, kc, t.e);
                    }
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
            // M = 256 across the pair, N = 256, A K-major, B MN-major
            constexpr uint32_t idesc = idesc_bf16_f32(2 * kTileM, kTileN, true);
            uint32_t stage = 0, phase = 0, it = 0;
            bool ok = true, issued = false;
            for (int tile = pair0; tile < total && ok; tile += npairs, ++it) {
                const PairTile t =
                    decode_pair(st, E, p.n_tile, p.n_tiles, p.band_m, tile, rank, p.swap_tails);
                // a swapped tail: M = 256 weight columns, N = the tail's tokens, A MN-major,
                // B K-major (the same two shared-memory operands, roles exchanged). The choice
                // is made once per tile: the issue loop below has no branch.
                const bool tail = t.tail_n != 0;
                const uint32_t idesc_t =
                    tail ? idesc_bf16_f32_ab(2 * kTileM, t.tail_n, true, false) : idesc;
                // A and B: offset of the operand in the stage, bytes per K=16 step, LBO
                const uint32_t a_off = tail ? (uint32_t)kABytes : 0u, b_off = tail ? 0u : kABytes;
                const uint32_t a_step = tail ? 2048u : 32u, b_step = tail ? 32u : 2048u;
                const uint32_t a_lbo = tail ? (uint32_t)kBBlockBytes : 16u;
                const uint32_t b_lbo = tail ? 16u : (uint32_t)kBBlockBytes;
                const uint32_t acc = it & 1u;
                if (!mbar_wait(&st.tempty[acc], ((it >> 1) & 1u) ^ 1u, abort_flag, kWaitLimitNs)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * kTileN;
                for (int kb = 0; kb < p.k_blocks; ++kb) {
                    if (!mbar_wait(&st.full[stage], phase, abort_flag, kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t st_addr = smem_u32(smem + (size_t)stage * kStageBytes);
                    const uint64_t adesc0 = smem_desc(st_addr + a_off, a_lbo, 1024);
                    const uint64_t bdesc0 = smem_desc(st_addr + b_off, b_lbo, 1024);
#pragma unroll
                    for (int kk = 0; kk < kTileK / 16; ++kk)
                        umma_bf16_2sm(d_tmem, adesc0 + (uint64_t)((a_step >> 4) * kk),
                                      bdesc0 + (uint64_t)((b_step >> 4) * kk), idesc_t,
                                      (kb | kk) != 0 ? 1u : 0u);
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
        const int q = warp & 3;
        uint32_t it = 0, xbuf = 0;
        const uint32_t tempty_leader0 = mapa(smem_u32(&st.tempty[0]), 0);
        const uint32_t tempty_leader1 = mapa(smem_u32(&st.tempty[1]), 0);
        for (int tile = pair0; tile < total; tile += npairs, ++it) {
            const PairTile t =
                decode_pair(st, E, p.n_tile, p.n_tiles, p.band_m, tile, rank, p.swap_tails);
            const uint32_t acc = it & 1u;
            const bool ok = mbar_wait(&st.tfull[acc], (it >> 1) & 1u, abort_flag, kWaitLimitNs);
            if (!ok && lane == 0) {
                st.abort = 1;
                set_status(p.status, MOE_ERR_TIMEOUT);
            }
            // the four epilogue warps leave together, so none is left at a named barrier
            if (epilogue_any(!ok || *abort_flag != 0)) break;
            tc_fence_after();
            if (KIND == kGateUp && t.tail_n) {
                // swapped tail: lanes 0..63 hold the gate of h columns n0 + 64 rank .. + 63,
                // lanes 64..127 their up; accumulator column j is the tail's token j. The up
                // warps pass their values to the gate warps through shared memory, 32 tokens at
                // a time (double-buffered).
                const uint32_t tb = tmem_base + acc * kTileN + ((uint32_t)(q * 32) << 16);
                const bool is_gate = q < 2;
                const int hc = (q & 1) * 32 + lane;
                const int col = t.n0 + 64 * (int)rank + hc;
                const bool col_ok = col < p.N;
                const int n_valid = t.row_end - t.tile_row0;
                __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out);
#pragma unroll 1
                for (int c = 0; c * 32 < n_valid; ++c, xbuf ^= 1u) {
                    const int tok0 = t.tile_row0 + c * 32;
                    uint32_t v[32];
                    tmem_ld_32x32b_x32(tb + c * 32, v);
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
                            const float sj = __shfl_sync(0xFFFFFFFFu, my_s, j);
                            const float gj = __uint_as_float(v[j]) * sj;
                            const float uj = xb[j * 64 + hc] * sj;
                            if (tok0 + j < t.row_end && col_ok)
                                out[(size_t)(tok0 + j) * p.N + col] =
                                    __float2bfloat16_rn(silu(gj) * uj);
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(acc ? tempty_leader1 : tempty_leader0);
                continue;
            }
            const int row = t.row0 + q * 32 + lane;
            const bool row_ok = row < t.row_end;
            float s = 1.0f;
            if (p.row_scale && row_ok) s = __ldg(p.topk_weights + __ldg(p.sorted_to_slot + row));
            const uint32_t tbase = tmem_base + acc * kTileN + ((uint32_t)(q * 32) << 16);
            if (KIND == kGateUp) {
                __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out);
#pragma unroll 1
                for (int c = 0; c < 4; ++c) {
                    uint32_t g[32], u[32];
                    tmem_ld_32x32b_x32(tbase + c * 32, g);
                    tmem_ld_32x32b_x32(tbase + 128 + c * 32, u);
                    tmem_ld_wait();
                    const int col0 = t.n0 + c * 32;
                    if (row_ok) {
                        uint4* dst = reinterpret_cast<uint4*>(out + (size_t)row * p.N + col0);
#pragma unroll
                        for (int v = 0; v < 4; ++v) {
                            if (col0 + v * 8 < p.N) {
                                uint32_t w[4];
#pragma unroll
                                for (int h2 = 0; h2 < 4; ++h2) {
                                    const int i = v * 8 + h2 * 2;
                                    const float g0 = __uint_as_float(g[i]) * s;
                                    const float g1 = __uint_as_float(g[i + 1]) * s;
                                    const float u0 = __uint_as_float(u[i]) * s;
                                    const float u1 = __uint_as_float(u[i + 1]) * s;
                                    w[h2] = pack_bf16x2(silu(g0) * u0, silu(g1) * u1);
                                }
                                dst[v] = make_uint4(w[0], w[1], w[2], w[3]);
                            }
                        }
                    }
                }
            } else {
                float* out = static_cast<float*>(p.out);
#pragma unroll 1
                for (int c = 0; c < kTileN / 32; ++c) {
                    uint32_t y[32];
                    tmem_ld_32x32b_x32(tbase + c * 32, y);
                    tmem_ld_wait();
                    const int col0 = t.n0 + c * 32;
                    if (row_ok) {
                        float4* dst = reinterpret_cast<float4*>(out + (size_t)row * p.N + col0);
#pragma unroll
                        for (int v = 0; v < 8; ++v) {
                            if (col0 + v * 4 < p.N) {
                                dst[v] = make_float4(__uint_as_float(y[v * 4]) * s,
                                                     __uint_as_float(y[v * 4 + 1]) * s,
                                                     __uint_as_float(y[v * 4 + 2]) * s,
                                                     __uint_as_float(y[v * 4 + 3]) * s);
                            }
                        }
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

template <int KIND>
cudaError_t launch_pair_kind(const GroupedGemmArgs& a, cudaStream_t s) {
    {
        const cudaError_t e = ensure_max_dynamic_smem(tc_grouped_gemm_2sm<KIND>, (int)kSmemBytes);
        if (e != cudaSuccess) return e;
    }

    const int groups = a.offsets ? a.E : 1;
    CUtensorMap tmA, tmB;
    const cuuint64_t a_dims[2] = {(cuuint64_t)a.K, (cuuint64_t)a.R};
    const cuuint64_t a_str[1] = {(cuuint64_t)a.K * 2};
    const cuuint32_t a_box[2] = {kTileK, kTileM};
    const cuuint64_t bn = (KIND == kGateUp) ? 2 * (cuuint64_t)a.N : (cuuint64_t)a.N;
    const cuuint64_t b_dims[3] = {bn, (cuuint64_t)a.K, (cuuint64_t)groups};
    const cuuint64_t b_str[2] = {bn * 2, bn * 2 * (cuuint64_t)a.K};
    const cuuint32_t b_box[3] = {64, kTileK, 1};
    const PackedGeom g = packed_geom(KIND, a.K, a.N);
    const cuuint64_t pk_dims[3] = {64, (cuuint64_t)g.kpad, (cuuint64_t)groups * g.nb};
    const cuuint64_t pk_str[2] = {128, (cuuint64_t)g.kpad * 128};
    const cuuint32_t pk_box[3] = {64, kTileK, 2};
    if (!encode_tensor_map_bf16(&tmA, a.a, 2, a_dims, a_str, a_box) ||
        !(a.packed ? encode_tensor_map_bf16(&tmB, a.b, 3, pk_dims, pk_str, pk_box)
                   : encode_tensor_map_bf16(&tmB, a.b, 3, b_dims, b_str, b_box)))
        return cudaErrorInvalidValue;
    // swapped gate_up tails: single packed weight blocks and token boxes of 64/32/16/8 rows
    // (down never has them: its maps stand in)
    CUtensorMap tmW1 = tmB, tmX[kTailBoxes];
    for (int i = 0; i < kTailBoxes; ++i) tmX[i] = tmA;
    const bool tails = KIND == kGateUp;
    if (tails) {
        const cuuint32_t pk1_box[3] = {64, kTileK, 1};
        if (a.packed && !encode_tensor_map_bf16(&tmW1, a.b, 3, pk_dims, pk_str, pk1_box))
            return cudaErrorInvalidValue;
        for (int i = 0; i < kTailBoxes; ++i) {
            const cuuint32_t x_box[2] = {kTileK, (cuuint32_t)(64 >> i)};
            if (!encode_tensor_map_bf16(&tmX[i], a.a, 2, a_dims, a_str, x_box))
                return cudaErrorInvalidValue;
        }
    }

    PairParams p;
    p.offsets = a.offsets;
    p.sorted_to_slot = a.sorted_to_slot;
    p.topk_weights = a.topk_weights;
    p.out = a.out;
    p.status = a.status;
    p.R = a.R;
    p.K = a.K;
    p.N = a.N;
    p.E = groups;
    p.n_tile = (KIND == kGateUp) ? 128 : 256;
    p.n_tiles = (a.N + p.n_tile - 1) / p.n_tile;
    p.k_blocks = (a.K + kTileK - 1) / kTileK;
    p.swap_tails = tails ? 1 : 0;
    p.row_scale = (KIND == kGateUp) ? (a.scale_rows ? 1 : 0) : (a.weight_rows ? 1 : 0);
    p.packed = a.packed ? 1 : 0;
    p.nb = g.nb;
    p.nbh = g.nbh;
    p.kpad = g.kpad;
    {
        // band a group when its rows outnumber its weight columns and its row panel exceeds
        // 64 MB (half the L2)
        const long long cols = (KIND == kGateUp) ? 2ll * a.N : (long long)a.N;
        long long rows = (64ll << 20) / (2ll * a.K);
        if (rows < cols) rows = cols;
        p.band_m = (int)((rows + kPairRows - 1) / kPairRows);
    }

    // clusters that can be resident at once (SMs pair up within a GPC)
    static std::atomic<int> max_clusters[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) dev = 0;
    int mc = max_clusters[dev].load(std::memory_order_relaxed);
    if (mc == 0) {
        mc = max_pair_clusters(tc_grouped_gemm_2sm<KIND>, kThreads, kSmemBytes);
        max_clusters[dev].store(mc, std::memory_order_relaxed);
    }
    const long long pair_ub = ((long long)(a.R + kPairRows - 1) / kPairRows + groups) * p.n_tiles;
    long long clusters = mc;
    if (pair_ub < clusters) clusters = pair_ub;
    if (clusters < 1) clusters = 1;
    return launch_kernel_ex(tc_grouped_gemm_2sm<KIND>, dim3((unsigned)(2 * clusters)),
                            dim3(kThreads), kSmemBytes, s, 2, tmA, tmB, tmW1, tmX[0], tmX[1],
                            tmX[2], tmX[3], p);
}

}  // namespace

cudaError_t launch_grouped_gemm_bf16_2sm(const GroupedGemmArgs& a, cudaStream_t s) {
    return a.kind == kGateUp ? launch_pair_kind<kGateUp>(a, s) : launch_pair_kind<kDown>(a, s);
}

}  // namespace rdg
