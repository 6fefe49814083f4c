// Backward grouped GEMMs of the expert layer on the sm_103a tensor cores (tcgen05 + TMEM + TMA),
// bf16 in, fp32 accumulate.
//
// The routing weights multiply the expert outputs (Expert parallelism page, introduction and
// "Token dispatch"), so a training step differentiates the layer: the gradient of each expert's
// SwiGLU feed-forward (Tensor parallelism page, "Packed strategies": gate_up [E, d, 2I] gate
// first, down [E, I, d]) on the rows routed to it. Two kernels, both persistent, one CTA per SM,
// with the forward GEMM's structure (TMA producer warp, one MMA-issuing warp, four epilogue
// warps over a double-buffered 2 x 256-column TMEM accumulator, 4-stage shared-memory ring):
//
//   dgrad (rows of an expert times the transposed expert weight; both operands K-major):
//     down:    dh = dy_sorted . W_down[e]^T, tiles of 128 rows x 256 h columns; the epilogue is
//              the SwiGLU backward. With a = x W_gate, b = x W_up (the saved accumulators), the
//              router score s (1 unless it scales the input), g = s a, u = s b and
//              sigma = 1 / (1 + exp(-g)):
//                dg = dh u sigma (1 + g (1 - sigma)),  du = dh g sigma,
//                d_ab = [s dg | s du] (rounded to bf16),  d_s += dg a + du b (per tile).
//     gate_up: dx_sorted = d_ab . W_gate_up[e]^T (K = 2I), fp32 output.
//   wgrad (both operands MN-major, K = the expert's rows):
//     dW[e] = a[rows of e]^T . b[rows of e], tiles of 128 x 256 of dW[e], fp32 output. The last
//     K block of an expert reaches into the next expert's rows; the MMA warp zeroes those rows
//     of both operand tiles in shared memory (then fences the generic-proxy stores against the
//     tensor core's reads) before it issues the block's MMAs.
//
// Every mbarrier wait is bounded in time; on expiry the kernel records MOE_ERR_TIMEOUT, drains
// its own copies and MMAs, frees TMEM and returns.

#include "moe_internal.cuh"

namespace rdg {
namespace {

constexpr int kMaxStages = 4;
constexpr int kABytes = 128 * 64 * 2;              // 16 KB: 128 rows x 64 K (dgrad) or 2 x 8 KB
constexpr int kBBytes = 256 * 64 * 2;              // 32 KB: 256 rows x 64 K or 4 x 8 KB
constexpr int kStageBytes = kABytes + kBBytes;     // 48 KB
constexpr int kBlk = 64 * 64 * 2;                  // 8 KB: one 64 x 64 MN-major block
constexpr int kThreads = 192;  // warps: 0 TMA, 1 MMA (+ tail zeroing), 2..5 epilogue
constexpr uint32_t kTmemCols = 512;
constexpr uint64_t kWaitLimitNs = 2000000000ull;

enum Mode { kModeDgradDown = 0, kModeDgradGateUp = 1, kModeWgrad = 2 };

struct BwdParams {
    const int32_t* offsets;
    const int32_t* sorted_to_slot;
    const float* topk_weights;
    const __nv_bfloat16* ab;   // dgrad down: saved accumulators [R, 2I]
    void* out;                 // d_ab (bf16) / dx_sorted (fp32) / dW (fp32 or bf16)
    float* scale_part;         // dgrad down with row scale: [R, n_tiles]
    int* status;
    int R, E;
    int M, N;                  // wgrad: dW[e] is M x N; dgrad: N output columns
    int I;                     // dgrad down: h width (N = I); gate_up: I for the K split
    int n_tiles, m_tiles;      // m_tiles: wgrad only
    int k_blocks;              // dgrad: K blocks of 64
    int row_scale;
    int packed;
    int nb_w, nbh;             // packed geometry of the weight
    int ldab;                  // 2I
    int dw_bf16;               // wgrad: dW rounded to bf16 (else fp32)
};

struct __align__(8) SmemTail {
    uint64_t full[kMaxStages];
    uint64_t empty[kMaxStages];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
    int total_tiles;
    int prefix[kMaxE + 1];  // dgrad: first tile of each expert
    int off[kMaxE + 1];     // row offsets
    int mt[kMaxE];          // dgrad: M blocks of each expert
    int order[kMaxE];       // wgrad: experts by descending row count
};

// Shared memory of each mode (after 1024-byte alignment):
//   dgrad: 4 stages | tail | (gate_up) a per-warp 32 x 32 fp32 transpose buffer, rows padded to
//          33 floats (no bank conflicts either way), so each store instruction writes 128
//          contiguous bytes of one row of dx_sorted;
//   wgrad: 3 stages | per-warp double-buffered 32 x 32 fp32 staging tiles in the 128-byte
//          swizzled layout of a TMA store (the tensor map clips the dW block's edges) | tail.
// The wgrad epilogue moves 128 KB per tile against a K loop of a few blocks: full-line TMA
// stores keep it off the shared-memory and L2 request paths that per-row stores saturate.
constexpr int kXposeFloats = 4 * 32 * 33;
constexpr int kStagingBytes = 4 * 2 * 32 * 32 * 4;  // 32 KB
template <int MODE>
struct Layout {
    static constexpr int stages = MODE == kModeWgrad ? 3 : 4;
    static constexpr size_t staging = (size_t)stages * kStageBytes;  // 1024-byte aligned
    static constexpr size_t tail = staging + (MODE == kModeWgrad ? kStagingBytes : 0);
    static constexpr size_t xpose = tail + sizeof(SmemTail);
    static constexpr size_t bytes =
        1024 + xpose + (MODE == kModeDgradGateUp ? (size_t)kXposeFloats * 4 : 0);
    static_assert(bytes <= 232448, "exceeds the 227 KB of shared memory a block may use");
};

struct Tile {
    int e;        // expert
    int row0;     // dgrad: first row; wgrad: first row of the expert
    int row_end;  // end of the expert's rows
    int m0, n0;   // wgrad: dW block; dgrad: n0 only
    int kbs;      // K blocks of this tile
};

template <int MODE>
__device__ __forceinline__ Tile decode_tile(const SmemTail& st, const BwdParams& p, int tile) {
    Tile t;
    if (MODE == kModeWgrad) {
        const int per = p.m_tiles * p.n_tiles;
        const int e = st.order[tile / per];
        const int local = tile - (tile / per) * per;
        // keep the smaller operand resident in L2: the M blocks of one N block run together
        // when the b block (N wide) is the larger stream, else the N blocks of one M block
        int mb, nb;
        if (p.N >= p.M) {
            nb = local / p.m_tiles;
            mb = local - nb * p.m_tiles;
        } else {
            mb = local / p.n_tiles;
            nb = local - mb * p.n_tiles;
        }
        t.e = e;
        t.row0 = st.off[e];
        t.row_end = st.off[e + 1];
        t.m0 = mb * 128;
        t.n0 = nb * 256;
        t.kbs = (t.row_end - t.row0 + 63) / 64;
    } else {
        int lo = 0, hi = p.E - 1;  // largest e with prefix[e] <= tile
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (st.prefix[mid] <= tile)
                lo = mid;
            else
                hi = mid - 1;
        }
        const int e = lo;
        const int local = tile - st.prefix[e];
        const int m = st.mt[e];
        const int nb = local / m, mb = local - nb * m;  // row blocks of one N block together
        t.e = e;
        t.row0 = st.off[e] + mb * 128;
        t.row_end = st.off[e + 1];
        t.m0 = 0;
        t.n0 = nb * 256;
        t.kbs = p.k_blocks;
    }
    return t;
}

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    tc_bwd_gemm(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmO, const BwdParams p) {
    constexpr int kStages = Layout<MODE>::stages;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    SmemTail& st = *reinterpret_cast<SmemTail*>(smem + Layout<MODE>::tail);
    float* xpose = reinterpret_cast<float*>(smem + Layout<MODE>::xpose);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int E = p.E;

    // ---- set-up: barriers, TMEM, tile table ----
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
    griddep_wait();
    if (warp == 2) {
        for (int e = lane; e <= E; e += 32)
            st.off[e] = p.offsets ? __ldg(p.offsets + e) : (e == 0 ? 0 : p.R);
        __syncwarp();
        if (MODE == kModeWgrad) {
            // experts by descending row count (ties: lower index first), so the longest K
            // loops are handed out first
            for (int e = lane; e < E; e += 32) {
                const int c = st.off[e + 1] - st.off[e];
                int rank = 0;
                for (int f = 0; f < E; ++f) {
                    const int cf = st.off[f + 1] - st.off[f];
                    rank += (cf > c || (cf == c && f < e)) ? 1 : 0;
                }
                st.order[rank] = e;
            }
            if (lane == 0) st.total_tiles = E * p.m_tiles * p.n_tiles;
        } else if (lane == 0) {
            int acc = 0;
            for (int e = 0; e < E; ++e) {
                int rows = st.off[e + 1] - st.off[e];
                if (rows < 0) rows = 0;
                const int m = (rows + 127) / 128;
                st.mt[e] = m > 0 ? m : 1;  // experts without rows own no tiles
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
            tma_prefetch_desc(&tmA);
            tma_prefetch_desc(&tmB);
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
                const Tile t = decode_tile<MODE>(st, p, tile);
                for (int kb = 0; kb < t.kbs; ++kb) {
                    if (!mbar_wait(&st.empty[stage], phase ^ 1u, abort_flag, kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&st.full[stage], kStageBytes);
                    armed[stage] = true;
                    armed_phase[stage] = phase;
                    const uint32_t a_dst = smem_u32(smem + (size_t)stage * kStageBytes);
                    const uint32_t b_dst = a_dst + kABytes;
                    if (MODE == kModeWgrad) {
                        const int r0 = t.row0 + 64 * kb;
                        tma_load_2d(a_dst, &tmA, &st.full[stage], t.m0, r0);
                        tma_load_2d(a_dst + kBlk, &tmA, &st.full[stage], t.m0 + 64, r0);
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            tma_load_2d(b_dst + j * kBlk, &tmB, &st.full[stage], t.n0 + 64 * j,
                                        r0);
                    } else {
                        // A: the tile's rows, K columns of this block (the gate_up K runs over
                        // the gate half, then the up half, when the weight is packed: each
                        // packed block holds one half's columns)
                        int acol = 64 * kb;
                        if (MODE == kModeDgradGateUp && p.packed && kb >= p.nbh)
                            acol = p.I + 64 * (kb - p.nbh);
                        tma_load_2d(a_dst, &tmA, &st.full[stage], acol, t.row0);
                        if (p.packed)
                            tma_load_3d(b_dst, &tmB, &st.full[stage], 0, t.n0,
                                        t.e * p.nb_w + kb);
                        else
                            tma_load_3d(b_dst, &tmB, &st.full[stage], 64 * kb, t.n0, t.e);
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
            // let every copy this thread started land before shared memory is released (after
            // an abort elsewhere nothing else waits for them)
            for (int s = 0; s < kStages; ++s)
                if (armed[s]) mbar_wait(&st.full[s], armed_phase[s], nullptr, kWaitLimitNs);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ================= MMA issuer (lane 0), tail zeroing (whole warp) =================
        constexpr bool kMN = MODE == kModeWgrad;
        constexpr uint32_t idesc = idesc_bf16_f32_ab(128, 256, kMN, kMN);
        uint32_t stage = 0, phase = 0, it = 0;
        bool ok = true, issued = false;
        if (MODE != kModeWgrad) {
            // dgrad: nothing to fix up in shared memory, so one thread waits and issues (a
            // warp-wide wait and shuffle per stage only lengthen the issue path)
            if (lane == 0) {
                for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x, ++it) {
                    const Tile t = decode_tile<MODE>(st, p, tile);
                    const uint32_t acc = it & 1u;
                    if (!mbar_wait(&st.tempty[acc], ((it >> 1) & 1u) ^ 1u, abort_flag,
                                   kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d_tmem = tmem_base + acc * 256;
                    for (int kb = 0; kb < t.kbs; ++kb) {
                        if (!mbar_wait(&st.full[stage], phase, abort_flag, kWaitLimitNs)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t a_addr = smem_u32(smem + (size_t)stage * kStageBytes);
                        const uint32_t b_addr = a_addr + kABytes;
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            // K-major: 128-byte rows, 8-row groups 1 KB apart, +32 B per step
                            umma_bf16(d_tmem, smem_desc(a_addr + kk * 32, 16, 1024),
                                      smem_desc(b_addr + kk * 32, 16, 1024), idesc,
                                      (kb | kk) != 0 ? 1u : 0u);
                        issued = true;
                        umma_commit(&st.empty[stage]);
                        if (++stage == kStages) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                    if (ok) umma_commit(&st.tfull[acc]);
                }
            }
        }
        for (int tile = blockIdx.x; MODE == kModeWgrad && tile < total && ok;
             tile += gridDim.x, ++it) {
            const Tile t = decode_tile<MODE>(st, p, tile);
            const uint32_t acc = it & 1u;
            bool w_ok = true;
            if (lane == 0)
                w_ok = mbar_wait(&st.tempty[acc], ((it >> 1) & 1u) ^ 1u, abort_flag,
                                 kWaitLimitNs);
            if (!__shfl_sync(0xFFFFFFFFu, w_ok ? 1 : 0, 0)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + acc * 256;
            for (int kb = 0; kb < t.kbs; ++kb) {
                // every lane waits: the tail rows below are overwritten after the copy landed
                w_ok = mbar_wait(&st.full[stage], phase, abort_flag, kWaitLimitNs);
                if (!__shfl_sync(0xFFFFFFFFu, w_ok ? 1 : 0, 0)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint8_t* sa = smem + (size_t)stage * kStageBytes;
                if (MODE == kModeWgrad) {
                    const int valid = t.row_end - (t.row0 + 64 * kb);  // K rows of this expert
                    if (valid < 64) {
                        // rows [valid, 64) belong to the next expert (or lie past R): zero them
                        // in the six 8 KB blocks (2 of a, 4 of b); a block row is 128 bytes
                        for (int i = valid * 8 + lane; i < 64 * 8; i += 32) {
                            // 16-byte chunk i & 7 of block row i >> 3, in all six blocks
                            uint8_t* row = sa + (i >> 3) * 128 + (i & 7) * 16;
#pragma unroll
                            for (int blk = 0; blk < 6; ++blk)
                                *reinterpret_cast<uint4*>(row + blk * kBlk) =
                                    make_uint4(0u, 0u, 0u, 0u);
                        }
                        fence_proxy_async_smem();  // generic stores -> tensor-core reads
                        __syncwarp();
                    }
                }
                if (lane == 0) {
                    const uint32_t a_addr = smem_u32(sa);
                    const uint32_t b_addr = a_addr + kABytes;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        uint64_t adesc, bdesc;
                        if (kMN) {
                            // MN-major: 64-element blocks 8 KB apart (LBO), 8-row groups 1 KB
                            // apart (SBO), +2 KB per K=16 step
                            adesc = smem_desc(a_addr + kk * 2048, kBlk, 1024);
                            bdesc = smem_desc(b_addr + kk * 2048, kBlk, 1024);
                        } else {
                            // K-major: 128-byte rows, 8-row groups 1 KB apart, +32 bytes per step
                            adesc = smem_desc(a_addr + kk * 32, 16, 1024);
                            bdesc = smem_desc(b_addr + kk * 32, 16, 1024);
                        }
                        umma_bf16(d_tmem, adesc, bdesc, idesc, (kb | kk) != 0 ? 1u : 0u);
                    }
                    issued = true;
                    umma_commit(&st.empty[stage]);
                }
                __syncwarp();
                if (++stage == kStages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            // a tile without K blocks (an expert with no rows) is committed without MMAs: its
            // epilogue writes zeros and reads no accumulator
            if (ok && lane == 0) umma_commit(&st.tfull[acc]);
            __syncwarp();
        }
        if (lane == 0) {
            if (!ok) {
                st.abort = 1;
                set_status(p.status, MOE_ERR_TIMEOUT);
            }
            if (*abort_flag && issued) {
                umma_commit(&st.drain);  // completes once every MMA issued above is done
                mbar_wait(&st.drain, 0, nullptr, kWaitLimitNs);
            }
        }
        __syncwarp();
    } else {
        // ================= epilogue (warps 2..5) =================
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        uint32_t it = 0;
        uint32_t n_store = 0;    // wgrad: TMA stores this warp issued
        for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++it) {
            const Tile t = decode_tile<MODE>(st, p, tile);
            const uint32_t acc = it & 1u;
            if (MODE == kModeDgradDown) {
                // the saved a, b of this thread's row do not depend on the accumulator: ask L2
                // for them while the tile's MMAs run (five 64-column steps cover the 256
                // columns' lines of each half)
                const int row = t.row0 + q * 32 + lane;
                if (row < t.row_end) {
                    const __nv_bfloat16* ra = p.ab + (size_t)row * p.ldab;
#pragma unroll
                    for (int k = 0; k < 5; ++k) {
                        const int col = min(t.n0 + 64 * k, t.n0 + 255);
                        if (col < p.I) {
                            asm volatile("prefetch.global.L2 [%0];" ::"l"(ra + col));
                            asm volatile("prefetch.global.L2 [%0];" ::"l"(ra + p.I + col));
                        }
                    }
                }
            }
            if (!mbar_wait(&st.tfull[acc], (it >> 1) & 1u, abort_flag, kWaitLimitNs)) {
                if (lane == 0) {
                    st.abort = 1;
                    set_status(p.status, MOE_ERR_TIMEOUT);
                }
                break;
            }
            tc_fence_after();
            const uint32_t tbase = tmem_base + acc * 256 + ((uint32_t)(q * 32) << 16);
            if (MODE == kModeWgrad) {
                // dW rows [m0 + 32 q, +32) of this warp, 32 columns at a time: lane = row writes
                // its 32 values into a swizzled staging tile (16-byte chunk c of row r at chunk
                // c ^ (r & 7)), then lane 0 stores the tile with TMA. Two tiles per warp: a tile
                // is rewritten only after the store issued two chunks earlier has read it.
                const uint32_t stg = smem_u32(smem + Layout<MODE>::staging) + q * 8192;
                const bool zero = t.kbs == 0;  // an expert without rows: zero gradient
                if (p.dw_bf16) {
                    // bf16 dW: 64 columns per staging tile (two TMEM loads), the same 32 rows x
                    // 128 bytes and swizzle as the fp32 tiles
#pragma unroll 1
                    for (int c = 0; c < 4; ++c) {
                        if (t.n0 + c * 64 >= p.N) break;
                        uint32_t v0[32], v1[32];
                        if (!zero) {
                            tmem_ld_32x32b_x32(tbase + c * 64, v0);
                            tmem_ld_32x32b_x32(tbase + c * 64 + 32, v1);
                            tmem_ld_wait();
                        } else {
#pragma unroll
                            for (int i = 0; i < 32; ++i) v0[i] = v1[i] = 0u;
                        }
                        const uint32_t buf = stg + (uint32_t)(n_store & 1) * 4096;
                        if (lane == 0) bulk_wait_read<1>();
                        __syncwarp();
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            // chunk j: columns 8j .. 8j+7 of the 64
                            const uint32_t* src = j < 4 ? v0 + 8 * j : v1 + 8 * (j - 4);
                            uint32_t w[4];
#pragma unroll
                            for (int h = 0; h < 4; ++h)
                                w[h] = pack_bf16x2(__uint_as_float(src[2 * h]),
                                                   __uint_as_float(src[2 * h + 1]));
                            const uint32_t a = buf + lane * 128 + ((j ^ (lane & 7)) << 4);
                            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a),
                                         "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3])
                                         : "memory");
                        }
                        fence_proxy_async_smem();  // generic stores -> the TMA engine's reads
                        __syncwarp();
                        if (lane == 0) {
                            tma_store_3d(&tmO, buf, t.n0 + c * 64, t.m0 + q * 32, t.e);
                            bulk_commit();
                        }
                        ++n_store;
                    }
                }
#pragma unroll 1
                for (int c = 0; c < 8 && !p.dw_bf16; ++c) {
                    if (t.n0 + c * 32 >= p.N) break;
                    uint32_t v[32];
                    if (!zero) {
                        tmem_ld_32x32b_x32(tbase + c * 32, v);
                        tmem_ld_wait();
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i) v[i] = 0u;
                    }
                    const uint32_t buf = stg + (uint32_t)(n_store & 1) * 4096;
                    if (lane == 0) bulk_wait_read<1>();
                    __syncwarp();
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const uint32_t a = buf + lane * 128 + ((j ^ (lane & 7)) << 4);
                        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a),
                                     "r"(v[4 * j]), "r"(v[4 * j + 1]), "r"(v[4 * j + 2]),
                                     "r"(v[4 * j + 3])
                                     : "memory");
                    }
                    fence_proxy_async_smem();  // generic stores -> the TMA engine's reads
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_3d(&tmO, buf, t.n0 + c * 32, t.m0 + q * 32, t.e);
                        bulk_commit();
                    }
                    ++n_store;
                }
            } else if (MODE == kModeDgradGateUp) {
                // fp32 rows [row0 + 32 q, +32) of dx_sorted, written row by row after a transpose
                // through shared memory (lane = column inside a 32-column chunk); rows past the
                // expert's end belong to another tile and are not written
                float* xp = xpose + q * 32 * 33;
                const int r0 = t.row0 + q * 32;
                float* base = static_cast<float*>(p.out);
#pragma unroll 1
                for (int c = 0; c < 8; ++c) {
                    const int col = t.n0 + c * 32 + lane;
                    if (t.n0 + c * 32 >= p.N) break;
                    uint32_t v[32];
                    tmem_ld_32x32b_x32(tbase + c * 32, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 32; ++j) xp[lane * 33 + j] = __uint_as_float(v[j]);
                    __syncwarp();
                    if (col < p.N) {
#pragma unroll 4
                        for (int r = 0; r < 32; ++r) {
                            if (r0 + r < t.row_end)
                                base[(size_t)(r0 + r) * p.N + col] = xp[r * 33 + lane];
                        }
                    }
                    __syncwarp();
                }
            } else {
                // SwiGLU backward on dh (the accumulator) with the saved a, b of this row
                const int row = t.row0 + q * 32 + lane;
                const bool row_ok = row < t.row_end;
                float s = 1.0f;
                if (p.row_scale && row_ok) s = __ldg(p.topk_weights + __ldg(p.sorted_to_slot + row));
                const size_t rbase = (size_t)(row_ok ? row : 0) * p.ldab;
                __nv_bfloat16* dab = static_cast<__nv_bfloat16*>(p.out);
                float ds = 0.0f;
                // a, b of 32 columns, loaded one chunk ahead of the math
                uint4 ca[4], cb[4], na[4], nb[4];
                auto load_chunk = [&](int c, uint4(&a_)[4], uint4(&b_)[4]) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int col = t.n0 + c * 32 + 8 * j;
                        if (row_ok && col < p.I) {
                            a_[j] = __ldg(reinterpret_cast<const uint4*>(p.ab + rbase + col));
                            b_[j] = __ldg(reinterpret_cast<const uint4*>(p.ab + rbase + p.I + col));
                        } else {
                            a_[j] = b_[j] = make_uint4(0u, 0u, 0u, 0u);
                        }
                    }
                };
                load_chunk(0, ca, cb);
#pragma unroll 1
                for (int c = 0; c < 8; ++c) {
                    if (c + 1 < 8) load_chunk(c + 1, na, nb);
                    uint32_t v[32];
                    tmem_ld_32x32b_x32(tbase + c * 32, v);
                    tmem_ld_wait();
                    const int col0 = t.n0 + c * 32;
                    if (row_ok) {
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const int col = col0 + 8 * j;
                            if (col < p.I) {
                                const uint4 av = ca[j];
                                const uint4 bv = cb[j];
                                const uint32_t aw[4] = {av.x, av.y, av.z, av.w};
                                const uint32_t bw[4] = {bv.x, bv.y, bv.z, bv.w};
                                uint32_t oa[4], ob[4];
#pragma unroll
                                for (int h2 = 0; h2 < 4; ++h2) {
                                    float da[2], db[2];
#pragma unroll
                                    for (int z = 0; z < 2; ++z) {
                                        const float a = __uint_as_float(
                                            z ? (aw[h2] & 0xFFFF0000u) : (aw[h2] << 16));
                                        const float b = __uint_as_float(
                                            z ? (bw[h2] & 0xFFFF0000u) : (bw[h2] << 16));
                                        const float dh = __uint_as_float(v[8 * j + 2 * h2 + z]);
                                        const float g = s * a, u = s * b;
                                        const float sig = __frcp_rn(1.0f + __expf(-g));
                                        const float dg = dh * u * sig * (1.0f + g * (1.0f - sig));
                                        const float du = dh * g * sig;
                                        ds = fmaf(dg, a, fmaf(du, b, ds));
                                        da[z] = s * dg;
                                        db[z] = s * du;
                                    }
                                    oa[h2] = pack_bf16x2(da[0], da[1]);
                                    ob[h2] = pack_bf16x2(db[0], db[1]);
                                }
                                *reinterpret_cast<uint4*>(dab + rbase + col) =
                                    make_uint4(oa[0], oa[1], oa[2], oa[3]);
                                *reinterpret_cast<uint4*>(dab + rbase + p.I + col) =
                                    make_uint4(ob[0], ob[1], ob[2], ob[3]);
                            }
                        }
                    }
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        ca[j] = na[j];
                        cb[j] = nb[j];
                    }
                }
                if (p.row_scale && row_ok)
                    p.scale_part[(size_t)row * p.n_tiles + t.n0 / 256] = ds;
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&st.tempty[acc]);
        }
        // the staging tiles must stay valid until the stores have read them, and the stores
        // must be done before the kernel ends
        if (MODE == kModeWgrad && lane == 0) bulk_wait_all();
        __syncwarp();
    }

    // ---- teardown ----
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, kTmemCols);
}

}  // namespace

namespace {

template <int MODE>
cudaError_t set_smem_attr() {
    return ensure_max_dynamic_smem(tc_bwd_gemm<MODE>, (int)Layout<MODE>::bytes);
}

template <int MODE>
cudaError_t launch_mode(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmO,
                        const BwdParams& p, long long tiles_ub, cudaStream_t s) {
    const cudaError_t e = set_smem_attr<MODE>();
    if (e != cudaSuccess) return e;
    int grid = device_sm_count();
    if (tiles_ub < grid) grid = (int)tiles_ub;
    if (grid < 1) grid = 1;
    return launch_kernel(tc_bwd_gemm<MODE>, dim3(grid), dim3(kThreads), Layout<MODE>::bytes, s,
                         tmA, tmB, tmO, p);
}

}  // namespace

cudaError_t launch_dgrad_bf16(const DgradArgs& a, cudaStream_t s) {
    const int groups = a.offsets ? a.E : 1;
    const bool down = a.kind == kDgradDown;
    const int K = down ? a.d : 2 * a.I;  // contraction: columns of the incoming gradient
    const int N = down ? a.I : a.d;      // output columns
    CUtensorMap tmA, tmB;
    const cuuint64_t a_dims[2] = {(cuuint64_t)K, (cuuint64_t)a.R};
    const cuuint64_t a_str[1] = {(cuuint64_t)K * 2};
    const cuuint32_t a_box[2] = {64, 128};
    const cuuint32_t b_box[3] = {64, 256, 1};
    // the weight read K-major: a row of the tile is one output column's 64 K values
    const PackedGeom g = down ? packed_geom(kDown, a.I, a.d) : packed_geom(kGateUp, a.d, a.I);
    bool ok = encode_tensor_map_bf16(&tmA, a.a, 2, a_dims, a_str, a_box);
    if (a.packed) {
        const cuuint64_t dims[3] = {64, (cuuint64_t)g.kpad, (cuuint64_t)groups * g.nb};
        const cuuint64_t str[2] = {128, (cuuint64_t)g.kpad * 128};
        ok = ok && encode_tensor_map_bf16(&tmB, a.w, 3, dims, str, b_box);
    } else {
        // w_down [E, I, d]: K = d innermost; w_gate_up [E, d, 2I]: K = 2I innermost
        const cuuint64_t dims[3] = {(cuuint64_t)K, (cuuint64_t)N, (cuuint64_t)groups};
        const cuuint64_t str[2] = {(cuuint64_t)K * 2, (cuuint64_t)K * 2 * N};
        ok = ok && encode_tensor_map_bf16(&tmB, a.w, 3, dims, str, b_box);
    }
    if (!ok) return cudaErrorInvalidValue;
    BwdParams p = {};
    p.offsets = a.offsets;
    p.sorted_to_slot = a.sorted_to_slot;
    p.topk_weights = a.topk_weights;
    p.ab = static_cast<const __nv_bfloat16*>(a.ab);
    p.out = a.out;
    p.scale_part = a.scale_part;
    p.status = a.status;
    p.R = a.R;
    p.E = groups;
    p.N = N;
    p.I = a.I;
    p.n_tiles = (N + 255) / 256;
    // packed: one K block per packed block (gate_up: the gate blocks, then the up blocks)
    p.k_blocks = a.packed ? g.nb : (K + 63) / 64;
    p.row_scale = a.scale_rows ? 1 : 0;
    p.packed = a.packed ? 1 : 0;
    p.nb_w = g.nb;
    p.nbh = g.nbh;
    p.ldab = 2 * a.I;
    const long long tiles_ub = ((long long)(a.R + 127) / 128 + groups) * p.n_tiles;
    // no tensor-map store in dgrad: tmA stands in for the unused output map
    return down ? launch_mode<kModeDgradDown>(tmA, tmB, tmA, p, tiles_ub, s)
                : launch_mode<kModeDgradGateUp>(tmA, tmB, tmA, p, tiles_ub, s);
}

cudaError_t launch_wgrad_bf16(const WgradArgs& a, cudaStream_t s) {
    const int groups = a.offsets ? a.E : 1;
    const cuuint64_t rows = a.R > 0 ? (cuuint64_t)a.R : 1;  // no copy is issued when R == 0
    CUtensorMap tmA, tmB;
    const cuuint64_t a_dims[2] = {(cuuint64_t)a.M, rows};
    const cuuint64_t a_str[1] = {(cuuint64_t)a.M * 2};
    const cuuint64_t b_dims[2] = {(cuuint64_t)a.N, rows};
    const cuuint64_t b_str[1] = {(cuuint64_t)a.N * 2};
    const cuuint32_t box[2] = {64, 64};
    // dW [E, M, N], stored 32 rows x 128 bytes at a time: 32 fp32 or 64 bf16 columns
    CUtensorMap tmO;
    const cuuint64_t esz = a.dw_bf16 ? 2 : 4;
    const cuuint64_t o_dims[3] = {(cuuint64_t)a.N, (cuuint64_t)a.M, (cuuint64_t)groups};
    const cuuint64_t o_str[2] = {(cuuint64_t)a.N * esz, (cuuint64_t)a.N * esz * a.M};
    const cuuint32_t o_box[3] = {a.dw_bf16 ? 64u : 32u, 32, 1};
    if (!encode_tensor_map_bf16(&tmA, a.a, 2, a_dims, a_str, box) ||
        !encode_tensor_map_bf16(&tmB, a.b, 2, b_dims, b_str, box) ||
        !(a.dw_bf16 ? encode_tensor_map_bf16(&tmO, a.dw, 3, o_dims, o_str, o_box)
                    : encode_tensor_map_f32(&tmO, a.dw, 3, o_dims, o_str, o_box)))
        return cudaErrorInvalidValue;
    BwdParams p = {};
    p.offsets = a.offsets;
    p.out = a.dw;
    p.dw_bf16 = a.dw_bf16 ? 1 : 0;
    p.status = a.status;
    p.R = a.R;
    p.E = groups;
    p.M = a.M;
    p.N = a.N;
    p.m_tiles = (a.M + 127) / 128;
    p.n_tiles = (a.N + 255) / 256;
    const long long tiles = (long long)groups * p.m_tiles * p.n_tiles;
    return launch_mode<kModeWgrad>(tmA, tmB, tmO, p, tiles, s);
}

}  // namespace rdg
