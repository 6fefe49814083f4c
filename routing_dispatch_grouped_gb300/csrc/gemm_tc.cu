// Grouped expert GEMM on the sm_103a tensor cores (tcgen05 + TMEM + TMA), bf16 in, fp32 accumulate.
//
// Tensor parallelism page, "Packed strategies": the experts' gate and up projections are one
// packed weight [E, hidden, 2*expert_dim] applied with a batched matmul and split in two along
// the last dimension (gate first). Expert parallelism page, "Adding an implementation":
// experts_forward runs each expert on the rows routed to it. Here both become one persistent
// grouped GEMM over ragged per-expert row ranges read from the device offsets (no host sync):
//
//   gate_up: for rows of expert e, accumulate [gate | up] = x_rows . W_gu[e][:, n0:n0+128 | I+n0:..]
//            in one 128 x 256 fp32 TMEM accumulator (one N=256 MMA covers both halves), then the
//            epilogue applies the optional row scale and SiLU(gate) * up and stores bf16 h.
//   down:    y = h . W_down[e][:, n0:n0+256] into a 128 x 256 accumulator; the epilogue applies
//            the optional row weight and stores fp32.
//
// Structure (one CTA per SM, 192 threads):
//   warp 0        TMA producer: A tile 128 x 64 (K-major, 128B swizzle) and four 64 x 64 weight
//                 blocks (MN-major, 128B swizzle) per stage, 4 stages in shared memory.
//   warp 1        allocates 512 TMEM columns (two 256-column accumulators), one lane issues
//                 tcgen05.mma (M=128, N=256, K=16) and commits stage/accumulator barriers.
//   warps 2..5    epilogue: tcgen05.ld of their 32 TMEM lanes, math, 16-byte global stores,
//                 while the MMA warp fills the other accumulator.
// Tiles are ordered expert-major, then by N block, then by M block, so the CTAs working at
// the same time share weight blocks through L2. Every mbarrier wait is bounded in time; on
// expiry the kernel records MOE_ERR_TIMEOUT, drains its own copies and MMAs, frees TMEM and
// returns.
#include <mutex>

#include "mx.cuh"

namespace rdg {
namespace {

constexpr int kStages = 4;
constexpr int kABytes = kTileM * kTileK * 2;       // 16 KB
constexpr int kBBlockBytes = 64 * kTileK * 2;      // 8 KB: 64 columns x 64 k-rows
constexpr int kBBytes = 4 * kBBlockBytes;          // 32 KB
constexpr int kStageBytes = kABytes + kBBytes;     // 48 KB
constexpr int kThreads = 224;  // 7 warps: A loads, MMA, 4 epilogue, weight loads
constexpr uint32_t kTmemCols = 512;
constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s for any single wait

struct TcParams {
    const int32_t* offsets;  // [E+1] or nullptr
    const int32_t* sorted_to_slot;
    const float* topk_weights;
    void* out;
    int* status;
    int R, K, N, E;
    int n_tile;      // output columns per tile: 128 (gate_up) or 256 (down)
    int n_tiles;     // ceil(N / n_tile)
    int k_blocks;    // ceil(K / 64)
    int row_scale;   // gate_up: scale accumulators; down: weight rows
    int packed;      // weights in the packed layout (PackedGeom below)
    int nb, nbh, kpad;
    __nv_bfloat16* ab;  // gate_up for training: [g | u] before the row scale, [R, 2N]
    int mx_h;           // gate_up: round h to MXFP8 (32-column blocks) before storing it
    uint32_t stall_ns;  // test hook: the MMA issuer first waits this long on a barrier that
                        // nothing completes, then gives up as on an expired wait (0 = off)
};

struct __align__(8) SmemTail {
    uint64_t full[kStages];
    uint64_t empty[kStages];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t drain;
    uint64_t never;  // completed by nothing: the stall_ns test hook waits on it
    uint32_t tmem_base;
    int abort;
    int total_tiles;
    int prefix[kMaxE + 1];  // first tile index of each expert
    int off[kMaxE + 1];     // row offsets
    int mt[kMaxE];          // M blocks of each expert
};

constexpr size_t kSmemBytes = 1024 + (size_t)kStages * kStageBytes + sizeof(SmemTail);

struct TileInfo {
    int e, row0, row_end, n0;
};

__device__ __forceinline__ TileInfo decode_tile(const SmemTail& st, int E, int n_tiles,
                                                int n_tile, int tile) {
    int lo = 0, hi = E - 1;  // largest e with prefix[e] <= tile
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
    const int nb = local / m, mb = local - nb * m;
    TileInfo ti;
    ti.e = e;
    ti.row0 = st.off[e] + mb * kTileM;
    ti.row_end = st.off[e + 1];
    ti.n0 = nb * n_tile;
    return ti;
}



template <int KIND>
__global__ void __launch_bounds__(kThreads, 1)
    tc_grouped_gemm(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const TcParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    SmemTail& st = *reinterpret_cast<SmemTail*>(smem + (size_t)kStages * kStageBytes);

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
        mbar_init(&st.never, 1);
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
                const int m = (rows + kTileM - 1) / kTileM;
                st.mt[e] = m > 0 ? m : 1;  // avoid division by zero; such experts own no tiles
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
                const TileInfo ti = decode_tile(st, E, p.n_tiles, p.n_tile, tile);
                for (int kb = 0; kb < p.k_blocks; ++kb) {
                    if (!mbar_wait(&st.empty[stage], phase ^ 1u, abort_flag, kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&st.full[stage], kStageBytes);
                    armed[stage] = true;
                    armed_phase[stage] = phase;
                    const uint32_t a_dst = smem_u32(smem + (size_t)stage * kStageBytes);
                    const uint32_t b_dst = a_dst + kABytes;
                    const int kc = kb * kTileK;
                    (void)b_dst;
                    tma_load_2d(a_dst, &tmA, &st.full[stage], kc, ti.row0);
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
            // let every copy this thread started land before shared memory is released: after
            // an abort elsewhere nothing else waits for them (on the normal path they have
            // landed already, as the MMA issuer waited for each stage)
            for (int s = 0; s < kStages; ++s)
                if (armed[s]) mbar_wait(&st.full[s], armed_phase[s], nullptr, kWaitLimitNs);
        }
        __syncwarp();
    } else if (warp == 6) {
        // ================= TMA producer, weight blocks =================
        // Same stage sequence as warp 0; warp 0 arms each stage's barrier for all 48 KB, this
        // warp's copies complete their share of it. Two issuing threads double the rate at which
        // copies are started.
        if (lane == 0) {
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
                const TileInfo ti = decode_tile(st, E, p.n_tiles, p.n_tile, tile);
                for (int kb = 0; kb < p.k_blocks; ++kb) {
                    if (!mbar_wait(&st.empty[stage], phase ^ 1u, abort_flag, kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    armed[stage] = true;
                    armed_phase[stage] = phase;
                    const uint32_t b_dst = smem_u32(smem + (size_t)stage * kStageBytes) + kABytes;
                    const int kc = kb * kTileK;
                    if (p.packed) {
                        // packed blocks of one expert are adjacent along the third dimension:
                        // gate_up = {gate n0, gate n0+64} + {up n0, up n0+64} (two copies of two
                        // blocks), down = the four blocks from n0 (one copy)
                        const int blk0 = ti.e * p.nb + (ti.n0 >> 6);
                        tma_load_3d(b_dst, &tmB, &st.full[stage], 0, kc, blk0);
                        if (KIND == kGateUp)
                            tma_load_3d(b_dst + 2 * kBBlockBytes, &tmB, &st.full[stage], 0, kc,
                                        blk0 + p.nbh);
                    } else if (KIND == kGateUp) {
                        tma_load_3d(b_dst, &tmB, &st.full[stage], ti.n0, kc, ti.e);
                        tma_load_3d(b_dst + kBBlockBytes, &tmB, &st.full[stage], ti.n0 + 64, kc,
                                    ti.e);
                        tma_load_3d(b_dst + 2 * kBBlockBytes, &tmB, &st.full[stage], p.N + ti.n0,
                                    kc, ti.e);
                        tma_load_3d(b_dst + 3 * kBBlockBytes, &tmB, &st.full[stage],
                                    p.N + ti.n0 + 64, kc, ti.e);
                    } else {
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            tma_load_3d(b_dst + j * kBBlockBytes, &tmB, &st.full[stage],
                                        ti.n0 + 64 * j, kc, ti.e);
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
            for (int s = 0; s < kStages; ++s)
                if (armed[s]) mbar_wait(&st.full[s], armed_phase[s], nullptr, kWaitLimitNs);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ================= MMA issuer =================
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(kTileM, kTileN, true);
            uint32_t stage = 0, phase = 0, it = 0;
            bool ok = true, issued = false;
            if (p.stall_ns != 0 && !mbar_wait(&st.never, 0, nullptr, p.stall_ns)) ok = false;
            for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x, ++it) {
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
                    const uint32_t a_addr = smem_u32(smem + (size_t)stage * kStageBytes);
                    const uint32_t b_addr = a_addr + kABytes;
#pragma unroll
                    for (int kk = 0; kk < kTileK / 16; ++kk) {
                        // A: K-major, +32 bytes per K=16 step inside the 128-byte swizzle row.
                        // B: MN-major, 64-column blocks 8 KB apart (LBO), 8-row groups 1 KB apart
                        //    (SBO), +2 KB per K=16 step.
                        const uint64_t adesc = smem_desc(a_addr + kk * 32, 16, 1024);
                        const uint64_t bdesc = smem_desc(b_addr + kk * 2048, kBBlockBytes, 1024);
                        umma_bf16(d_tmem, adesc, bdesc, idesc, (kb | kk) != 0 ? 1u : 0u);
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
                umma_commit(&st.drain);  // completes once every MMA issued above is done
                mbar_wait(&st.drain, 0, nullptr, kWaitLimitNs);
            }
        }
        __syncwarp();
    } else {
        // ================= epilogue (warps 2..5) =================
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        uint32_t it = 0;
        for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++it) {
            const TileInfo ti = decode_tile(st, E, p.n_tiles, p.n_tile, tile);
            const uint32_t acc = it & 1u;
            if (!mbar_wait(&st.tfull[acc], (it >> 1) & 1u, abort_flag, kWaitLimitNs)) {
                if (lane == 0) {
                    st.abort = 1;
                    set_status(p.status, MOE_ERR_TIMEOUT);
                }
                break;
            }
            tc_fence_after();
            const int row = ti.row0 + q * 32 + lane;
            const bool row_ok = row < ti.row_end;
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
                    const int col0 = ti.n0 + c * 32;
                    if (row_ok && p.ab) {
                        // the unscaled accumulators, kept for the backward pass
                        __nv_bfloat16* ab = p.ab + (size_t)row * 2 * p.N + col0;
#pragma unroll
                        for (int v = 0; v < 4; ++v) {
                            if (col0 + v * 8 < p.N) {
                                uint32_t wg[4], wu[4];
#pragma unroll
                                for (int h2 = 0; h2 < 4; ++h2) {
                                    const int i = v * 8 + h2 * 2;
                                    wg[h2] = pack_bf16x2(__uint_as_float(g[i]),
                                                         __uint_as_float(g[i + 1]));
                                    wu[h2] = pack_bf16x2(__uint_as_float(u[i]),
                                                         __uint_as_float(u[i + 1]));
                                }
                                reinterpret_cast<uint4*>(ab)[v] = make_uint4(wg[0], wg[1], wg[2], wg[3]);
                                reinterpret_cast<uint4*>(ab + p.N)[v] =
                                    make_uint4(wu[0], wu[1], wu[2], wu[3]);
                            }
                        }
                    }
                    if (row_ok && p.mx_h) {
                        // the chunk's 32 columns are one MX block of h (col0 is a multiple of
                        // 32): SwiGLU in fp32, rounded to MXFP8 (exact in bf16)
                        float hv[32];
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            const float gi = __uint_as_float(g[i]) * s;
                            hv[i] = silu(gi) * (__uint_as_float(u[i]) * s);
                        }
                        mx_fakequant_e4m3_block(hv, min(32, p.N - col0));
                        uint4* dst = reinterpret_cast<uint4*>(out + (size_t)row * p.N + col0);
#pragma unroll
                        for (int v = 0; v < 4; ++v) {
                            if (col0 + v * 8 < p.N)
                                dst[v] = make_uint4(pack_bf16x2(hv[8 * v], hv[8 * v + 1]),
                                                    pack_bf16x2(hv[8 * v + 2], hv[8 * v + 3]),
                                                    pack_bf16x2(hv[8 * v + 4], hv[8 * v + 5]),
                                                    pack_bf16x2(hv[8 * v + 6], hv[8 * v + 7]));
                        }
                    } else if (row_ok) {
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
                    const int col0 = ti.n0 + c * 32;
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
            if (lane == 0) mbar_arrive(&st.tempty[acc]);
        }
    }

    // ---- teardown ----
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, kTmemCols);
}

}  // namespace

// ---------------------------------------------------------------------------------------------
// host side: tensor maps (shared with the swapped-operand kernel) and launch
// ---------------------------------------------------------------------------------------------
namespace {
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}
}  // namespace

bool encode_tensor_map_bf16(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims,
                            const cuuint64_t* strides, const cuuint32_t* box) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint32_t elem[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, const_cast<void*>(base), dims,
              strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_tensor_map(CUtensorMap* m, CUtensorMapDataType type, int rank, const void* base,
                       const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box,
                       bool swizzle128) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint32_t elem[3] = {1, 1, 1};
    return fn(m, type, (cuuint32_t)rank, const_cast<void*>(base), dims, strides, box, elem,
              CU_TENSOR_MAP_INTERLEAVE_NONE,
              swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_tensor_map_f32(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims,
                           const cuuint64_t* strides, const cuuint32_t* box) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint32_t elem[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, (cuuint32_t)rank, const_cast<void*>(base), dims,
              strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {

template <int KIND>
cudaError_t launch_kind(const GroupedGemmArgs& a, cudaStream_t s) {
    {
        const cudaError_t e = ensure_max_dynamic_smem(tc_grouped_gemm<KIND>, (int)kSmemBytes);
        if (e != cudaSuccess) return e;
    }

    CUtensorMap tmA, tmB;
    const cuuint64_t a_dims[2] = {(cuuint64_t)a.K, (cuuint64_t)a.R};
    const cuuint64_t a_str[1] = {(cuuint64_t)a.K * 2};
    const cuuint32_t a_box[2] = {kTileK, kTileM};
    const int groups = a.offsets ? a.E : 1;
    const cuuint64_t bn = (KIND == kGateUp) ? 2 * (cuuint64_t)a.N : (cuuint64_t)a.N;
    const cuuint64_t b_dims[3] = {bn, (cuuint64_t)a.K, (cuuint64_t)groups};
    const cuuint64_t b_str[2] = {bn * 2, bn * 2 * (cuuint64_t)a.K};
    const cuuint32_t b_box[3] = {64, kTileK, 1};
    const PackedGeom g = packed_geom(KIND, a.K, a.N);
    // packed: {64 columns, Kpad rows, blocks}; one copy = 2 (gate_up) or 4 (down) blocks
    const cuuint64_t pk_dims[3] = {64, (cuuint64_t)g.kpad, (cuuint64_t)groups * g.nb};
    const cuuint64_t pk_str[2] = {128, (cuuint64_t)g.kpad * 128};
    const cuuint32_t pk_box[3] = {64, kTileK, (KIND == kGateUp) ? 2u : 4u};
    if (!encode_tensor_map_bf16(&tmA, a.a, 2, a_dims, a_str, a_box) ||
        !(a.packed ? encode_tensor_map_bf16(&tmB, a.b, 3, pk_dims, pk_str, pk_box)
                   : encode_tensor_map_bf16(&tmB, a.b, 3, b_dims, b_str, b_box)))
        return cudaErrorInvalidValue;

    TcParams p;
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
    p.row_scale = (KIND == kGateUp) ? (a.scale_rows ? 1 : 0) : (a.weight_rows ? 1 : 0);
    p.packed = a.packed ? 1 : 0;
    p.nb = g.nb;
    p.nbh = g.nbh;
    p.kpad = g.kpad;
    p.ab = static_cast<__nv_bfloat16*>(a.ab);
    p.mx_h = a.mx_h ? 1 : 0;
    p.stall_ns = debug_gemm_stall_ns();

    // upper bound on tiles: sum_e ceil(n_e / 128) <= R / 128 + groups
    const long long m_ub = (long long)(a.R + kTileM - 1) / kTileM + groups;
    const long long tiles_ub = m_ub * p.n_tiles;
    int grid = device_sm_count();
    if (tiles_ub < grid) grid = (int)tiles_ub;
    if (grid < 1) grid = 1;
    return launch_kernel(tc_grouped_gemm<KIND>, dim3(grid), dim3(kThreads), kSmemBytes, s, tmA, tmB, p);
}

}  // namespace

cudaError_t launch_grouped_gemm_bf16_rows(const GroupedGemmArgs& a, cudaStream_t s) {
    return a.kind == kGateUp ? launch_kind<kGateUp>(a, s) : launch_kind<kDown>(a, s);
}

}  // namespace rdg
