// Block-scaled FP8 x FP4 grouped expert GEMM on the sm_103a tensor cores:
// tcgen05.mma.kind::mxf8f6f4.block_scale, operands from shared memory by TMA, E8M0 block scales
// copied into tensor memory with tcgen05.cp, fp32 accumulators in tensor memory.
//
// Expert parallelism page, the Mega MoE paragraph: the fused expert kernel of the newest GPUs
// multiplies 8-bit activations by 4-bit expert weights with block scales. The formats are the
// OCP Microscaling ones (32 consecutive K elements share one E8M0 scale): activations MXFP8
// (E4M3), expert weights MXFP4 (E2M1). The tensor core applies both scales itself, so the
// product needs no dequantized copy of anything:
//
//   gate_up: h = SiLU(s g) (s u) with [g | u] = x_rows . W_gu[e] (128 h columns per tile, gate
//            and up of the same h columns in one 128 x 256 accumulator), rounded to MXFP8 in the
//            epilogue (codes and scales in the layout the down GEMM reads);
//   down:    y = h . W_down[e] (256 output columns per tile), fp32.
//
// Layouts (all written by this library):
//   weights ("MX tensor-core layout", quantised once at load): per group g, the E2M1 codes of
//     logical column c (gate_up: gate columns [0, I) then up columns [I, 2I); down: [0, d)) are
//     Kp / 2 contiguous bytes (Kp = K rounded up to 128; even k in the low nibble), at
//     (g * C + c) * Kp / 2. The scales follow (1024-byte aligned) as 512-byte atoms, one per
//     (g, 128-column block cb, 128-element K chunk kc): byte 16 (n % 32) + 4 (n / 32) + j of
//     atom (g, cb, kc) holds the scale (s + 127) of column n of the block and K block 4 kc + j
//     (127, i.e. 2^0, where the column or the K block lies past the end). gate_up blocks its
//     gate and up halves separately (ceil(I / 128) blocks each).
//   activations (x rows and h, per call): rows grouped by expert with every expert's rows
//     starting at a multiple of 128 (padded row p' = poff[e] + (p - off[e]), poff the prefix of
//     ceil(count / 128) * 128): E4M3 codes [Rp][K], and scale atoms [Rp / 128][ceil(K / 128)]
//     in the same 512-byte form (row m of the 128-row block for n).
//   An atom is exactly what tcgen05.cp.32x128b.warpx4 takes: 32 rows of 16 bytes, copied to
//   every lane quarter of 4 tensor-memory columns, so column c of lane 32 w + r holds the four
//   K-block scales of row r + 32 c; the MMA reads row m's scale at column m / 32, byte j (the
//   scale-factor id of its K step).
//
// Structure (one CTA per SM, 352 threads, tiles expert-major, then N block, then M block):
//   warp 0      A producer: one 128 x 128-byte FP8 box (128B swizzle) and the A scale atom per
//               stage; arms the stage barrier for all of the stage's bytes.
//   warp 10     B producer: two 128-column x 128-element FP4 boxes (TMA type 16U4_ALIGN16B: each
//               16 codes land in 16 bytes, the layout the MMA reads 4-bit operands in) and the
//               two B scale atoms.
//   warp 1      allocates 512 TMEM columns (accumulator 0..255, scale atoms from 256), one lane
//               copies each stage's scale atoms into TMEM and issues 4 MMAs (M=128, N=256, K=32)
//               per stage.
//   warps 2..9  epilogue, two warps per TMEM lane quarter, each over half of the columns.
// The accumulator is single-buffered (the scale columns take the room of a second one), so each
// epilogue warp first loads its 128 accumulator columns into registers and releases the
// accumulator: the next tile's MMAs then overlap the SwiGLU, the MXFP8 rounding and the
// stores. Every mbarrier wait is bounded in time; on expiry the kernel records MOE_ERR_TIMEOUT,
// lets its own copies and MMAs finish, frees TMEM and returns.

#include "mx_tc.cuh"

namespace rdg {
namespace {

constexpr int kStages = 4;
constexpr int kTileRows = 128;
constexpr int kChunk = 128;                          // K elements per stage
constexpr int kABytes = kTileRows * kChunk;          // 16 KB of E4M3
constexpr int kBBoxBytes = 128 * 128;                // 16 KB: 128 columns x 128 K (4-bit, padded)
constexpr int kBBytes = 2 * kBBoxBytes;              // 32 KB
constexpr int kStageBytes = kABytes + kBBytes;       // 48 KB
// a 16U4_ALIGN16B box completes the transaction bytes of the packed codes it reads (8 KB for
// 128 x 128 codes), not the 16 KB it fills in shared memory (measured)
constexpr int kBBoxTxBytes = 128 * 128 / 2;
constexpr int kStageTxBytes = kABytes + 2 * kBBoxTxBytes;  // 32 KB
constexpr int kSfStageBytes = 3 * kAtom;             // A atom + two B atoms
constexpr int kThreads = 352;  // 11 warps: A loads, MMA, 8 epilogue, B loads
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSfCol0 = 256;                    // first TMEM column of the scale atoms
constexpr uint32_t kSfColsPerStage = 16;             // A: +0..3, B: +4..11
constexpr uint64_t kWaitLimitNs = 2000000000ull;     // 2 s for any single wait

struct MxTcParams {
    const int32_t* offsets;         // [E+1] expert row offsets (nullptr: one group of R rows)
    const int32_t* sorted_to_slot;  // gate_up row scale: slot of each sorted row
    const float* topk_weights;
    const uint8_t* a_sf;            // A scale atoms [Rp / 128][KC][512]
    const uint8_t* b_sf;            // B scale atoms [G][CB][KC][512]
    void* out;                      // gate_up: h codes [Rp][N]; down: y fp32 [R][N]
    uint8_t* h_sf;                  // gate_up: h scale atoms [Rp / 128][ceil(N / 128)][512]
    int* status;
    int R, K, N, E;
    int KC;        // ceil(K / 128)
    int CB;        // B scale atoms per group along the columns
    int cbh;       // gate_up: atoms per half (the up half starts at cbh)
    int n_tile;    // 128 (gate_up: h columns) or 256 (down)
    int n_tiles;   // ceil(N / n_tile)
    int row_scale; // gate_up: scale the accumulators by the row's routing weight
};

struct __align__(8) SmemTail {
    uint64_t full[kStages];
    uint64_t empty[kStages];
    uint64_t tfull;
    uint64_t tempty;
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
    int total_tiles;
    int prefix[kMaxE + 1];  // first tile of each expert
    int off[kMaxE + 1];     // row offsets
    int poff[kMaxE + 1];    // padded row offsets (multiples of 128)
    int mt[kMaxE];          // 128-row blocks of each expert
};

constexpr size_t kSmemBytes =
    1024 + (size_t)kStages * (kStageBytes + kSfStageBytes) + sizeof(SmemTail);

struct Tile {
    int e, row0, rows, prow0, n0;
};

__device__ __forceinline__ Tile decode_tile(const SmemTail& st, int E, int n_tile, int tile) {
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
    Tile t;
    t.e = e;
    t.row0 = st.off[e] + mb * kTileRows;
    t.rows = min(kTileRows, st.off[e + 1] - t.row0);
    t.prow0 = st.poff[e] + mb * kTileRows;
    t.n0 = nb * n_tile;
    return t;
}

template <int KIND>
__global__ void __launch_bounds__(kThreads, 1)
    tc_mx_gemm(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
               const MxTcParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* sf_smem = smem + (size_t)kStages * kStageBytes;
    SmemTail& st = *reinterpret_cast<SmemTail*>(sf_smem + (size_t)kStages * kSfStageBytes);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int E = p.E;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&st.full[s], 1);
            mbar_init(&st.empty[s], 1);
        }
        mbar_init(&st.tfull, 1);
        mbar_init(&st.tempty, 8);
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
        if (lane == 0) {
            int acc = 0, pacc = 0;
            for (int e = 0; e < E; ++e) {
                int rows = st.off[e + 1] - st.off[e];
                if (rows < 0) rows = 0;
                const int m = (rows + kTileRows - 1) / kTileRows;
                st.poff[e] = pacc;
                st.mt[e] = m > 0 ? m : 1;  // such experts own no tiles
                st.prefix[e] = acc;
                acc += m * p.n_tiles;
                pacc += m * kTileRows;
            }
            st.poff[E] = pacc;
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

    if (warp == 0 || warp == 10) {
        // ================= TMA producers: warp 0 A codes + A scales, warp 10 B codes + scales
        if (lane == 0) {
            const bool a_side = warp == 0;
            if (a_side) tma_prefetch_desc(&tmA);
            else tma_prefetch_desc(&tmB);
            uint32_t stage = 0, phase = 0;
            uint32_t armed_mask = 0, armed_par = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
                const Tile t = decode_tile(st, E, p.n_tile, tile);
                // B columns of the two boxes and the two scale atoms
                int c_lo, c_hi, cb_lo, cb_hi;
                if (KIND == kGateUp) {
                    c_lo = t.n0;
                    c_hi = p.N + t.n0;
                    cb_lo = t.n0 >> 7;
                    cb_hi = p.cbh + (t.n0 >> 7);
                } else {
                    c_lo = t.n0;
                    c_hi = t.n0 + 128;
                    cb_lo = t.n0 >> 7;
                    cb_hi = cb_lo + 1 < p.CB ? cb_lo + 1 : -1;  // past the last atom: none
                }
                const uint32_t bytes = kStageTxBytes + 2 * kAtom + (cb_hi >= 0 ? kAtom : 0);
                for (int kc = 0; kc < p.KC; ++kc) {
                    if (!mbar_wait(&st.empty[stage], phase ^ 1u, abort_flag, kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    const uint32_t a_dst = smem_u32(smem + (size_t)stage * kStageBytes);
                    const uint32_t sf_dst = smem_u32(sf_smem + (size_t)stage * kSfStageBytes);
                    if (a_side) {
                        mbar_arrive_expect_tx(&st.full[stage], bytes);
                        armed_mask |= 1u << stage;
                        armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
                        tma_load_2d(a_dst, &tmA, &st.full[stage], kc * kChunk, t.prow0);
                        bulk_copy(sf_dst,
                                  p.a_sf + ((size_t)(t.prow0 >> 7) * p.KC + kc) * kAtom, kAtom,
                                  &st.full[stage]);
                    } else {
                        armed_mask |= 1u << stage;
                        armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
                        const uint32_t b_dst = a_dst + kABytes;
                        tma_load_3d(b_dst, &tmB, &st.full[stage], kc * kChunk, c_lo, t.e);
                        tma_load_3d(b_dst + kBBoxBytes, &tmB, &st.full[stage], kc * kChunk, c_hi,
                                    t.e);
                        const uint8_t* bs = p.b_sf + (size_t)t.e * p.CB * p.KC * kAtom;
                        bulk_copy(sf_dst + kAtom, bs + ((size_t)cb_lo * p.KC + kc) * kAtom,
                                  kAtom, &st.full[stage]);
                        if (cb_hi >= 0)
                            bulk_copy(sf_dst + 2 * kAtom,
                                      bs + ((size_t)cb_hi * p.KC + kc) * kAtom, kAtom,
                                      &st.full[stage]);
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
            // every stage this thread filled lands before shared memory is released
            for (int s = 0; s < kStages; ++s)
                if ((armed_mask >> s) & 1u)
                    mbar_wait(&st.full[s], (armed_par >> s) & 1u, nullptr, kWaitLimitNs);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ================= scale copies and MMA issue =================
        if (lane == 0) {
            uint32_t stage = 0, phase = 0, it = 0;
            bool ok = true, issued = false;
            for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x, ++it) {
                if (!mbar_wait(&st.tempty, (it & 1u) ^ 1u, abort_flag, kWaitLimitNs)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                for (int kc = 0; kc < p.KC; ++kc) {
                    if (!mbar_wait(&st.full[stage], phase, abort_flag, kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(smem + (size_t)stage * kStageBytes);
                    const uint32_t b_addr = a_addr + kABytes;
                    const uint32_t sf_addr = smem_u32(sf_smem + (size_t)stage * kSfStageBytes);
                    const uint32_t sf_col = tmem_base + kSfCol0 + stage * kSfColsPerStage;
                    tmem_cp_atom(sf_col, smem_desc_plain(sf_addr));
                    tmem_cp_atom(sf_col + 4, smem_desc_plain(sf_addr + kAtom));
                    tmem_cp_atom(sf_col + 8, smem_desc_plain(sf_addr + 2 * kAtom));
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        // A and B: K-major, 128-byte swizzle, +32 bytes per K=32 step
                        const uint64_t adesc = smem_desc(a_addr + j * 32, 16, 1024);
                        const uint64_t bdesc = smem_desc(b_addr + j * 32, 16, 1024);
                        umma_mx(tmem_base, adesc, bdesc, idesc_mx(kTileRows, 256, (uint32_t)j),
                                sf_col, sf_col + 4, (kc | j) != 0 ? 1u : 0u);
                    }
                    issued = true;
                    umma_commit(&st.empty[stage]);
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (ok) umma_commit(&st.tfull);
            }
            if (!ok) {
                st.abort = 1;
                set_status(p.status, MOE_ERR_TIMEOUT);
            }
            if (*abort_flag && issued) {
                umma_commit(&st.drain);  // completes once every MMA and copy issued above is done
                mbar_wait(&st.drain, 0, nullptr, kWaitLimitNs);
            }
        }
        __syncwarp();
    } else {
        // ================= epilogue (warps 2..9) =================
        // Two warps per TMEM lane quarter, each owning half of the tile's columns (gate_up: 64
        // h columns, i.e. their 64 gate and 64 up accumulator columns; down: 128 output
        // columns). A warp loads its 128 accumulator columns into registers and releases the
        // accumulator at once, so the next tile's MMAs run while it computes and stores.
        const int q = warp & 3;          // TMEM lane quarter of this warp
        const int hf = (warp - 2) >> 2;  // which half of the columns
        uint32_t it = 0;
        for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++it) {
            const Tile t = decode_tile(st, E, p.n_tile, tile);
            if (!mbar_wait(&st.tfull, it & 1u, abort_flag, kWaitLimitNs)) {
                if (lane == 0) {
                    st.abort = 1;
                    set_status(p.status, MOE_ERR_TIMEOUT);
                }
                break;
            }
            tc_fence_after();
            const int m = q * 32 + lane;
            const bool row_ok = m < t.rows;
            const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16);
            uint32_t a0[32], a1[32], a2[32], a3[32];
            if (KIND == kGateUp) {
                tmem_ld_32x32b_x32(tbase + hf * 64, a0);
                tmem_ld_32x32b_x32(tbase + hf * 64 + 32, a1);
                tmem_ld_32x32b_x32(tbase + 128 + hf * 64, a2);
                tmem_ld_32x32b_x32(tbase + 128 + hf * 64 + 32, a3);
            } else {
                tmem_ld_32x32b_x32(tbase + hf * 128, a0);
                tmem_ld_32x32b_x32(tbase + hf * 128 + 32, a1);
                tmem_ld_32x32b_x32(tbase + hf * 128 + 64, a2);
                tmem_ld_32x32b_x32(tbase + hf * 128 + 96, a3);
            }
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&st.tempty);
            if (KIND == kGateUp) {
                float s = 1.0f;
                if (p.row_scale && row_ok)
                    s = __ldg(p.topk_weights + __ldg(p.sorted_to_slot + t.row0 + m));
                uint8_t* hc = static_cast<uint8_t*>(p.out) + (size_t)(t.prow0 + m) * p.N;
                const int col0 = t.n0 + hf * 64;
                const uint32_t sc0 = h_block_mxfp8(a0, a2, s, col0, p.N, row_ok, hc);
                const uint32_t sc1 = h_block_mxfp8(a1, a3, s, col0 + 32, p.N, row_ok, hc);
                if (row_ok) {
                    // this warp's two of the four scales of the row's 128-column chunk
                    const int hkc = (p.N + 127) >> 7;
                    uint8_t* atom = p.h_sf + ((size_t)(t.prow0 >> 7) * hkc + (t.n0 >> 7)) * kAtom;
                    *reinterpret_cast<uint16_t*>(atom + 16 * lane + 4 * q + 2 * hf) =
                        (uint16_t)(sc0 | (sc1 << 8));
                }
            } else if (row_ok) {
                float* yr = static_cast<float*>(p.out) + (size_t)(t.row0 + m) * p.N;
                const int col0 = t.n0 + hf * 128;
                store_y_block(a0, col0, p.N, yr);
                store_y_block(a1, col0 + 32, p.N, yr);
                store_y_block(a2, col0 + 64, p.N, yr);
                store_y_block(a3, col0 + 96, p.N, yr);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, kTmemCols);
}

// ---------------------------------------------------------------------------------------------
// quantisation into the tensor-core layouts
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Logical column of column n of scale block cb (-1: past the end).
__device__ __forceinline__ int tc_block_col(bool gate_up, int N, int cbh, int cb, int n) {
    if (gate_up) {
        const bool up = cb >= cbh;
        const int c = (cb - (up ? cbh : 0)) * 128 + n;
        return c < N ? c + (up ? N : 0) : -1;
    }
    const int c = cb * 128 + n;
    return c < N ? c : -1;
}

// One thread per (group, logical column, K block): 32 bf16 weights of one column (strided by the
// row length in the pages' layout) to 16 bytes of E2M1 codes and one scale byte.
__global__ void __launch_bounds__(256)
    mx_tc_quant_weights_kernel(const __nv_bfloat16* __restrict__ w, int G, int K, int C,
                               int Kp, uint8_t* __restrict__ codes, int N, int cbh, int CB,
                               int KC, uint8_t* __restrict__ sf, int gate_up) {
    griddep_wait();
    const int KBp = Kp / 32;
    const long long total = (long long)G * C * KBp;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        // consecutive threads take consecutive columns (coalesced reads of a weight row)
        const int c = (int)(i % C);
        const long long r = i / C;
        const int kb = (int)(r % KBp);
        const int g = (int)(r / KBp);
        const int k0 = kb * 32;
        float v[32];
        float amax = 0.0f;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            v[j] = k0 + j < K ? __bfloat162float(w[((size_t)g * K + k0 + j) * C + c]) : 0.0f;
            amax = fmaxf(amax, fabsf(v[j]));
        }
        const bool valid = k0 < K;
        const int s = valid ? mx_scale_exp(amax, 2) : 0;
        const float inv = pow2_f32(-s);
        uint32_t wd[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            uint32_t x = 0;
#pragma unroll
            for (int b = 0; b < 4; ++b)
                x |= e2m1x2(v[8 * q + 2 * b] * inv, v[8 * q + 2 * b + 1] * inv) << (8 * b);
            wd[q] = x;
        }
        *reinterpret_cast<uint4*>(codes + ((size_t)g * C + c) * (Kp / 2) + kb * 16) =
            make_uint4(wd[0], wd[1], wd[2], wd[3]);
        // scale byte in the atom of the column's block
        const int half = gate_up && c >= N ? 1 : 0;
        const int cc = c - half * N;
        const int cb = half * cbh + (cc >> 7), n = cc & 127;
        sf[((size_t)(g * CB + cb) * KC + (kb >> 2)) * kAtom + 16 * (n & 31) + 4 * (n >> 5) +
           (kb & 3)] = (uint8_t)(s + 127);
    }
}

// Scale bytes of the atoms' padding (columns past the end of a block): 127.
__global__ void __launch_bounds__(256)
    mx_tc_pad_scales_kernel(int G, int N, int cbh, int CB, int KC, uint8_t* __restrict__ sf,
                            int gate_up) {
    griddep_wait();
    const long long total = (long long)G * CB * KC * 128;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const int n = (int)(i & 127);
        const long long a = i >> 7;  // (g * CB + cb) * KC + kc
        const int cb = (int)((a / KC) % CB);
        if (tc_block_col(gate_up != 0, N, cbh, cb, n) >= 0) continue;
        uint32_t* word = reinterpret_cast<uint32_t*>(sf + a * kAtom + 16 * (n & 31) + 4 * (n >> 5));
        *word = 0x7F7F7F7Fu;
    }
}

// Dequantize the tensor-core layout back to bf16 [G, K, C] (for checks against a host
// quantisation).
__global__ void __launch_bounds__(256)
    mx_tc_dequant_weights_kernel(const uint8_t* __restrict__ codes, const uint8_t* __restrict__ sf,
                                 int G, int K, int C, int Kp, int N, int cbh, int CB, int KC,
                                 int gate_up, __nv_bfloat16* __restrict__ w) {
    griddep_wait();
    const int KB = K / 32;
    const long long total = (long long)G * C * KB;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const int c = (int)(i % C);
        const long long r = i / C;
        const int kb = (int)(r % KB);
        const int g = (int)(r / KB);
        const int half = gate_up && c >= N ? 1 : 0;
        const int cc = c - half * N;
        const int cb = half * cbh + (cc >> 7), n = cc & 127;
        const int s = (int)sf[((size_t)(g * CB + cb) * KC + (kb >> 2)) * kAtom +
                              16 * (n & 31) + 4 * (n >> 5) + (kb & 3)] - 127;
        const float sc = pow2_f32(s);
        const uint8_t* cp = codes + ((size_t)g * C + c) * (Kp / 2) + kb * 16;
        for (int b = 0; b < 16; ++b) {
            const float2 q = e2m1x2_to_f32(cp[b]);
            const int k = kb * 32 + 2 * b;
            w[((size_t)g * K + k) * C + c] = __float2bfloat16_rn(q.x * sc);
            w[((size_t)g * K + k + 1) * C + c] = __float2bfloat16_rn(q.y * sc);
        }
    }
}

// x rows to MXFP8 in the padded tensor-core layout, one warp per token: lane l takes K blocks
// l, l + 32, ...; each block's 32 codes are written to every padded row the token was sent to
// (its routed slots, and with codes_sh its own row of the shared expert's one group), and the
// four scales of a 128-element chunk are gathered into one word of the row's atom.
__global__ void __launch_bounds__(256)
    mx_tc_quant_rows_kernel(const __nv_bfloat16* __restrict__ x, int T, int d, int k, int E,
                            const int32_t* __restrict__ topk_ids,
                            const int32_t* __restrict__ slot_to_sorted,
                            const int32_t* __restrict__ offsets, uint8_t* __restrict__ codes,
                            uint8_t* __restrict__ sf, uint8_t* __restrict__ codes_sh,
                            uint8_t* __restrict__ sf_sh, int KC) {
    __shared__ int s_off[kMaxE + 1], s_poff[kMaxE + 1];
    griddep_wait();
    if (offsets != nullptr) {
        for (int e = threadIdx.x; e <= E; e += blockDim.x) s_off[e] = __ldg(offsets + e);
        __syncthreads();
        if (threadIdx.x == 0) {
            int pacc = 0;
            for (int e = 0; e <= E; ++e) {
                s_poff[e] = pacc;
                if (e < E) {
                    const int rows = s_off[e + 1] - s_off[e];
                    pacc += (rows > 0 ? (rows + kTileRows - 1) / kTileRows : 0) * kTileRows;
                }
            }
        }
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int KB = d / 32, KBp = 4 * KC;
    const int nwarps = gridDim.x * (blockDim.x >> 5);
    for (int t = blockIdx.x * (blockDim.x >> 5) + warp; t < T; t += nwarps) {
        // destinations: padded rows of the token's slots (-1: an id the dispatch skipped)
        int dst[kMaxK + 1];
        int nd = 0;
        if (offsets != nullptr) {
            for (int j = 0; j < k; ++j) {
                const int e = __ldg(topk_ids + (size_t)t * k + j);
                const int pos = __ldg(slot_to_sorted + (size_t)t * k + j);
                dst[nd++] = (e >= 0 && e < E && pos >= 0) ? s_poff[e] + (pos - s_off[e]) : -1;
            }
        }
        for (int kb0 = 0; kb0 < KBp; kb0 += 32) {
            const int kb = kb0 + lane;
            uint32_t w[8] = {0, 0, 0, 0, 0, 0, 0, 0};
            uint32_t sc = 127;
            if (kb < KB) {
                const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * d + kb * 32);
                float v[32];
                float amax = 0.0f;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint4 u = src[q];
                    const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        v[8 * q + 2 * h] = bf_lo(w4[h]);
                        v[8 * q + 2 * h + 1] = bf_hi(w4[h]);
                    }
                }
#pragma unroll
                for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
                const int s = mx_scale_exp(amax, 8);
                const float inv = pow2_f32(-s);
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    w[i] = e4m3x2(v[4 * i] * inv, v[4 * i + 1] * inv) |
                           (e4m3x2(v[4 * i + 2] * inv, v[4 * i + 3] * inv) << 16);
                sc = (uint32_t)(s + 127);
            }
            // the word of four scales (K blocks 4 c .. 4 c + 3) lands on the lane of block 4 c
            uint32_t word = sc;
            word |= __shfl_down_sync(0xffffffffu, sc, 1) << 8;
            word |= __shfl_down_sync(0xffffffffu, sc, 2) << 16;
            word |= __shfl_down_sync(0xffffffffu, sc, 3) << 24;
            const bool has_codes = kb < KB, has_word = (kb & 3) == 0 && kb < KBp;
            for (int i = 0; i <= nd; ++i) {
                int row;
                uint8_t *cd, *sfp;
                if (i < nd) {
                    row = dst[i];
                    cd = codes;
                    sfp = sf;
                } else {
                    if (codes_sh == nullptr) break;
                    row = t;
                    cd = codes_sh;
                    sfp = sf_sh;
                }
                if (row < 0) continue;
                if (has_codes) {
                    uint4* o = reinterpret_cast<uint4*>(cd + (size_t)row * d + kb * 32);
                    o[0] = make_uint4(w[0], w[1], w[2], w[3]);
                    o[1] = make_uint4(w[4], w[5], w[6], w[7]);
                }
                if (has_word) {
                    const int m = row & 127;
                    *reinterpret_cast<uint32_t*>(sfp + ((size_t)(row >> 7) * KC + (kb >> 2)) * kAtom +
                                                 16 * (m & 31) + 4 * (m >> 5)) = word;
                }
            }
        }
    }
}

int grid_for(long long work) {
    const long long cap = (long long)device_sm_count() * 8;
    long long g = (work + 255) / 256;
    if (g > cap) g = cap;
    return (int)(g < 1 ? 1 : g);
}

}  // namespace

MxTcGeom mx_tc_geom(bool gate_up, int K, int N, int G) {
    MxTcGeom m;
    m.C = gate_up ? 2 * N : N;
    m.Kp = (K + 127) / 128 * 128;
    m.KC = m.Kp / 128;
    m.cbh = (N + 127) / 128;
    m.CB = gate_up ? 2 * m.cbh : m.cbh;
    m.sf_off = ((size_t)G * m.C * (m.Kp / 2) + 1023) / 1024 * 1024;
    m.total = m.sf_off + (size_t)G * m.CB * m.KC * kAtom;
    return m;
}

cudaError_t launch_mx_tc_quant_weights(bool gate_up, const void* w, int G, int K, int N, void* mx,
                                       cudaStream_t s) {
    const MxTcGeom m = mx_tc_geom(gate_up, K, N, G);
    uint8_t* base = static_cast<uint8_t*>(mx);
    cudaError_t e = launch_kernel(mx_tc_pad_scales_kernel,
                                  dim3(grid_for((long long)G * m.CB * m.KC * 128)), dim3(256), 0,
                                  s, G, N, m.cbh, m.CB, m.KC, base + m.sf_off, gate_up ? 1 : 0);
    if (e != cudaSuccess) return e;
    // the codes of the padding K blocks must be zero: the quantiser writes every K block up to Kp
    return launch_kernel(mx_tc_quant_weights_kernel,
                         dim3(grid_for((long long)G * m.C * (m.Kp / 32))), dim3(256), 0, s,
                         static_cast<const __nv_bfloat16*>(w), G, K, m.C, m.Kp, base, N, m.cbh,
                         m.CB, m.KC, base + m.sf_off, gate_up ? 1 : 0);
}

cudaError_t launch_mx_tc_dequant_weights(bool gate_up, const void* mx, int G, int K, int N,
                                         void* w, cudaStream_t s) {
    const MxTcGeom m = mx_tc_geom(gate_up, K, N, G);
    const uint8_t* base = static_cast<const uint8_t*>(mx);
    return launch_kernel(mx_tc_dequant_weights_kernel,
                         dim3(grid_for((long long)G * m.C * (K / 32))), dim3(256), 0, s, base,
                         base + m.sf_off, G, K, m.C, m.Kp, N, m.cbh, m.CB, m.KC,
                         gate_up ? 1 : 0, static_cast<__nv_bfloat16*>(w));
}

cudaError_t launch_mx_tc_quant_rows(const void* x, int T, int d, int k, int E,
                                    const int32_t* topk_ids, const int32_t* slot_to_sorted,
                                    const int32_t* offsets, void* codes, void* sf, void* codes_sh,
                                    void* sf_sh, cudaStream_t s) {
    const int KC = (d + 127) / 128;
    long long blocks = ((long long)T + 7) / 8;
    const long long cap = (long long)device_sm_count() * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    return launch_kernel(mx_tc_quant_rows_kernel, dim3((unsigned)blocks), dim3(256), 0, s,
                         static_cast<const __nv_bfloat16*>(x), T, d, k, E, topk_ids,
                         slot_to_sorted, offsets, static_cast<uint8_t*>(codes),
                         static_cast<uint8_t*>(sf), static_cast<uint8_t*>(codes_sh),
                         static_cast<uint8_t*>(sf_sh), KC);
}

namespace {
template <int KIND>
cudaError_t launch_mx_tc_kind(const MxTcGemmArgs& a, cudaStream_t s) {
    {
        const cudaError_t e = ensure_max_dynamic_smem(tc_mx_gemm<KIND>, (int)kSmemBytes);
        if (e != cudaSuccess) return e;
    }
    const bool gu = KIND == kGateUp;
    const MxTcGeom wg = mx_tc_geom(gu, a.K, a.N, a.groups);
    const int KC = (a.K + 127) / 128;
    CUtensorMap tmA, tmB;
    // A: E4M3 codes [Rp][K], boxes of 128 rows x 128 bytes
    const cuuint64_t a_dims[2] = {(cuuint64_t)a.K, (cuuint64_t)a.Rp};
    const cuuint64_t a_str[1] = {(cuuint64_t)a.K};
    const cuuint32_t a_box[2] = {128, 128};
    // B: E2M1 codes [G][C][Kp] (packed two per byte), boxes of 128 columns x 128 elements that
    // land 16 codes per 16 bytes
    const cuuint64_t b_dims[3] = {(cuuint64_t)wg.Kp, (cuuint64_t)wg.C, (cuuint64_t)a.groups};
    const cuuint64_t b_str[2] = {(cuuint64_t)wg.Kp / 2, (cuuint64_t)wg.C * wg.Kp / 2};
    const cuuint32_t b_box[3] = {128, 128, 1};
    if (!encode_tensor_map(&tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, a.a, a_dims, a_str, a_box) ||
        !encode_tensor_map(&tmB, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 3, a.b, b_dims, b_str,
                           b_box))
        return cudaErrorInvalidValue;
    MxTcParams p;
    p.offsets = a.offsets;
    p.sorted_to_slot = a.sorted_to_slot;
    p.topk_weights = a.topk_weights;
    p.a_sf = static_cast<const uint8_t*>(a.a_sf);
    p.b_sf = static_cast<const uint8_t*>(a.b) + wg.sf_off;
    p.out = a.out;
    p.h_sf = static_cast<uint8_t*>(a.h_sf);
    p.status = a.status;
    p.R = a.R;
    p.K = a.K;
    p.N = a.N;
    p.E = a.groups;
    p.KC = KC;
    p.CB = wg.CB;
    p.cbh = wg.cbh;
    p.n_tile = gu ? 128 : 256;
    p.n_tiles = (a.N + p.n_tile - 1) / p.n_tile;
    p.row_scale = a.scale_rows ? 1 : 0;
    const long long m_ub = (long long)(a.R + kTileRows - 1) / kTileRows + a.groups;
    const long long tiles_ub = m_ub * p.n_tiles;
    int grid = device_sm_count();
    if (tiles_ub < grid) grid = (int)tiles_ub;
    if (grid < 1) grid = 1;
    return launch_kernel(tc_mx_gemm<KIND>, dim3(grid), dim3(kThreads), kSmemBytes, s, tmA, tmB,
                         p);
}
}  // namespace

cudaError_t launch_mx_tc_gemm(const MxTcGemmArgs& a, cudaStream_t s) {
    return a.kind == kGateUp ? launch_mx_tc_kind<kGateUp>(a, s) : launch_mx_tc_kind<kDown>(a, s);
}

}  // namespace rdg
