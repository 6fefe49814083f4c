// Fused decode layer: router top-k, dispatch, gate_up + SwiGLU, down and the weighted combine
// for a handful of tokens in one persistent kernel.
//
// Same definitions as the multi-kernel path (Expert parallelism page, "Adding an
// implementation": the router returns top_k_index and top_k_weights, each expert runs on the
// rows routed to it and the outputs are combined with the routing weights; "Token dispatch":
// rows of an expert in ascending slot order; Tensor parallelism page, "Packed strategies":
// gate_up [E, d, 2I] with the gate half first), organised for decode (Expert parallelism page,
// "Choosing an implementation": a decode step must need no host synchronisation and be
// graph-capturable). With at most 16 tokens every weight element meets at most 16 rows: the
// layer is a stream of the touched experts' weights, and its cost is keeping every SM's memory
// pipe full and the few dependent steps short.
//
// Every block first routes all tokens and builds the dispatch indices in shared memory (the
// same warp router and counting sort as the stand-alone kernels, so the ids and the order
// agree bit for bit; with at most 32 slots one warp builds the same indices by votes); block 0
// also writes them out. Then the work takes one of two layouts, picked on the host from the
// sizes (one kernel instantiation each).
//
// Stream-K layout. Work items are 32 KB weight chunks:
//   gate_up item (q, jb, kc): K rows [128 kc, 128 kc + 128) of gate columns [64 jb, 64 jb + 64)
//     of the q-th touched expert and the same rows of the matching up columns. Items are
//     ordered (q, jb, kc); a group (q, jb) is one 64-column block of h.
//   down item (c, q, kc): K rows [256 kc, 256 kc + 256) of output columns [64 c, 64 c + 64) of
//     expert q. Items are ordered (c, q, kc); a group c is one 64-column block of the output.
// Each list is split into G equal contiguous ranges (one per block, "stream-K"), so every SM
// streams the same number of bytes. A producer warp streams a block's gate_up range and then
// its down range through a 6-stage TMA ring; consumer warp w owns stage w and multiplies each
// of its items alone with warp-level mma.sync (m16n8k16, bf16 in, fp32 accumulate: the weights
// are the M side, read with ldmatrix.trans from the TMA tile, the at most 16 rows the N side),
// so six items are in flight per SM and no barrier is taken per item. The layer is bound by
// HBM, not by the tensor pipe: the MMAs only keep each warp's work per 32 KB item small. At
// the end of a group the consumer warps hand their register sums to an epilogue warp through
// a shared-memory buffer (an mbarrier pair) and go on streaming; the epilogue warp adds them
// up and does everything that follows:
//   - gate_up: a block that covers a whole group applies SwiGLU (and the router scale when it
//     applies to the input) to its register sums, rounds h to bf16 and stores it. A group
//     split between blocks leaves one fp32 partial per block; the last of them to arrive (a
//     per-group counter) sums the partials in block order and stores h. Either way the writer
//     then raises the group's h flag.
//   - down: a consumer warp waits (bounded) until every h block of its expert is flagged and
//     loads h; the epilogue warp adds weight * y of the expert's rows into a per-token
//     accumulator in shared memory (the combine: an expert appears at most once per token).
//     At the end of an output block it either writes bf16 out (sole contributor) or leaves
//     the block's per-token partial; the last contributor sums them in block order, one
//     rounding.
// While a block waits, its producer keeps streaming down weights.
//
// Owner layout (taken while the final sums below come to at most two units per block). Every
// block owns whole h blocks: h block b while there are fewer h blocks than blocks (T = 1 at the
// decode shape), else an equal contiguous share (4 or 5 at T = 8). For each of them it streams
// the gate_up items, then, through the same ring, the down weight rows of those 64 h columns for
// every output column: bf16 items of four [64 K][64 column] boxes (256 output columns), MX
// items of both 32-row K blocks of 14 output column blocks. The gate_up items of the next owned
// h block are streamed ahead of the down items of the current one, so the ring keeps streaming
// while h is finished. The epilogue warp stores h as above and also keeps it in shared memory
// (two buffers, one mbarrier each), so the consumer warps multiply the down items by it at
// once: h crosses no SM and no flag is waited on. Each consumer writes its item's weighted sums
// per token row as an fp32 partial and bumps the item's counter. Then, per (64 output columns,
// token), the blocks past the owners (or all blocks, once their own h blocks are done) sum the
// partials of the token's rows (sorted row order) and h blocks (block order) and store bf16
// out: one rounding, in a fixed order.
//
// The launch is cooperative, so every block is resident and the waits end. Every sum runs in an order fixed by the sizes
// alone: results do not depend on timing. The counters are zeroed by the caller's memset of
// the workspace head that precedes the launch.

#include "mx.cuh"
#include "decode_route.cuh"

namespace rdg {
namespace {

constexpr int kStages = 6;
constexpr int kConsumerWarps = kStages;         // warp w consumes the items of stage w
constexpr int kProducerWarp = kConsumerWarps;  // streams the weights
constexpr int kEpilogueWarp = kConsumerWarps + 1;  // reductions, h, combine
constexpr int kThreads = (kConsumerWarps + 2) * 32;
constexpr int kWarps = kThreads / 32;
constexpr int kKcA = 128;                       // K rows of a gate_up item (two boxes)
constexpr int kKcB = 256;                       // K rows of a down item (one box)
constexpr int kBoxBytesA = 64 * kKcA * 2;       // 16 KB
constexpr int kStageBytes = 64 * kKcB * 2;      // 32 KB
constexpr int kPass = 8;                        // rows per MMA n-tile and reduction pass
constexpr int kStrideA = 132;                   // reduction row strides (padded: no bank
constexpr int kStrideB = 68;                    // conflicts on the fragment-layout stores)
constexpr int kRedFloats = kConsumerWarps * kPass * kStrideA;  // [6][8][132] >= [6][8][68]
constexpr int kOutFloats = kDecodeFusedMaxTokens * 64;         // per-token output accumulator
constexpr uint64_t kWaitLimitNs = 2000000000ull;
// MX weights (MXFP4 codes in 1 KB blocks of 64 columns x 32 K rows, 64 scale bytes each): a
// gate_up item is up to 15 K blocks of its gate and up column blocks, a down item up to 30 K
// blocks of one output column block; codes, then scales, within the 32 KB stage.
constexpr int kMxKbA = 15;  // at most; the launch picks 15 (T = 1) or 11 (Params::kba)
constexpr int kMxKbB = 30;
constexpr uint32_t kMxUpCodes = 15 * 1024;     // up codes after the gate codes (gate_up item)
constexpr uint32_t kMxScales = 30 * 1024;      // scales after the codes
constexpr uint32_t kMxUpScales = kMxScales + 15 * 64;
// owner layout, MX: a down item holds the 64 h rows (two 32-row K blocks) of up to 6 output
// column blocks (six items cover the decode shape's 32, one per consumer warp): codes [column
// block][K block][1 KB], then scales [column block][K block][64]
constexpr int kMxOwnCb = 6;
constexpr uint32_t kMxOwnScales = kMxOwnCb * 2 * 1024;
static_assert(kMxOwnScales + kMxOwnCb * 2 * 64 <= kStageBytes, "owner MX item exceeds a stage");
constexpr int kMxHsScales = kDecodeFusedMaxTokens * 64;  // h_s (MX): codes, then 2 scales a row
static_assert(kMxUpScales + 15 * 64 <= kStageBytes && kMxScales + 30 * 64 <= kStageBytes,
              "MX items exceed a stage");
constexpr int kDecodeWaves = 1;                 // expert waves (gate_up of wave w + 1 hides the
                                                // finishing of wave w's h)

constexpr size_t kOffRed = (size_t)kStages * kStageBytes;
constexpr size_t kOffOut = kOffRed + kRedFloats * 4;
constexpr size_t kOffLists = kOffOut + kOutFloats * 4;
constexpr size_t kListInts = 3 * kMaxE + 2 * kDecodeFusedMaxRows;
constexpr size_t kOffBars = kOffLists + kListInts * 4;
constexpr size_t kSmemBytes = kOffBars + (2 * kStages + 4) * 8 + 64 + 1024;  // + align slack
static_assert(kSmemBytes <= 232448, "exceeds the 227 KB of shared memory a block may use");

struct Params {
    const __nv_bfloat16* x;  // [T, d]
    const float* logits;     // [T, E]
    int32_t* topk_ids;       // [T, k] out
    float* topk_w;           // [T, k] out
    int32_t* counts;         // [E] out
    int32_t* offsets;        // [E + 1] out
    int32_t* s2p;            // [R] out: sorted row -> slot t*k + j
    int32_t* p2s;            // [R] out: slot -> sorted row
    __nv_bfloat16* h;        // [R, I] out
    __nv_bfloat16* out;      // [T, d] out
    float* part_a;           // [G + groups_a][T][128] gate/up partials
    float* part_b;           // [G + nbd][T][64] per-token partials of split output blocks
    int* cnt_a;              // [R * nbh] contributors arrived, per h block
    int* hflag;              // [R * nbh] h block stored
    int* cnt_b;              // [nbd] per output block
    // owner layout (see the schedule): down partials [nbh][R][d] (weighted, fp32; null when
    // the layout cannot occur) and, per 256 output columns, the owners done with them
    float* part_c;
    int* cnt_c;
    int* status;
    int T, d, E, k, I, R;
    int score_fn, renorm;
    int nbh, nka, nbd, nkb;
    int scale_input, packed;
    int gu_nb, dn_nb;        // packed blocks per expert (gate_up, down); MX: column blocks
    // MX layers: weights as MX buffers (codes then scales), h rounded to MXFP8 into h_codes
    // [R, I] / h_scales [R, kbi] for the down items (and its values into h, bf16)
    const uint8_t* mx_gu;
    const uint8_t* mx_dn;
    size_t mx_gu_scales, mx_dn_scales;  // scale offsets in the buffers
    uint8_t* h_codes;
    uint8_t* h_scales;
    int kbd, kbi;            // 32-row K blocks of d and I
    int kba;                 // MX gate_up items: 32-row K blocks per item (<= kMxKbA)
    int mx;
};

// What a block's consumers share.
struct Ctx {
    uint32_t stage0;         // shared address of stage 0
    float* red;              // cross-warp reduction buffer
    float* outacc;           // [T][64] per-token output accumulator
    const int* s_off;        // touched expert q -> first sorted row
    const int* s_tq;         // -> row count
    const int* s_tok;        // sorted row -> token
    const float* s_w;        // sorted row -> routing weight
    uint64_t* full;
    uint64_t* empty;
    uint64_t* red_full;      // the consumer warps have written a dump
    uint64_t* red_empty;     // the epilogue warp has read it
    volatile int* flags;     // [0] something timed out
    int warp, lane, G;
    int GA;                  // blocks [0, GA) share the gate_up items
    int B0, GB;              // blocks [B0, B0 + GB) share the down items
    int nA;                  // gate_up items of the current wave
    int slot_off;            // partial slot offset of the current wave (see the schedule)
    int W, nq;               // waves, touched experts
    int ready_q;             // touched expert whose h blocks ready_mask covers (-1: none)
    bool owner;              // owner layout: h stays in this block (h_s), no flags
    __nv_bfloat16* h_s;      // [rows of the block's expert][64]: its h block
    uint64_t* h_full;        // h_s written
    uint64_t ready_mask;     // h blocks of ready_q this warp has seen stored (all ones: every)
    int dumps;               // hand-overs so far
};

// First item of block b's range when n items are split into G ranges, and the block whose
// range holds item u.
__device__ __forceinline__ int range_lo(int n, int b, int G) {
    return (int)((long long)n * b / G);
}
__device__ __forceinline__ int block_of(int n, int u, int G) {
    return (int)(((long long)(u + 1) * G - 1) / n);
}
// With fewer items than blocks some ranges are empty; such blocks take part in no group.
__device__ __forceinline__ bool range_empty(int n, int b, int G) {
    return n < G && range_lo(n, b, G) == range_lo(n, b + 1, G);
}
__device__ __forceinline__ int contributors(int n, int G, int b_first, int b_last) {
    if (n >= G) return b_last - b_first + 1;
    int m = 0;
    for (int b = b_first; b <= b_last; ++b) m += range_empty(n, b, G) ? 0 : 1;
    return m;
}

// One m16n8k16 step: the A fragment of columns [m0, m0 + 16) x K rows [k0, k0 + 16) of a
// 128-byte-swizzled [k][64 column] box, read with ldmatrix.trans (lanes 0-7 address rows
// k0..k0+7 at columns m0.. -> a0, lanes 8-15 columns m0+8.. -> a1, lanes 16-23 rows k0+8.. ->
// a2, lanes 24-31 both -> a3; PTX ISA, "Matrix fragments for mma.m16n8k16"), times NTILE B
// fragments (8 rows each), accumulated into acc[n] (C: m = l/4 [+8], n = 2 (l%4) [+1]).
template <int NTILE>
__device__ __forceinline__ void mma_step(uint32_t box, int k0, int m0, int lane,
                                         const uint32_t (&b)[NTILE][2], float (&acc)[NTILE][4]) {
    const int k = k0 + (lane & 7) + ((lane >> 4) << 3);
    const int chunk = (m0 >> 3) + ((lane >> 3) & 1);
    const uint32_t addr = box + (uint32_t)k * 128 + (uint32_t)((chunk ^ (k & 7)) << 4);
    uint32_t a0, a1, a2, a3;
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(a0), "=r"(a1), "=r"(a2), "=r"(a3)
                 : "r"(addr));
#pragma unroll
    for (int n = 0; n < NTILE; ++n) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
            "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
            : "+f"(acc[n][0]), "+f"(acc[n][1]), "+f"(acc[n][2]), "+f"(acc[n][3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b[n][0]), "r"(b[n][1]));
    }
}

// ---- MX helpers ----
// f16x2 from one byte of two E2M1 codes (low nibble in the low half) / two E4M3 codes.
__device__ __forceinline__ uint32_t e2m1x2_f16x2(uint32_t byte) {
    uint32_t h2;
    asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}"
        : "=r"(h2)
        : "r"(byte));
    return h2;
}
__device__ __forceinline__ uint32_t e4m3x2_f16x2(uint32_t two) {
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"((uint16_t)two));
    return h2;
}
// acc[n] += A (16 x 16, f16) . B[n] (16 x 8, f16), fp32 accumulate
template <int NTILE>
__device__ __forceinline__ void mma_f16(const uint32_t (&a)[4], const uint32_t (&b)[NTILE][2],
                                        float (&acc)[NTILE][4]) {
#pragma unroll
    for (int n = 0; n < NTILE; ++n)
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
            "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
            : "+f"(acc[n][0]), "+f"(acc[n][1]), "+f"(acc[n][2]), "+f"(acc[n][3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[n][0]), "r"(b[n][1]));
}
// 1D bulk copy global -> shared completing on an mbarrier, with an L2 policy.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint64_t* bar, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(pol)
        : "memory");
}
__device__ __forceinline__ uint32_t lds32(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}
// An E8M0 scale code c as fp32: 2^(c - 127) (c = 0: 2^-127, a subnormal; 255 is not produced).
__device__ __forceinline__ float e8m0_f32(uint32_t c) {
    return __uint_as_float(c ? c << 23 : 0x400000u);
}
__device__ __forceinline__ uint32_t lds8(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.u8 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}

// B fragments of the gate_up step for K rows [k0, k0 + 16): lane l holds row 8 n + l/4 of the
// group (rows[n] points at that token's x row; null past the group's rows), K pairs
// k0 + 2 (l%4) and k0 + 8 + 2 (l%4). K past d is zero.
template <int NTILE>
__device__ __forceinline__ void load_b_x(const unsigned int* const (&rows)[NTILE], int k0, int d,
                                         int lane, uint32_t (&b)[NTILE][2]) {
#pragma unroll
    for (int n = 0; n < NTILE; ++n) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int kk = k0 + 8 * h + 2 * (lane & 3);
            b[n][h] = (rows[n] != nullptr && kk < d) ? __ldg(rows[n] + kk / 2) : 0u;
        }
    }
}

// B fragments of the down step for K rows [k0, k0 + 16) (h columns): like load_b_x, from the
// expert's h rows, which other blocks stored in this launch (read through L2).
template <int NTILE>
__device__ __forceinline__ void load_b_h(const unsigned int* const (&rows)[NTILE], int k0, int I,
                                         int lane, uint32_t (&b)[NTILE][2]) {
#pragma unroll
    for (int n = 0; n < NTILE; ++n) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int kk = k0 + 8 * h + 2 * (lane & 3);
            b[n][h] = (rows[n] != nullptr && kk < I) ? __ldcg(rows[n] + kk / 2) : 0u;
        }
    }
}

// Wait for the stage of block-local item i (warp i % kStages owns it).
__device__ __forceinline__ bool take_stage(Ctx& c, const Params& p, int i) {
    const bool ok = mbar_wait(&c.full[c.warp], (uint32_t)(i / kStages) & 1u, c.flags,
                              kWaitLimitNs);
    if (!ok) {
        set_status(p.status, MOE_ERR_TIMEOUT);
        c.flags[0] = 1;
    }
    return ok;
}
__device__ __forceinline__ void release_stage(Ctx& c) {
    __syncwarp();
    if (c.lane == 0) mbar_arrive(&c.empty[c.warp]);
}

// gate_up item in this warp's stage: 128 K rows x (64 gate + 64 up) columns; acc[mt], m-tiles
// 0-3 gate, 4-7 up. The item's B fragments are all loaded before the first MMA.
template <int NTILE>
__device__ __forceinline__ void item_a(Ctx& c, const Params& p, int i, int kc,
                                       const unsigned int* const (&rows)[NTILE],
                                       float (&acc)[8][NTILE][4]) {
    const uint32_t stage = c.stage0 + (uint32_t)c.warp * kStageBytes;
    uint32_t b[kKcA / 16][NTILE][2];
#pragma unroll
    for (int ks = 0; ks < kKcA / 16; ++ks)
        load_b_x<NTILE>(rows, kc * kKcA + 16 * ks, p.d, c.lane, b[ks]);
    if (take_stage(c, p, i)) {
#pragma unroll
        for (int ks = 0; ks < kKcA / 16; ++ks)
#pragma unroll
            for (int mt = 0; mt < 8; ++mt)
                mma_step<NTILE>(stage + (uint32_t)(mt >> 2) * kBoxBytesA, 16 * ks,
                                16 * (mt & 3), c.lane, b[ks], acc[mt]);
    }
    release_stage(c);
}

// down item in this warp's stage: 256 K rows x 64 output columns; acc[mt], m-tiles of 16
// columns. All B fragments are loaded before the first MMA.
template <int NTILE>
__device__ __forceinline__ void item_b(Ctx& c, const Params& p, int i, int kc,
                                       const unsigned int* const (&rows)[NTILE],
                                       float (&acc)[4][NTILE][4]) {
    const uint32_t stage = c.stage0 + (uint32_t)c.warp * kStageBytes;
    uint32_t b[kKcB / 16][NTILE][2];
#pragma unroll
    for (int ks = 0; ks < kKcB / 16; ++ks)
        load_b_h<NTILE>(rows, kc * kKcB + 16 * ks, p.I, c.lane, b[ks]);
    if (take_stage(c, p, i)) {
#pragma unroll
        for (int ks = 0; ks < kKcB / 16; ++ks)
#pragma unroll
            for (int mt = 0; mt < 4; ++mt)
                mma_step<NTILE>(stage, 16 * ks, 16 * mt, c.lane, b[ks], acc[mt]);
    }
    release_stage(c);
}

__device__ __forceinline__ __nv_bfloat16 store_h(const Params& p, const Ctx& c, int row, int hc,
                                                 float g, float u) {
    const float s = p.scale_input ? c.s_w[row] : 1.0f;
    const __nv_bfloat16 v = __float2bfloat16_rn(silu(g * s) * (u * s));
    p.h[(size_t)row * p.I + hc] = v;
    return v;
}

// MX layers: h rounded to MXFP8 (blocks of 32 along I). Called by all 32 lanes of the epilogue
// warp together, lane l holding column hc of the same 32-column block of one row (valid: hc < I):
// the block's largest magnitude is a warp maximum. Stores the E4M3 code and scale the down items
// read, and the rounded value into h.
__device__ __forceinline__ uint32_t store_h_mx(const Params& p, const Ctx& c, int row, int hc,
                                               float g, float u, bool valid) {
    const float s = p.scale_input ? c.s_w[row] : 1.0f;
    const float hv = valid ? silu(g * s) * (u * s) : 0.0f;
    float amax = fabsf(hv);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    const int se = mx_scale_exp(amax, 8);
    const uint32_t code = e4m3x2(hv * pow2_f32(-se), 0.0f) & 0xFFu;
    if (valid) {
        p.h_codes[(size_t)row * p.I + hc] = (uint8_t)code;
        p.h[(size_t)row * p.I + hc] = __float2bfloat16_rn(e4m3x2_to_f32(code).x * pow2_f32(se));
        if (c.lane == 0) p.h_scales[(size_t)row * p.kbi + hc / 32] = (uint8_t)(se + 127);
    }
    return (valid ? code : 0u) | ((uint32_t)(se + 127) << 8);
}

// First item of [i0, ...) that warp w owns (item i belongs to warp i % kStages).
__device__ __forceinline__ int first_owned(int i0, int w) {
    return i0 + ((w - i0 % kStages) + kStages) % kStages;
}

// ---- hand-over of register sums from the consumer warps to the epilogue warp: one
// reduction buffer and an mbarrier pair (red_full: the six consumer warps have written dump d;
// red_empty: the epilogue warp has read it)
__device__ __forceinline__ void dump_begin(Ctx& c, const Params& p) {
    if (!mbar_wait(c.red_empty, ((uint32_t)c.dumps & 1u) ^ 1u, c.flags, kWaitLimitNs)) {
        set_status(p.status, MOE_ERR_TIMEOUT);
        c.flags[0] = 1;
    }
}
__device__ __forceinline__ void dump_end(Ctx& c) {
    __syncwarp();
    if (c.lane == 0) mbar_arrive(c.red_full);
    ++c.dumps;
}
__device__ __forceinline__ void epi_take(Ctx& c, const Params& p) {
    if (!mbar_wait(c.red_full, (uint32_t)c.dumps & 1u, c.flags, kWaitLimitNs)) {
        set_status(p.status, MOE_ERR_TIMEOUT);
        c.flags[0] = 1;
    }
}
__device__ __forceinline__ void epi_give(Ctx& c) {
    __syncwarp();
    if (c.lane == 0) mbar_arrive(c.red_empty);
    ++c.dumps;
}

// Bump a group counter after this warp's partial stores; true for the last contributor.
__device__ __forceinline__ bool epi_arrive_last(const Ctx& c, int* counter, int contributors) {
    __syncwarp();
    int prev = 0;
    if (c.lane == 0)  // releases this warp's partial stores, acquires the others'
        asm volatile("atom.add.acq_rel.gpu.global.s32 %0, [%1], 1;"
                     : "=r"(prev)
                     : "l"(counter)
                     : "memory");
    prev = __shfl_sync(0xFFFFFFFFu, prev, 0);
    return prev == contributors - 1;
}

// ---- MX items (MXFP4 weights, MXFP8 activations) ----
// Per 32-row K block: the lanes' A fragments are one word each (two k-steps per block), the
// MMA runs on the element values in f16 (exact), and the block's partial sums are added to the
// fp32 accumulators times the weight column's and the token's block scales.

// This lane's x words of K block kbg (bf16 pairs): for token row 8 n + l/4, K values
// kbg 32 + 16 ks + 8 h + 2 (l & 3) + {0, 1} in w[n][2 ks + h]. Loaded ahead of their use.
template <int NTILE>
__device__ __forceinline__ void mx_x_load(const unsigned int* const (&rows)[NTILE], int kbg,
                                          int d, int lane, uint32_t (&w)[NTILE][4]) {
#pragma unroll
    for (int n = 0; n < NTILE; ++n)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int kk = kbg * 32 + 16 * (j >> 1) + 8 * (j & 1) + 2 * (lane & 3);
            w[n][j] = (rows[n] != nullptr && kk < d) ? __ldg(rows[n] + kk / 2) : 0u;
        }
}

// B fragments of one K block from its x words, rounded to MXFP8 as the row quantiser rounds x:
// the four lanes of a token hold its 32 values, so two shuffles give the block's largest
// magnitude. sxc[n][j]: the block scale of token 8 n + 2 (l & 3) + j (the C fragment's columns).
template <int NTILE>
__device__ __forceinline__ void mx_x_quant(const uint32_t (&w)[NTILE][4], int lane,
                                           uint32_t (&b)[2][NTILE][2], float (&sxc)[NTILE][2]) {
#pragma unroll
    for (int n = 0; n < NTILE; ++n) {
        float v[4][2];
        float amax = 0.0f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            v[j][0] = __uint_as_float(w[n][j] << 16);
            v[j][1] = __uint_as_float(w[n][j] & 0xFFFF0000u);
            amax = fmaxf(amax, fmaxf(fabsf(v[j][0]), fabsf(v[j][1])));
        }
        amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
        const int se = mx_scale_exp(amax, 8);
        const float inv = pow2_f32(-se), sc = pow2_f32(se);
#pragma unroll
        for (int j = 0; j < 4; ++j)
            b[j >> 1][n][j & 1] = e4m3x2_f16x2(e4m3x2(v[j][0] * inv, v[j][1] * inv));
        sxc[n][0] = __shfl_sync(0xFFFFFFFFu, sc, 8 * (lane & 3));
        sxc[n][1] = __shfl_sync(0xFFFFFFFFu, sc, 8 * (lane & 3) + 4);
    }
}

// A fragment registers of m-tile mt, k-step ks of K block kbl from a stage's code words.
__device__ __forceinline__ void mx_a(uint32_t codes, int kbl, int ks, int mt, int lane,
                                     uint32_t (&a)[4]) {
    const uint32_t w = lds32(codes + ((((kbl * 2 + ks) * 4 + mt) * 32 + lane) << 2));
    a[0] = e2m1x2_f16x2(w & 0xFF);
    a[1] = e2m1x2_f16x2((w >> 8) & 0xFF);
    a[2] = e2m1x2_f16x2((w >> 16) & 0xFF);
    a[3] = e2m1x2_f16x2(w >> 24);
}

// acc[n] += part[n] times the scales of its rows (weight columns: sw0 for l/4, sw1 for l/4 + 8)
// and columns (tokens: sxc[n][0], sxc[n][1])
template <int NTILE>
__device__ __forceinline__ void mx_rescale(const float (&part)[NTILE][4], float sw0, float sw1,
                                           const float (&sxc)[NTILE][2], float (&acc)[NTILE][4]) {
#pragma unroll
    for (int n = 0; n < NTILE; ++n) {
        acc[n][0] = fmaf(part[n][0], sw0 * sxc[n][0], acc[n][0]);
        acc[n][1] = fmaf(part[n][1], sw0 * sxc[n][1], acc[n][1]);
        acc[n][2] = fmaf(part[n][2], sw1 * sxc[n][0], acc[n][2]);
        acc[n][3] = fmaf(part[n][3], sw1 * sxc[n][1], acc[n][3]);
    }
}

// gate_up item: K blocks [15 kc, ...) of the gate and up column blocks; acc[mt], m-tiles 0-3
// gate, 4-7 up.
template <int NTILE>
__device__ __forceinline__ void item_a_mx(Ctx& c, const Params& p, int i, int kc,
                                          const unsigned int* const (&rows)[NTILE],
                                          float (&acc)[8][NTILE][4]) {
    const uint32_t stage = c.stage0 + (uint32_t)c.warp * kStageBytes;
    const int kb0 = kc * p.kba, nk = min(p.kba, p.kbd - kb0);
    // x words two K blocks ahead of the math (the first two before the stage wait)
    uint32_t w0[NTILE][4], w1[NTILE][4], w2[NTILE][4];
    mx_x_load<NTILE>(rows, kb0, p.d, c.lane, w0);
    mx_x_load<NTILE>(rows, kb0 + 1, p.d, c.lane, w1);
    if (take_stage(c, p, i)) {
        for (int kbl = 0; kbl < nk; ++kbl) {
            mx_x_load<NTILE>(rows, kb0 + kbl + 2, p.d, c.lane, w2);  // past d: zeros, no load
            uint32_t b[2][NTILE][2];
            float sxc[NTILE][2];
            mx_x_quant<NTILE>(w0, c.lane, b, sxc);
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
                const uint32_t half = (uint32_t)(mt >> 2);
                const uint32_t codes = stage + half * kMxUpCodes;
                const uint32_t scl = stage + kMxScales + half * (kMxUpScales - kMxScales) +
                                     kbl * 64 + (mt & 3) * 16 + (c.lane >> 2);
                float part[NTILE][4];
#pragma unroll
                for (int n = 0; n < NTILE; ++n)
#pragma unroll
                    for (int j = 0; j < 4; ++j) part[n][j] = 0.0f;
#pragma unroll
                for (int ks = 0; ks < 2; ++ks) {
                    uint32_t a[4];
                    mx_a(codes, kbl, ks, mt & 3, c.lane, a);
                    mma_f16<NTILE>(a, b[ks], part);
                }
                mx_rescale<NTILE>(part, e8m0_f32(lds8(scl)), e8m0_f32(lds8(scl + 8)), sxc,
                                  acc[mt]);
            }
#pragma unroll
            for (int n = 0; n < NTILE; ++n)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    w0[n][j] = w1[n][j];
                    w1[n][j] = w2[n][j];
                }
        }
    }
    release_stage(c);
}

// down item: K blocks [30 kc, ...) of one output column block. hrow[n]: the expert's h code row
// of this lane's B token (8 n + l/4); hsc[n][j]: the h scale row of token 8 n + 2 (l & 3) + j.
// This lane's h words of K block kbg: codes (two per 16 bits) of its B token row for
// k-steps and halves, and the block scales of its C fragment's token rows.
template <int NTILE>
__device__ __forceinline__ void mx_h_load(const Params& p, const uint8_t* const (&hrow)[NTILE],
                                          const uint8_t* const (&hsc)[NTILE][2], int kbg,
                                          int lane, uint32_t (&w)[NTILE][6]) {
#pragma unroll
    for (int n = 0; n < NTILE; ++n) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int kk = kbg * 32 + 16 * (j >> 1) + 8 * (j & 1) + 2 * (lane & 3);
            w[n][j] = (hrow[n] != nullptr && kk < p.I)
                          ? (uint32_t)__ldcg(reinterpret_cast<const unsigned short*>(hrow[n] + kk))
                          : 0u;
        }
#pragma unroll
        for (int j = 0; j < 2; ++j)
            w[n][4 + j] = (hsc[n][j] != nullptr && kbg < p.kbi) ? (uint32_t)__ldcg(hsc[n][j] + kbg)
                                                                 : 0u;
    }
}

template <int NTILE>
__device__ __forceinline__ void item_b_mx(Ctx& c, const Params& p, int i, int kc,
                                          const uint8_t* const (&hrow)[NTILE],
                                          const uint8_t* const (&hsc)[NTILE][2],
                                          float (&acc)[4][NTILE][4]) {
    const uint32_t stage = c.stage0 + (uint32_t)c.warp * kStageBytes;
    const int kb0 = kc * kMxKbB, nk = min(kMxKbB, p.kbi - kb0);
    uint32_t w0[NTILE][6], w1[NTILE][6], w2[NTILE][6];
    mx_h_load<NTILE>(p, hrow, hsc, kb0, c.lane, w0);
    mx_h_load<NTILE>(p, hrow, hsc, kb0 + 1, c.lane, w1);
    if (take_stage(c, p, i)) {
        for (int kbl = 0; kbl < nk; ++kbl) {
            mx_h_load<NTILE>(p, hrow, hsc, kb0 + kbl + 2, c.lane, w2);
            uint32_t b[2][NTILE][2];
            float sxc[NTILE][2];
#pragma unroll
            for (int n = 0; n < NTILE; ++n) {
#pragma unroll
                for (int j = 0; j < 4; ++j) b[j >> 1][n][j & 1] = e4m3x2_f16x2(w0[n][j]);
#pragma unroll
                for (int j = 0; j < 2; ++j)
                    sxc[n][j] = hsc[n][j] != nullptr ? e8m0_f32(w0[n][4 + j]) : 0.0f;
            }
#pragma unroll
            for (int mt = 0; mt < 4; ++mt) {
                const uint32_t scl = stage + kMxScales + kbl * 64 + mt * 16 + (c.lane >> 2);
                float part[NTILE][4];
#pragma unroll
                for (int n = 0; n < NTILE; ++n)
#pragma unroll
                    for (int j = 0; j < 4; ++j) part[n][j] = 0.0f;
#pragma unroll
                for (int ks = 0; ks < 2; ++ks) {
                    uint32_t a[4];
                    mx_a(stage, kbl, ks, mt, c.lane, a);
                    mma_f16<NTILE>(a, b[ks], part);
                }
                mx_rescale<NTILE>(part, e8m0_f32(lds8(scl)), e8m0_f32(lds8(scl + 8)), sxc,
                                  acc[mt]);
            }
#pragma unroll
            for (int n = 0; n < NTILE; ++n)
#pragma unroll
                for (int j = 0; j < 6; ++j) {
                    w0[n][j] = w1[n][j];
                    w1[n][j] = w2[n][j];
                }
        }
    }
    release_stage(c);
}

// ================= consumer side =================

// gate_up group (q, jb) of this block: block-local items [i0, i0 + kc1 - kc0) = K chunks
// [kc0, kc1); then its register sums go to the epilogue warp, 8 rows per dump, as
// red[warp][row][column] (columns 0-63 gate, 64-127 up).
template <int NTILE, bool MX>
__device__ void group_a(Ctx& c, const Params& p, int q, int i0, int kc0, int kc1) {
    const int row0 = c.s_off[q], tq = c.s_tq[q];
    const unsigned int* rows[NTILE];
#pragma unroll
    for (int n = 0; n < NTILE; ++n) {
        const int r = 8 * n + (c.lane >> 2);
        rows[n] = r < tq ? reinterpret_cast<const unsigned int*>(
                               p.x + (size_t)c.s_tok[row0 + r] * p.d)
                         : nullptr;
    }
    float acc[8][NTILE][4];
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
        for (int n = 0; n < NTILE; ++n)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[mt][n][j] = 0.0f;
    for (int i = first_owned(i0, c.warp); i < i0 + (kc1 - kc0); i += kStages) {
        if (MX)
            item_a_mx<NTILE>(c, p, i, kc0 + (i - i0), rows, acc);
        else
            item_a<NTILE>(c, p, i, kc0 + (i - i0), rows, acc);
    }
#pragma unroll
    for (int pass = 0; pass < NTILE; ++pass) {
        if (pass * kPass < tq) {
            dump_begin(c, p);
            float* rd = c.red + (c.warp * kPass + 2 * (c.lane & 3)) * kStrideA + (c.lane >> 2);
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
                rd[16 * mt] = acc[mt][pass][0];
                rd[kStrideA + 16 * mt] = acc[mt][pass][1];
                rd[16 * mt + 8] = acc[mt][pass][2];
                rd[kStrideA + 16 * mt + 8] = acc[mt][pass][3];
            }
            dump_end(c);
        }
    }
}

// Down items of expert q for one output block: block-local items [i0, i0 + kc1 - kc0) = K
// chunks [kc0, kc1); then the register sums go to the epilogue warp as red[warp][row][column].
template <int NTILE, bool MX>
__device__ void group_b(Ctx& c, const Params& p, int q, int i0, int kc0, int kc1) {
    const int row0 = c.s_off[q], tq = c.s_tq[q];
    const unsigned int* rows[NTILE];
    const uint8_t* hrow[NTILE];
    const uint8_t* hsc[NTILE][2];
#pragma unroll
    for (int n = 0; n < NTILE; ++n) {
        const int r = 8 * n + (c.lane >> 2);
        rows[n] = r < tq ? reinterpret_cast<const unsigned int*>(p.h + (size_t)(row0 + r) * p.I)
                         : nullptr;
        if (MX) {
            hrow[n] = r < tq ? p.h_codes + (size_t)(row0 + r) * p.I : nullptr;
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int t = 8 * n + 2 * (c.lane & 3) + j;
                hsc[n][j] = t < tq ? p.h_scales + (size_t)(row0 + t) * p.kbi : nullptr;
            }
        }
    }
    float acc[4][NTILE][4];
#pragma unroll
    for (int mt = 0; mt < 4; ++mt)
#pragma unroll
        for (int n = 0; n < NTILE; ++n)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[mt][n][j] = 0.0f;
    for (int i = first_owned(i0, c.warp); i < i0 + (kc1 - kc0); i += kStages) {
        if (c.ready_q != q) {
            c.ready_q = q;
            c.ready_mask = 0;
        }
        // the h blocks this item reads must be stored (bounded wait; the launch is
        // cooperative): an item covers K rows [K_item kc, K_item kc + K_item) of h (256 rows,
        // or 30 MX blocks = 960 rows), i.e. its 64-column blocks K_item / 64 * kc onwards, so
        // the item waits for those and not for the rest of the expert's h. Lane j watches
        // block j of the range (the whole expert, lanes j, j + 32, ..., when it has more than
        // 64 blocks and no mask covers them).
        {
            constexpr int kBlocksPerItem = (MX ? kMxKbB * 32 : kKcB) / 64;
            static_assert((MX ? kMxKbB * 32 : kKcB) % 64 == 0, "items cover whole h blocks");
            const int kc = kc0 + (i - i0);
            const bool masked = p.nbh <= 64;
            const int jb_lo = masked ? kBlocksPerItem * kc : 0;
            const int jb_hi = masked ? min(p.nbh, jb_lo + kBlocksPerItem) : p.nbh;
            const uint64_t need =
                masked ? (((jb_hi - jb_lo) >= 64 ? ~0ull : ((1ull << (jb_hi - jb_lo)) - 1)) << jb_lo)
                       : ~0ull;
            if ((c.ready_mask & need) != need) {
                for (int jb = jb_lo + c.lane; jb < jb_hi; jb += 32) {
                    const uint64_t t0 = globaltimer_ns();
                    while (ld_acquire(p.hflag + q * p.nbh + jb) == 0) {
                        if (c.flags[0] || globaltimer_ns() - t0 > kWaitLimitNs) {
                            set_status(p.status, MOE_ERR_TIMEOUT);
                            c.flags[0] = 1;
                            break;
                        }
                    }
                }
                __syncwarp();
                c.ready_mask |= need;
            }
        }
        if (MX)
            item_b_mx<NTILE>(c, p, i, kc0 + (i - i0), hrow, hsc, acc);
        else
            item_b<NTILE>(c, p, i, kc0 + (i - i0), rows, acc);
    }
#pragma unroll
    for (int pass = 0; pass < NTILE; ++pass) {
        if (pass * kPass < tq) {
            dump_begin(c, p);
            float* rd = c.red + (c.warp * kPass + 2 * (c.lane & 3)) * kStrideB + (c.lane >> 2);
#pragma unroll
            for (int mt = 0; mt < 4; ++mt) {
                rd[16 * mt] = acc[mt][pass][0];
                rd[kStrideB + 16 * mt] = acc[mt][pass][1];
                rd[16 * mt + 8] = acc[mt][pass][2];
                rd[kStrideB + 16 * mt + 8] = acc[mt][pass][3];
            }
            dump_end(c);
        }
    }
}

// ---- owner layout: down partials of the block's own h block ----
// Item g4 of h block (q, jb): W_down rows [64 jb, 64 jb + 64) x output columns
// [256 g4, 256 g4 + 256), four [64 K][64 column] boxes; h block from h_s as the B side. Each
// token row's sums, times its routing weight, go to part_c[jb][row], then the group's counter
// is bumped (release) for the summing blocks.
template <int NTILE>
__device__ void owner_down(Ctx& c, const Params& p, int q, int jb, int i0, int n4,
                           uint32_t hphase) {
    const int row0 = c.s_off[q], tq = c.s_tq[q];
    bool have_h = false;
    uint32_t b[4][NTILE][2];
    for (int g4 = (c.warp - i0 % kStages + kStages) % kStages; g4 < n4; g4 += kStages) {
        const int i = i0 + g4;
        if (!have_h) {
            if (!mbar_wait(c.h_full, hphase, c.flags, kWaitLimitNs)) {
                set_status(p.status, MOE_ERR_TIMEOUT);
                c.flags[0] = 1;
            }
            // B fragments: lane l holds token row 8 n + l/4, h columns 16 ks + 2 (l%4) (+8)
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
#pragma unroll
                for (int n = 0; n < NTILE; ++n) {
                    const int r = 8 * n + (c.lane >> 2);
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        const int kk = 16 * ks + 8 * hh + 2 * (c.lane & 3);
                        b[ks][n][hh] =
                            r < tq ? *reinterpret_cast<const uint32_t*>(c.h_s + r * 64 + kk) : 0u;
                    }
                }
            have_h = true;
        }
        float acc[16][NTILE][4];
#pragma unroll
        for (int m = 0; m < 16; ++m)
#pragma unroll
            for (int n = 0; n < NTILE; ++n)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[m][n][j] = 0.0f;
        if (take_stage(c, p, i)) {
            const uint32_t stage = c.stage0 + (uint32_t)c.warp * kStageBytes;
#pragma unroll
            for (int j = 0; j < 4; ++j)
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
#pragma unroll
                    for (int mt = 0; mt < 4; ++mt)
                        mma_step<NTILE>(stage + (uint32_t)j * 8192u, 16 * ks, 16 * mt, c.lane,
                                        b[ks], acc[4 * j + mt]);
        }
        release_stage(c);
        // C fragment: m = output column 16 m + l/4 (+8), n = token row 8 n + 2 (l%4) (+1)
#pragma unroll
        for (int n = 0; n < NTILE; ++n)
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
                const int r = 8 * n + 2 * (c.lane & 3) + (jj & 1);
                if (r >= tq) continue;
                const float wgt = p.scale_input ? 1.0f : c.s_w[row0 + r];
                float* dst = p.part_c + ((size_t)jb * p.R + row0 + r) * p.d;
#pragma unroll
                for (int m = 0; m < 16; ++m) {
                    const int col = 256 * g4 + 16 * m + (c.lane >> 2) + ((jj & 2) ? 8 : 0);
                    if (col < p.d) __stcg(dst + col, wgt * acc[m][n][jj]);
                }
            }
        __syncwarp();
        if (c.lane == 0)
            asm volatile("red.release.gpu.global.add.s32 [%0], 1;" ::"l"(p.cnt_c + g4) : "memory");
    }
}

// Owner layout, MX: down item g4 of h block (q, jb) holds W_down's two 32-row K blocks of the
// 64 h rows (one when I ends inside them) for output column blocks [14 g4, 14 g4 + 14). The B
// side is the h block's MXFP8 codes and scales from h_s; per K block the partial sums are
// added times the weight column's and the token's scales, as in the stream-K items.
template <int NTILE>
__device__ void owner_down_mx(Ctx& c, const Params& p, int q, int jb, int i0, int n4,
                              uint32_t hphase) {
    const int row0 = c.s_off[q], tq = c.s_tq[q];
    const int nkb = min(2, p.kbi - 2 * jb);
    const uint8_t* hb = reinterpret_cast<const uint8_t*>(c.h_s);
    bool have_h = false;
    uint32_t b[2][2][NTILE][2];
    float sxc[2][NTILE][2];
    for (int g4 = (c.warp - i0 % kStages + kStages) % kStages; g4 < n4; g4 += kStages) {
        const int i = i0 + g4;
        if (!have_h) {
            if (!mbar_wait(c.h_full, hphase, c.flags, kWaitLimitNs)) {
                set_status(p.status, MOE_ERR_TIMEOUT);
                c.flags[0] = 1;
            }
            // lane l: B codes of token row 8 n + l/4 at h columns 32 kb + 16 ks + 8 h + 2 (l%4),
            // and the K block scales of its C fragment's token rows 8 n + 2 (l%4) + {0, 1}
#pragma unroll
            for (int kb = 0; kb < 2; ++kb)
#pragma unroll
                for (int n = 0; n < NTILE; ++n) {
                    const int r = 8 * n + (c.lane >> 2);
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int kk = 32 * kb + 16 * (j >> 1) + 8 * (j & 1) + 2 * (c.lane & 3);
                        const uint32_t w =
                            r < tq ? *reinterpret_cast<const unsigned short*>(hb + r * 64 + kk) : 0u;
                        b[kb][j >> 1][n][j & 1] = e4m3x2_f16x2(w);
                    }
#pragma unroll
                    for (int jj = 0; jj < 2; ++jj) {
                        const int rt = 8 * n + 2 * (c.lane & 3) + jj;
                        sxc[kb][n][jj] = rt < tq ? e8m0_f32(hb[kMxHsScales + rt * 2 + kb]) : 0.0f;
                    }
                }
            have_h = true;
        }
        const int cb0 = g4 * kMxOwnCb, ncb = min(kMxOwnCb, p.nbd - cb0);
        const bool taken = take_stage(c, p, i);
        const uint32_t stage = c.stage0 + (uint32_t)c.warp * kStageBytes;
        for (int cbl = 0; cbl < ncb; ++cbl) {
            float acc[4][NTILE][4];
#pragma unroll
            for (int mt = 0; mt < 4; ++mt)
#pragma unroll
                for (int n = 0; n < NTILE; ++n)
#pragma unroll
                    for (int j = 0; j < 4; ++j) acc[mt][n][j] = 0.0f;
            if (taken) {
                for (int kb = 0; kb < nkb; ++kb) {
#pragma unroll
                    for (int mt = 0; mt < 4; ++mt) {
                        float part[NTILE][4];
#pragma unroll
                        for (int n = 0; n < NTILE; ++n)
#pragma unroll
                            for (int j = 0; j < 4; ++j) part[n][j] = 0.0f;
#pragma unroll
                        for (int ks = 0; ks < 2; ++ks) {
                            uint32_t a[4];
                            mx_a(stage + (uint32_t)cbl * 2048u, kb, ks, mt, c.lane, a);
                            mma_f16<NTILE>(a, b[kb][ks], part);
                        }
                        const uint32_t scl = stage + kMxOwnScales + (uint32_t)(cbl * 2 + kb) * 64u +
                                             mt * 16 + (c.lane >> 2);
                        mx_rescale<NTILE>(part, e8m0_f32(lds8(scl)), e8m0_f32(lds8(scl + 8)),
                                          sxc[kb], acc[mt]);
                    }
                }
            }
            // C fragment: m = output column 16 mt + l/4 (+8), n = token row 8 n + 2 (l%4) (+1)
#pragma unroll
            for (int n = 0; n < NTILE; ++n)
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    const int r = 8 * n + 2 * (c.lane & 3) + (jj & 1);
                    if (r >= tq) continue;
                    const float wgt = p.scale_input ? 1.0f : c.s_w[row0 + r];
                    float* dst = p.part_c + ((size_t)jb * p.R + row0 + r) * p.d;
#pragma unroll
                    for (int mt = 0; mt < 4; ++mt) {
                        const int col = 64 * (cb0 + cbl) + 16 * mt + (c.lane >> 2) +
                                        ((jj & 2) ? 8 : 0);
                        if (col < p.d) __stcg(dst + col, wgt * acc[mt][n][jj]);
                    }
                }
        }
        release_stage(c);
        __syncwarp();
        if (c.lane == 0)
            asm volatile("red.release.gpu.global.add.s32 [%0], 1;" ::"l"(p.cnt_c + g4) : "memory");
    }
}

// Owner layout, the summing step: unit u = (output block cb = u / T, token t = u % T) is the
// sum over the token's rows (ascending sorted row: an expert appears once per token) and each
// row's h blocks (block order) of part_c, taken once every h block's owner is done with the
// 256-column group of cb. 224 threads (the consumer warps and the epilogue warp): thread
// (grp, c4) sums terms grp, grp + 14, ... of four columns; the 14 partial sums are then added
// in group order. Units first, first + stride, ...
__device__ void owner_reduce(const Params& p, volatile int* flags, float* red, const int* s_tok,
                             int tid, int first, int stride, int owners, int cb_per_group) {
    constexpr int kGroups = 14;
    const int c4 = tid & 15, grp = tid >> 4;
    const int terms = p.k * p.nbh;
    float4* red4 = reinterpret_cast<float4*>(red);
    int* rows = reinterpret_cast<int*>(red4 + kGroups * 16);  // the token's sorted rows
    for (int u = first; u < p.nbd * p.T; u += stride) {
        const int cb = u / p.T, t = u - cb * p.T;
        // every warp of the block is done with its own items (the epilogue warp with the last
        // hand-over in this buffer) and with the previous unit's sums
        asm volatile("bar.sync 1, 224;" ::: "memory");
        if (tid < 32) {
            if (tid == 0) {
                const uint64_t t0 = globaltimer_ns();
                while (ld_acquire(p.cnt_c + cb / cb_per_group) < owners) {
                    if (flags[0] || globaltimer_ns() - t0 > kWaitLimitNs) {
                        set_status(p.status, MOE_ERR_TIMEOUT);
                        flags[0] = 1;
                        break;
                    }
                }
            }
            int n = 0;
            for (int r0 = 0; r0 < p.R; r0 += 32) {
                const bool mine = r0 + tid < p.R && s_tok[r0 + tid] == t;
                const unsigned m = __ballot_sync(0xFFFFFFFFu, mine);
                if (mine) rows[n + __popc(m & ((1u << tid) - 1u))] = r0 + tid;
                n += __popc(m);
            }
        }
        asm volatile("bar.sync 1, 224;" ::: "memory");
        if (flags[0]) return;
        const int col = cb * 64 + 4 * c4;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (col < p.d) {
            for (int m0 = grp; m0 < terms; m0 += 8 * kGroups) {
                float4 v[8];
#pragma unroll
                for (int x = 0; x < 8; ++x) {
                    const int m = m0 + x * kGroups;
                    v[x] = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (m < terms) {
                        const int j = m / p.nbh, jb = m - j * p.nbh;
                        v[x] = __ldcg(reinterpret_cast<const float4*>(
                            p.part_c + ((size_t)jb * p.R + rows[j]) * p.d + col));
                    }
                }
#pragma unroll
                for (int x = 0; x < 8; ++x) {
                    acc.x += v[x].x;
                    acc.y += v[x].y;
                    acc.z += v[x].z;
                    acc.w += v[x].w;
                }
            }
        }
        red4[grp * 16 + c4] = acc;
        asm volatile("bar.sync 1, 224;" ::: "memory");
        if (tid < 16 && col < p.d) {
            float4 s4 = red4[c4];
            for (int g = 1; g < kGroups; ++g) {
                const float4 v = red4[g * 16 + c4];
                s4.x += v.x;
                s4.y += v.y;
                s4.z += v.z;
                s4.w += v.w;
            }
            __nv_bfloat162 lo = __floats2bfloat162_rn(s4.x, s4.y);
            __nv_bfloat162 hi = __floats2bfloat162_rn(s4.z, s4.w);
            uint2 packed;
            packed.x = *reinterpret_cast<uint32_t*>(&lo);
            packed.y = *reinterpret_cast<uint32_t*>(&hi);
            *reinterpret_cast<uint2*>(p.out + (size_t)t * p.d + col) = packed;
        }
        asm volatile("bar.sync 1, 224;" ::: "memory");
    }
}

// ================= epilogue side (one warp) =================

// h of group g (rows of expert q at row0, h block jb) from the partials of its contributors,
// summed in block order: per output of this lane, the loads of up to 8 contributors are issued
// together before any of them is added.
__device__ void epi_finish_h(const Ctx& c, const Params& p, int row0, int tq, int jb, int g,
                             int b_first, int b_last) {
    constexpr int kBatch = 8;
    const int n = tq * 64;
    for (int o = c.lane; o < n; o += 32) {
        const int t = o >> 6, col = o & 63;
        float gs = 0.0f, us = 0.0f;
        for (int b0 = b_first; b0 <= b_last; b0 += kBatch) {
            float gv[kBatch], uv[kBatch];
#pragma unroll
            for (int j = 0; j < kBatch; ++j) {
                const int b = b0 + j;
                gv[j] = uv[j] = 0.0f;
                if (b <= b_last && !range_empty(c.nA, b, c.GA)) {
                    const float* src =
                        p.part_a + ((size_t)(b + g + c.slot_off) * p.T + t) * 128 + col;
                    gv[j] = __ldcg(src);
                    uv[j] = __ldcg(src + 64);
                }
            }
#pragma unroll
            for (int j = 0; j < kBatch; ++j) {
                gs += gv[j];
                us += uv[j];
            }
        }
        if (p.mx)
            store_h_mx(p, c, row0 + t, jb * 64 + col, gs, us, jb * 64 + col < p.I);
        else if (jb * 64 + col < p.I)
            store_h(p, c, row0 + t, jb * 64 + col, gs, us);
    }
}

// gate_up group (q, jb) = g: take the consumers' dumps, store h (whole group) or this block's
// partial, and flag h once stored.
template <int NTILE>
__device__ void epi_a(Ctx& c, const Params& p, int q, int jb, int g, int b_first, int b_last) {
    const int row0 = c.s_off[q], tq = c.s_tq[q];
    const bool whole = b_first == b_last;
    float* part = p.part_a + (size_t)(blockIdx.x + g + c.slot_off) * p.T * 128;
#pragma unroll
    for (int pass = 0; pass < NTILE; ++pass) {
        if (pass * kPass < tq) {
            epi_take(c, p);
            const int nr = min(kPass, tq - pass * kPass);
            for (int o = c.lane; o < nr * (whole ? 64 : 128); o += 32) {
                const int t = whole ? (o >> 6) : (o >> 7), col = whole ? (o & 63) : (o & 127);
                float v = 0.0f, uu = 0.0f;
#pragma unroll
                for (int w = 0; w < kConsumerWarps; ++w) {
                    const float* rr = c.red + (w * kPass + t) * kStrideA + col;
                    v += rr[0];
                    if (whole) uu += rr[64];
                }
                if (whole) {
                    if (p.mx) {
                        const uint32_t cs = store_h_mx(p, c, row0 + pass * kPass + t,
                                                       jb * 64 + col, v, uu, jb * 64 + col < p.I);
                        if (c.owner) {
                            uint8_t* hb = reinterpret_cast<uint8_t*>(c.h_s);
                            const int r = pass * kPass + t;
                            hb[r * 64 + col] = (uint8_t)(cs & 0xFFu);
                            if ((col & 31) == 0) hb[kMxHsScales + r * 2 + (col >> 5)] = (uint8_t)(cs >> 8);
                        }
                    } else {
                        const __nv_bfloat16 hv =
                            jb * 64 + col < p.I
                                ? store_h(p, c, row0 + pass * kPass + t, jb * 64 + col, v, uu)
                                : __float2bfloat16_rn(0.0f);
                        if (c.owner) c.h_s[(pass * kPass + t) * 64 + col] = hv;
                    }
                } else {
                    __stcg(part + (size_t)(pass * kPass + t) * 128 + col, v);
                }
            }
            epi_give(c);
        }
    }
    if (c.owner) {  // the down partials of this h block are computed in this block
        __syncwarp();
        if (c.lane == 0) mbar_arrive(c.h_full);
        return;
    }
    bool stored = whole;
    if (!whole && epi_arrive_last(c, p.cnt_a + g, contributors(c.nA, c.GA, b_first, b_last))) {
        epi_finish_h(c, p, row0, tq, jb, g, b_first, b_last);
        stored = true;
    }
    if (stored) {
        __syncwarp();  // every h store of this warp is issued
        if (c.lane == 0)
            asm volatile("st.release.gpu.global.s32 [%0], 1;" ::"l"(p.hflag + g) : "memory");
    }
}

// Down sub-group of expert q: take the consumers' dumps and add weight * y of the expert's
// rows into the per-token accumulator (the combine; an expert appears once per token).
template <int NTILE>
__device__ void epi_b(Ctx& c, const Params& p, int q) {
    const int row0 = c.s_off[q], tq = c.s_tq[q];
#pragma unroll
    for (int pass = 0; pass < NTILE; ++pass) {
        if (pass * kPass < tq) {
            epi_take(c, p);
            const int nr = min(kPass, tq - pass * kPass);
            for (int o = c.lane; o < nr * 64; o += 32) {
                const int t = o >> 6, col = o & 63;
                float y = 0.0f;
#pragma unroll
                for (int w = 0; w < kConsumerWarps; ++w) y += c.red[(w * kPass + t) * kStrideB + col];
                const int row = row0 + pass * kPass + t;
                const float wgt = p.scale_input ? 1.0f : c.s_w[row];
                c.outacc[c.s_tok[row] * 64 + col] += wgt * y;
            }
            epi_give(c);
        }
    }
}

// Down items of wave w: experts [q_lo, q_hi), ordered (c, q, kc), perC per output block.
struct WaveB {
    int q_lo, perC, n;
};
__device__ __forceinline__ WaveB wave_b(const Ctx& c, const Params& p, int w) {
    WaveB v;
    v.q_lo = range_lo(c.nq, w, c.W);
    v.perC = (range_lo(c.nq, w + 1, c.W) - v.q_lo) * p.nkb;
    v.n = p.nbd * v.perC;
    return v;
}

// End of output block cb in this block's range of the current wave: write out (when this is
// the block's only contributor over all waves) or leave the per-token partial; the last
// contributor sums them, waves in order and blocks in order within a wave. Clears the
// accumulator.
__device__ void epi_flush(Ctx& c, const Params& p, int cb) {
    const int dc0 = cb * 64, n = p.T * 64;
    int total = 0;
    for (int w = 0; w < c.W; ++w) {
        const WaveB v = wave_b(c, p, w);
        total += contributors(v.n, c.GB, block_of(v.n, cb * v.perC, c.GB),
                              block_of(v.n, (cb + 1) * v.perC - 1, c.GB));
    }
    __syncwarp();
    if (total == 1) {
        for (int o = c.lane; o < n; o += 32) {
            const int t = o >> 6, col = o & 63;
            if (dc0 + col < p.d)
                p.out[(size_t)t * p.d + dc0 + col] = __float2bfloat16_rn(c.outacc[o]);
            c.outacc[o] = 0.0f;
        }
    } else {
        float* part = p.part_b + (size_t)(blockIdx.x - c.B0 + cb + c.slot_off) * n;
        for (int o = c.lane; o < n; o += 32) {
            __stcg(part + o, c.outacc[o]);
            c.outacc[o] = 0.0f;
        }
        if (epi_arrive_last(c, p.cnt_b + cb, total)) {
            constexpr int kPer = kOutFloats / 32;
            float acc[kPer];
#pragma unroll
            for (int i = 0; i < kPer; ++i) acc[i] = 0.0f;
            for (int w = 0; w < c.W; ++w) {
                const WaveB v = wave_b(c, p, w);
                const int bf = block_of(v.n, cb * v.perC, c.GB);
                const int bl = block_of(v.n, (cb + 1) * v.perC - 1, c.GB);
                for (int b = bf; b <= bl; ++b) {
                    if (range_empty(v.n, b, c.GB)) continue;
                    const float* base = p.part_b + (size_t)(b + cb + w * (c.GB + p.nbd)) * n;
#pragma unroll
                    for (int i = 0; i < kPer; ++i) {
                        const int o = c.lane + 32 * i;
                        if (o < n) acc[i] += __ldcg(base + o);
                    }
                }
            }
#pragma unroll
            for (int i = 0; i < kPer; ++i) {
                const int o = c.lane + 32 * i;
                if (o < n && dc0 + (o & 63) < p.d)
                    p.out[(size_t)(o >> 6) * p.d + dc0 + (o & 63)] = __float2bfloat16_rn(acc[i]);
            }
        }
    }
    __syncwarp();
}

template <int N>
struct NtTag {
    static constexpr int value = N;
};

// Run a group with one MMA n-tile per 8 of its rows (SMALL: at most 8 tokens, so one n-tile
// always and only that form is compiled).
template <bool SMALL, typename F>
__device__ __forceinline__ void by_rows(int tq, F&& f) {
    if constexpr (SMALL) {
        f(NtTag<1>{});
    } else {
        if (tq <= kPass)
            f(NtTag<1>{});
        else
            f(NtTag<2>{});
    }
}

// OWNER: the owner layout; SMALL: at most 8 tokens. Both are chosen on the host from the sizes
// alone, so that each instantiation holds only the code its batches run.
template <bool MX, bool OWNER, bool SMALL>
__global__ void __launch_bounds__(kThreads, 1)
decode_fused_kernel(const __grid_constant__ CUtensorMap tmGU,
                    const __grid_constant__ CUtensorMap tmD,
                    const __grid_constant__ CUtensorMap tmO, Params p, int vpl) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    int* s_eq = reinterpret_cast<int*>(smem + kOffLists);
    int* s_off = s_eq + kMaxE;
    int* s_tq = s_off + kMaxE;
    int* s_tok = s_tq + kMaxE;
    float* s_w = reinterpret_cast<float*>(s_tok + kDecodeFusedMaxRows);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kOffBars);
    uint64_t* empty = full + kStages;
    uint64_t* red_full = empty + kStages;
    uint64_t* red_empty = red_full + 1;
    uint64_t* h_full = red_empty + 1;  // [2]: one per h buffer (owner layout)
    volatile int* flags = reinterpret_cast<volatile int*>(h_full + 2);
    // flags: [0] a wait timed out (every bounded wait gives up at once after that; the status
    // word says so and the results are void), [2] number of touched experts.

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    griddep_wait();

    // ---- router top-k and dispatch indices, in every block (scratch in the stage buffers,
    // which no copy uses yet); the set-up below runs beside the routing.
    const int R = p.R, E = p.E;
    const DecodeRouteIO rio{p.logits, p.T, E, p.k, R, p.score_fn, p.renorm, p.topk_ids,
                            p.topk_w, p.counts, p.offsets, p.s2p, p.p2s};
    DecodeRouteSmem rsm;
    rsm.eq = s_eq;
    rsm.tq = s_tq;
    rsm.offq = s_off;
    rsm.tok = s_tok;
    rsm.wrow = s_w;
    rsm.pos = nullptr;
    rsm.nq = flags + 2;
    decode_route_scratch(rsm, smem);
    decode_route_tokens<kWarps>(rio, rsm, vpl);
    if (warp == kEpilogueWarp && lane == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        mbar_init(red_full, kConsumerWarps);
        mbar_init(red_empty, 1);
        mbar_init(&h_full[0], 1);
        mbar_init(&h_full[1], 1);
        fence_barrier_init();
        for (int f = 0; f < 4; ++f) flags[f] = 0;
    }
    if (!MX && warp == kProducerWarp && lane == 0) {  // MX items are plain bulk copies
        tma_prefetch_desc(&tmGU);
        tma_prefetch_desc(&tmD);
        tma_prefetch_desc(&tmO);
    }
    float* outacc = reinterpret_cast<float*>(smem + kOffOut);
    for (int i = threadIdx.x; i < kOutFloats; i += blockDim.x) outacc[i] = 0.0f;
    __syncthreads();
    const int nq = decode_dispatch(rio, rsm, blockIdx.x == 0);
    // the stage buffers are free for the copies again

    // Schedule. The touched experts form W waves; every block takes its stream-K share of the
    // gate_up items of wave 0, then of wave 1, ..., then of the down items of wave 0, 1, ...
    // The h of wave 0 is finished while the later waves' gate_up items stream, so the down
    // items rarely wait for it.
    const int G = gridDim.x, b = blockIdx.x;
    const int W = nq < kDecodeWaves ? nq : kDecodeWaves;
    // Partition. Stream-K: both lists over all G blocks. When there are fewer h blocks than
    // SMs and the down items, spread over the remaining blocks, are not much more than one h
    // block's worth of bytes each, blocks [0, ngA) each take one whole h block (no partial
    // sums, h flagged as soon as it is stored) and blocks [ngA, G) take the down items,
    // prefetching them while the gate_up items stream.
    const int ngA = nq * p.nbh;
    // Owner layout (bf16 weights, one wave): block b owns whole h blocks [ob_lo, ob_hi): h
    // block b alone while there are fewer h blocks than blocks, else an equal contiguous share.
    // For each owned h block it streams the gate_up items and then the down weight rows of
    // those 64 h columns for all output columns (n4 items of four 64-column boxes), and
    // multiplies them by h kept in its own shared memory. The weighted partials are then summed
    // per (output block, token) by the blocks past the owners (fewer h blocks than blocks) or by
    // every block once its own h blocks are done. No h crosses SMs.
    // (Taken while the final sums are at most two (output block, token) units per block; past
    // that, as at T = 16 on the decode shape, the stream-K layout measured faster. The host
    // picks the instantiation: see launch_decode_fused.)
    constexpr bool owner = OWNER;
    const int cb_per_item = MX ? kMxOwnCb : 4;  // output column blocks per owner down item
    const int n4 = (p.nbd + cb_per_item - 1) / cb_per_item;
    const int ob_lo = ngA <= G ? min(b, ngA) : (int)((long long)ngA * b / G);
    const int ob_hi = ngA <= G ? min(b + 1, ngA) : (int)((long long)ngA * (b + 1) / G);
    const bool whole_groups = W == 1 && ngA < G &&
                              (long long)p.nbd * nq * p.nkb * 4 <= 5ll * p.nka * (G - ngA);
    const int GA = whole_groups ? ngA : G;
    const int B0 = whole_groups ? ngA : 0, GB = G - B0;
    const int ba = b < GA ? b : GA;            // gate_up range index (GA: empty)
    const int bb = b >= B0 ? b - B0 : GB;      // down range index (GB: empty)
    auto wave_a = [&](int w, int& q_lo, int& n) {
        q_lo = range_lo(nq, w, W);
        n = (range_lo(nq, w + 1, W) - q_lo) * p.nbh * p.nka;
    };

    if (warp == kProducerWarp) {
        // ============ producer: the block's items in schedule order ============
        if (lane == 0) {
            const uint32_t stage0 = smem_u32(smem);
            // the weights are read once: evict-first, so x, h and the partial sums stay in L2
            const uint64_t pol = l2_evict_first();
            int i = 0;
            bool ok = true;
            auto next_stage = [&](uint32_t& dst, uint64_t*& bar, uint32_t bytes) {
                const int st = i % kStages;
                const uint32_t ph = (uint32_t)(i / kStages) & 1u;
                if (!mbar_wait(&empty[st], ph ^ 1u, flags, kWaitLimitNs)) {
                    set_status(p.status, MOE_ERR_TIMEOUT);
                    flags[0] = 1;
                    return false;
                }
                mbar_arrive_expect_tx(&full[st], bytes);
                dst = stage0 + (uint32_t)st * kStageBytes;
                bar = &full[st];
                ++i;
                return true;
            };
            if (owner) {
                // per owned h block j: its gate_up items, and the down items of h block j - 1
                // behind them, so the ring streams while the epilogue warp finishes h
                for (int j = 0; ok && j <= ob_hi - ob_lo; ++j) {
                    if (j < ob_hi - ob_lo) {
                        const int g = ob_lo + j;
                        const int q = g / p.nbh, jb = g % p.nbh, e = s_eq[q];
                        for (int kc = 0; ok && kc < p.nka; ++kc) {
                            uint32_t dst;
                            uint64_t* bar;
                            if (MX) {
                                const int kb0 = kc * p.kba, nk = min(p.kba, p.kbd - kb0);
                                const size_t bg = ((size_t)e * p.gu_nb + jb) * p.kbd + kb0;
                                const size_t bu = ((size_t)e * p.gu_nb + p.nbh + jb) * p.kbd + kb0;
                                if (!(ok = next_stage(dst, bar, (uint32_t)nk * 2 * (1024 + 64))))
                                    break;
                                bulk_load(dst, p.mx_gu + bg * 1024, nk * 1024, bar, pol);
                                bulk_load(dst + kMxUpCodes, p.mx_gu + bu * 1024, nk * 1024, bar, pol);
                                bulk_load(dst + kMxScales, p.mx_gu + p.mx_gu_scales + bg * 64,
                                          nk * 64, bar, pol);
                                bulk_load(dst + kMxUpScales, p.mx_gu + p.mx_gu_scales + bu * 64,
                                          nk * 64, bar, pol);
                                continue;
                            }
                            if (!(ok = next_stage(dst, bar, kStageBytes))) break;
                            if (p.packed) {
                                tma_load_3d_hint(dst, &tmGU, bar, 0, kc * kKcA,
                                                 e * p.gu_nb + jb, pol);
                                tma_load_3d_hint(dst + kBoxBytesA, &tmGU, bar, 0, kc * kKcA,
                                                 e * p.gu_nb + p.nbh + jb, pol);
                            } else {
                                tma_load_3d_hint(dst, &tmGU, bar, 64 * jb, kc * kKcA, e, pol);
                                tma_load_3d_hint(dst + kBoxBytesA, &tmGU, bar, p.I + 64 * jb,
                                                 kc * kKcA, e, pol);
                            }
                        }
                    }
                    if (j >= 1) {
                        // the down weight rows of h block j - 1: output columns 256 g4 ..
                        const int g = ob_lo + j - 1;
                        const int q = g / p.nbh, jb = g % p.nbh, e = s_eq[q];
                        for (int g4 = 0; ok && g4 < n4; ++g4) {
                            uint32_t dst;
                            uint64_t* bar;
                            if (MX) {
                                // K blocks 2 jb, 2 jb + 1 (those below I) of 14 column blocks
                                const int cb0 = g4 * kMxOwnCb, ncb = min(kMxOwnCb, p.nbd - cb0);
                                const int nkb = min(2, p.kbi - 2 * jb);
                                if (!(ok = next_stage(dst, bar,
                                                      (uint32_t)(ncb * nkb * (1024 + 64)))))
                                    break;
                                for (int cbl = 0; cbl < ncb; ++cbl) {
                                    const size_t bd =
                                        ((size_t)e * p.dn_nb + cb0 + cbl) * p.kbi + 2 * jb;
                                    bulk_load(dst + (uint32_t)cbl * 2048u, p.mx_dn + bd * 1024,
                                              nkb * 1024, bar, pol);
                                    bulk_load(dst + kMxOwnScales + (uint32_t)cbl * 128u,
                                              p.mx_dn + p.mx_dn_scales + bd * 64, nkb * 64, bar,
                                              pol);
                                }
                                continue;
                            }
                            if (!(ok = next_stage(dst, bar, kStageBytes))) break;
                            if (p.packed) {
                                tma_load_3d_hint(dst, &tmO, bar, 0, 64 * jb,
                                                 e * p.dn_nb + 4 * g4, pol);
                            } else {
                                for (int x = 0; x < 4; ++x)
                                    tma_load_3d_hint(dst + 8192u * x, &tmO, bar,
                                                     64 * (4 * g4 + x), 64 * jb, e, pol);
                            }
                        }
                    }
                }
            }
            for (int w = 0; !owner && ok && w < W; ++w) {
                int q_lo, n;
                wave_a(w, q_lo, n);
                const int lo = ba < GA ? range_lo(n, ba, GA) : 0;
                const int hi = ba < GA ? range_lo(n, ba + 1, GA) : 0;
                for (int u = lo; ok && u < hi; ++u) {
                    uint32_t dst;
                    uint64_t* bar;
                    const int g = q_lo * p.nbh + u / p.nka, kc = u % p.nka;
                    const int q = g / p.nbh, jb = g % p.nbh, e = s_eq[q];
                    if (MX) {
                        // K blocks [15 kc, ...) of the gate and up column blocks: runs of 1 KB
                        // code blocks and 64 B scale blocks
                        const int kb0 = kc * p.kba, nk = min(p.kba, p.kbd - kb0);
                        const size_t bg = ((size_t)e * p.gu_nb + jb) * p.kbd + kb0;
                        const size_t bu = ((size_t)e * p.gu_nb + p.nbh + jb) * p.kbd + kb0;
                        if (!(ok = next_stage(dst, bar, (uint32_t)nk * 2 * (1024 + 64)))) break;
                        bulk_load(dst, p.mx_gu + bg * 1024, nk * 1024, bar, pol);
                        bulk_load(dst + kMxUpCodes, p.mx_gu + bu * 1024, nk * 1024, bar, pol);
                        bulk_load(dst + kMxScales, p.mx_gu + p.mx_gu_scales + bg * 64, nk * 64,
                                  bar, pol);
                        bulk_load(dst + kMxUpScales, p.mx_gu + p.mx_gu_scales + bu * 64, nk * 64,
                                  bar, pol);
                        continue;
                    }
                    if (!(ok = next_stage(dst, bar, kStageBytes))) break;
                    if (p.packed) {
                        tma_load_3d_hint(dst, &tmGU, bar, 0, kc * kKcA, e * p.gu_nb + jb, pol);
                        tma_load_3d_hint(dst + kBoxBytesA, &tmGU, bar, 0, kc * kKcA,
                                    e * p.gu_nb + p.nbh + jb, pol);
                    } else {
                        tma_load_3d_hint(dst, &tmGU, bar, 64 * jb, kc * kKcA, e, pol);
                        tma_load_3d_hint(dst + kBoxBytesA, &tmGU, bar, p.I + 64 * jb, kc * kKcA, e, pol);
                    }
                }
            }
            for (int w = 0; !owner && ok && w < W; ++w) {
                const int q_lo = range_lo(nq, w, W);
                const int perC = (range_lo(nq, w + 1, W) - q_lo) * p.nkb, n = p.nbd * perC;
                const int lo = bb < GB ? range_lo(n, bb, GB) : 0;
                const int hi = bb < GB ? range_lo(n, bb + 1, GB) : 0;
                for (int u = lo; ok && u < hi; ++u) {
                    uint32_t dst;
                    uint64_t* bar;
                    const int cb = u / perC, rem = u % perC;
                    const int e = s_eq[q_lo + rem / p.nkb], kc = rem % p.nkb;
                    if (MX) {
                        const int kb0 = kc * kMxKbB, nk = min(kMxKbB, p.kbi - kb0);
                        const size_t bd = ((size_t)e * p.dn_nb + cb) * p.kbi + kb0;
                        if (!(ok = next_stage(dst, bar, (uint32_t)nk * (1024 + 64)))) break;
                        bulk_load(dst, p.mx_dn + bd * 1024, nk * 1024, bar, pol);
                        bulk_load(dst + kMxScales, p.mx_dn + p.mx_dn_scales + bd * 64, nk * 64,
                                  bar, pol);
                        continue;
                    }
                    if (!(ok = next_stage(dst, bar, kStageBytes))) break;
                    if (p.packed)
                        tma_load_3d_hint(dst, &tmD, bar, 0, kc * kKcB, e * p.dn_nb + cb, pol);
                    else
                        tma_load_3d_hint(dst, &tmD, bar, 64 * cb, kc * kKcB, e, pol);
                }
            }
            // leave no copy in flight: the last (up to) kStages issued items must have landed
            for (int j = i > kStages ? i - kStages : 0; j < i; ++j)
                mbar_wait(&full[j % kStages], (uint32_t)(j / kStages) & 1u, nullptr,
                          kWaitLimitNs);
        }
        return;
    }

    Ctx c;
    c.stage0 = smem_u32(smem);
    c.red = reinterpret_cast<float*>(smem + kOffRed);
    c.outacc = outacc;
    c.s_off = s_off;
    c.s_tq = s_tq;
    c.s_tok = s_tok;
    c.s_w = s_w;
    c.full = full;
    c.empty = empty;
    c.red_full = red_full;
    c.red_empty = red_empty;
    c.flags = flags;
    c.warp = warp;
    c.lane = lane;
    c.G = G;
    c.GA = GA;
    c.B0 = B0;
    c.GB = GB;
    c.W = W;
    c.nq = nq;
    c.ready_q = -1;
    c.ready_mask = 0;
    c.dumps = 0;
    c.owner = owner;
    // owner layout: two h buffers in the (then unused) combine accumulator
    __nv_bfloat16* const h_buf = reinterpret_cast<__nv_bfloat16*>(outacc);
    c.h_s = h_buf;
    c.h_full = h_full;
    const bool epilogue = warp == kEpilogueWarp;

    // consumers (warp w: the items of stage w) and the epilogue warp walk the same groups
    int i0 = 0;  // block-local index of the next item
    if constexpr (OWNER) {
        // the producer's order: gate_up of h block j (h into buffer j & 1), then the down
        // items of h block j - 1 (h from buffer (j - 1) & 1, its barrier's use (j - 1) >> 1)
        const int n_own = ob_hi - ob_lo;
        for (int j = 0; j <= n_own; ++j) {
            if (j < n_own) {
                const int g = ob_lo + j, q = g / p.nbh, jb = g % p.nbh;
                c.h_s = h_buf + (j & 1) * kDecodeFusedMaxTokens * 64;
                c.h_full = &h_full[j & 1];
                if (epilogue)
                    by_rows<SMALL>(s_tq[q], [&](auto tag) {
                        epi_a<decltype(tag)::value>(c, p, q, jb, g, b, b);
                    });
                else
                    by_rows<SMALL>(s_tq[q], [&](auto tag) {
                        group_a<decltype(tag)::value, MX>(c, p, q, i0, 0, p.nka);
                    });
                i0 += p.nka;
            }
            if (j >= 1) {
                const int g = ob_lo + j - 1, q = g / p.nbh, jb = g % p.nbh;
                c.h_s = h_buf + ((j - 1) & 1) * kDecodeFusedMaxTokens * 64;
                c.h_full = &h_full[(j - 1) & 1];
                if (!epilogue)
                    by_rows<SMALL>(s_tq[q], [&](auto tag) {
                        if (MX)
                            owner_down_mx<decltype(tag)::value>(c, p, q, jb, i0, n4,
                                                                (uint32_t)((j - 1) >> 1) & 1u);
                        else
                            owner_down<decltype(tag)::value>(c, p, q, jb, i0, n4,
                                                             (uint32_t)((j - 1) >> 1) & 1u);
                    });
                i0 += n4;
            }
        }
        const int tid = (warp < kProducerWarp ? warp : warp - 1) * 32 + lane;
        if (ngA < G) {
            if (b >= ngA)
                owner_reduce(p, flags, c.red, s_tok, tid, b - ngA, G - ngA, ngA, cb_per_item);
        } else {
            owner_reduce(p, flags, c.red, s_tok, tid, b, G, ngA, cb_per_item);
        }
    } else {
        for (int w = 0; w < W; ++w) {
            int q_lo, n;
            wave_a(w, q_lo, n);
            c.nA = n;
            c.slot_off = w * G;
            const int hi = ba < GA ? range_lo(n, ba + 1, GA) : 0;
            for (int u = ba < GA ? range_lo(n, ba, GA) : 0; u < hi;) {
                const int gl = u / p.nka, kc0 = u % p.nka;  // group within the wave, K chunk
                const int kc1 = min(p.nka, kc0 + (hi - u));
                const int g = q_lo * p.nbh + gl, q = g / p.nbh, jb = g % p.nbh;
                if (epilogue) {
                    const int bf = block_of(n, gl * p.nka, GA);
                    const int bl = block_of(n, (gl + 1) * p.nka - 1, GA);
                    by_rows<SMALL>(s_tq[q],
                            [&](auto tag) { epi_a<decltype(tag)::value>(c, p, q, jb, g, bf, bl); });
                } else {
                    by_rows<SMALL>(s_tq[q], [&](auto tag) {
                        group_a<decltype(tag)::value, MX>(c, p, q, i0, kc0, kc1);
                    });
                }
                u += kc1 - kc0;
                i0 += kc1 - kc0;
            }
        }
        for (int w = 0; w < W; ++w) {
            const WaveB v = wave_b(c, p, w);
            c.slot_off = w * (GB + p.nbd);
            const int hi = bb < GB ? range_lo(v.n, bb + 1, GB) : 0;
            for (int u = bb < GB ? range_lo(v.n, bb, GB) : 0; u < hi;) {
                const int cb = u / v.perC;
                const int c_end = min(hi, (cb + 1) * v.perC);
                while (u < c_end) {
                    const int rem = u % v.perC, q = v.q_lo + rem / p.nkb, kc0 = rem % p.nkb;
                    const int kc1 = min(p.nkb, kc0 + (c_end - u));
                    if (epilogue)
                        by_rows<SMALL>(s_tq[q], [&](auto tag) { epi_b<decltype(tag)::value>(c, p, q); });
                    else
                        by_rows<SMALL>(s_tq[q], [&](auto tag) {
                            group_b<decltype(tag)::value, MX>(c, p, q, i0, kc0, kc1);
                        });
                    u += kc1 - kc0;
                    i0 += kc1 - kc0;
                }
                if (epilogue) epi_flush(c, p, cb);
            }
        }
    }
}

}  // namespace

// MX gate_up items: 32-row K blocks per item. At T = 1 fewer, larger items measured faster; from
// T = 2 up, 11 (more items to share among the consumer warps).
static int mx_kba(int T) { return T == 1 ? kMxKbA : 11; }

bool decode_fused_applies(moe_dtype dt, int T, int k, int Is) {
    return dt == MOE_BF16 && Is == 0 && T >= 1 && T <= kDecodeFusedMaxTokens &&
           T * k <= kDecodeFusedMaxRows;
}

DecodeFusedLayout decode_fused_layout(int T, int d, int k, int I, bool mx) {
    DecodeFusedLayout L;
    const size_t R = (size_t)T * k;
    L.nbh = (I + 63) / 64;
    L.nbd = (d + 63) / 64;
    if (mx) {  // items of up to 15 (gate_up) / 30 (down) 32-row K blocks
        L.nka = ((d + 31) / 32 + mx_kba(T) - 1) / mx_kba(T);
        L.nkb = ((I + 31) / 32 + kMxKbB - 1) / kMxKbB;
    } else {
        L.nka = (d + kKcA - 1) / kKcA;
        L.nkb = (I + kKcB - 1) / kKcB;
    }
    auto up = [](size_t v) { return (v + 255) / 256 * 256; };
    L.counter_bytes = up((2 * R * L.nbh + L.nbd + (L.nbd + 3) / 4) * 4);
    // partial slots: contributor block b of group g writes slot b + g (unique: a block's groups
    // are consecutive and the next block starts at or after its last one)
    // (gate_up slot b + g + w G and down slot b + c + w (G + nbd) for wave w: unique across
    // waves too, as the gate_up groups of later waves have larger g)
    L.part_a = 0;
    L.part_b = up(((size_t)kDecodeWaves * kDecodeFusedMaxGrid + R * L.nbh) * T * 128 * 4);
    L.part_bytes = L.part_b + up((size_t)kDecodeWaves * (kDecodeFusedMaxGrid + L.nbd) * T *
                                 64 * 4);
    // owner layout: the down partials [nbh][R][d] fp32 (only where the layout can be taken on
    // any grid: at most two (output block, token) summing units per block of the largest grid)
    L.part_c = 0;
    if (L.nbh < kDecodeFusedMaxGrid && (long long)L.nbd * T <= 2ll * kDecodeFusedMaxGrid) {
        L.part_c = L.part_bytes;
        L.part_bytes += up((size_t)L.nbh * R * d * 4);
    }
    return L;
}

cudaError_t launch_decode_fused(const DecodeFusedArgs& a, cudaStream_t s) {
    const DecodeFusedLayout L = decode_fused_layout(a.T, a.d, a.k, a.I, a.mx);
    // one block per SM (its shared memory allows no more), all resident: cooperative launch.
    // It is the first kernel of the layer, so it follows the caller's work in stream order.
    int grid = device_sm_count();
    if (grid > kDecodeFusedMaxGrid) grid = kDecodeFusedMaxGrid;
    // the owner layout while its final sums come to at most two (output block, token) units
    // per block (and its partial region exists)
    const bool owner = L.part_c != 0 && (long long)L.nbd * a.T <= 2ll * grid;
    using Kern = void (*)(CUtensorMap, CUtensorMap, CUtensorMap, Params, int);
    static const Kern kKern[2][2][2] = {
        {{decode_fused_kernel<false, false, false>, decode_fused_kernel<false, false, true>},
         {decode_fused_kernel<false, true, false>, decode_fused_kernel<false, true, true>}},
        {{decode_fused_kernel<true, false, false>, decode_fused_kernel<true, false, true>},
         {decode_fused_kernel<true, true, false>, decode_fused_kernel<true, true, true>}}};
    const Kern kern = kKern[a.mx ? 1 : 0][owner ? 1 : 0][a.T <= kPass ? 1 : 0];
    {
        const cudaError_t e = ensure_max_dynamic_smem(kern, (int)kSmemBytes);
        if (e != cudaSuccess) return e;
    }
    const int R = a.T * a.k;
    CUtensorMap tmGU = {}, tmD = {}, tmO = {};  // MX: unused (items are plain bulk copies)
    const cuuint32_t box_a[3] = {64, kKcA, 1}, box_b[3] = {64, kKcB, 1};
    bool ok = true;
    if (a.mx) {
    } else if (a.packed) {
        const PackedGeom gg = packed_geom(kGateUp, a.d, a.I);
        const PackedGeom gd = packed_geom(kDown, a.I, a.d);
        const cuuint64_t gu_dims[3] = {64, (cuuint64_t)gg.kpad, (cuuint64_t)a.E * gg.nb};
        const cuuint64_t gu_str[2] = {128, (cuuint64_t)gg.kpad * 128};
        const cuuint64_t dn_dims[3] = {64, (cuuint64_t)gd.kpad, (cuuint64_t)a.E * gd.nb};
        const cuuint64_t dn_str[2] = {128, (cuuint64_t)gd.kpad * 128};
        // owner layout: 64 K rows of four consecutive 64-column blocks
        const cuuint32_t box_o[3] = {64, 64, 4};
        ok = encode_tensor_map_bf16(&tmGU, a.w_gate_up, 3, gu_dims, gu_str, box_a) &&
             encode_tensor_map_bf16(&tmD, a.w_down, 3, dn_dims, dn_str, box_b) &&
             encode_tensor_map_bf16(&tmO, a.w_down, 3, dn_dims, dn_str, box_o);
    } else {
        const cuuint64_t gu_dims[3] = {2 * (cuuint64_t)a.I, (cuuint64_t)a.d, (cuuint64_t)a.E};
        const cuuint64_t gu_str[2] = {4 * (cuuint64_t)a.I, 4 * (cuuint64_t)a.I * a.d};
        const cuuint64_t dn_dims[3] = {(cuuint64_t)a.d, (cuuint64_t)a.I, (cuuint64_t)a.E};
        const cuuint64_t dn_str[2] = {2 * (cuuint64_t)a.d, 2 * (cuuint64_t)a.d * a.I};
        const cuuint32_t box_o[3] = {64, 64, 1};  // owner layout: four loads per item
        ok = encode_tensor_map_bf16(&tmGU, a.w_gate_up, 3, gu_dims, gu_str, box_a) &&
             encode_tensor_map_bf16(&tmD, a.w_down, 3, dn_dims, dn_str, box_b) &&
             encode_tensor_map_bf16(&tmO, a.w_down, 3, dn_dims, dn_str, box_o);
    }
    if (!ok) return cudaErrorInvalidValue;

    uint8_t* parts = static_cast<uint8_t*>(a.partials);
    Params p;
    p.x = static_cast<const __nv_bfloat16*>(a.x);
    p.logits = a.logits;
    p.topk_ids = a.topk_ids;
    p.topk_w = a.topk_weights;
    p.counts = a.counts;
    p.offsets = a.offsets;
    p.s2p = a.sorted_to_slot;
    p.p2s = a.slot_to_sorted;
    p.h = static_cast<__nv_bfloat16*>(a.h);
    p.out = static_cast<__nv_bfloat16*>(a.out);
    p.cnt_a = a.counters;
    p.hflag = a.counters + (size_t)R * L.nbh;
    p.cnt_b = a.counters + (size_t)2 * R * L.nbh;
    p.cnt_c = p.cnt_b + L.nbd;
    p.part_c = L.part_c ? reinterpret_cast<float*>(parts + L.part_c) : nullptr;
    p.part_a = reinterpret_cast<float*>(parts + L.part_a);
    p.part_b = reinterpret_cast<float*>(parts + L.part_b);
    p.status = a.status;
    p.T = a.T;
    p.d = a.d;
    p.E = a.E;
    p.k = a.k;
    p.I = a.I;
    p.R = R;
    p.score_fn = a.score_fn;
    p.renorm = a.renorm ? 1 : 0;
    p.nbh = L.nbh;
    p.nka = L.nka;
    p.nbd = L.nbd;
    p.nkb = L.nkb;
    p.scale_input = a.scale_input ? 1 : 0;
    p.packed = a.packed ? 1 : 0;
    p.gu_nb = packed_geom(kGateUp, a.d, a.I).nb;
    p.dn_nb = packed_geom(kDown, a.I, a.d).nb;
    p.mx = a.mx ? 1 : 0;
    p.mx_gu = p.mx_dn = nullptr;
    p.mx_gu_scales = p.mx_dn_scales = 0;
    p.h_codes = p.h_scales = nullptr;
    p.kbd = (a.d + 31) / 32;
    p.kbi = (a.I + 31) / 32;
    p.kba = mx_kba(a.T);
    if (a.mx) {
        const MxGeom gg = mx_geom(true, a.d, a.I, a.E), gd = mx_geom(false, a.I, a.d, a.E);
        p.mx_gu = static_cast<const uint8_t*>(a.w_gate_up);
        p.mx_dn = static_cast<const uint8_t*>(a.w_down);
        p.mx_gu_scales = gg.scales_off;
        p.mx_dn_scales = gd.scales_off;
        p.gu_nb = gg.blocks.nb;
        p.dn_nb = gd.blocks.nb;
        p.h_codes = static_cast<uint8_t*>(a.h_codes);
        p.h_scales = static_cast<uint8_t*>(a.h_scales);
    }
    const int vpl = a.E <= 32 ? 1 : a.E <= 64 ? 2 : a.E <= 128 ? 4 : 8;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, tmGU, tmD, tmO, p, vpl);
}

}  // namespace rdg
