// One-kernel MX decode layer on the block-scaled tensor cores: router top-k, dispatch, gate_up +
// SwiGLU, down and the weighted combine for at most 16 tokens, with the experts' weights in the
// MX tensor-core layout (gemm_mx_tc.cu) multiplied by tcgen05.mma.kind::mxf8f6f4.block_scale.
//
// What it computes is the MX layer of moe_forward_mx_tc (Expert parallelism page, "Adding an
// implementation": every expert runs on the rows routed to it and the outputs are combined
// with the routing weights; the Mega MoE paragraph: 8-bit activations times 4-bit expert
// weights with block scales). x is rounded to MXFP8 (E4M3 codes, one E8M0 scale per 32
// elements) once per token, h = SiLU(s g) (s u) is rounded to MXFP8 per 32 h columns, and the
// tensor cores multiply those codes by the E2M1 weight codes, applying both scales themselves.
//
// Shape of the work. With at most 16 tokens every weight element meets at most 16 rows, so the
// layer is a stream of the touched experts' weights (a quarter of the bf16 bytes); what costs
// is keeping the memory pipes full and the dependent steps few. The MMAs take the weights as
// the M side (128 weight columns per instruction, E2M1 codes landed by TMA in the form of 16
// codes per 16 bytes that the tensor core reads 4-bit operands in) and the tokens as the N side:
// N = 16 columns, one per token of the batch, whether or not it was routed to the expert. A
// token's column never mixes with another's, so the rows routed to the expert are simply the
// columns read out, and one x tile and one set of x scales serve every expert: each block
// rounds x once into shared memory (16 rows x 128 bytes per 128-element K chunk, 128-byte
// swizzle) and copies x's scale atoms into tensor memory once.
//
// Owner layout. The touched experts' h blocks (128 h columns of one expert: 128 gate and 128
// up weight columns) are dealt to the blocks: h block b to block b while there are fewer h
// blocks than blocks, else equal contiguous shares. For each h block a block streams its
// gate_up weights (per 128-element K chunk: the gate box, the up box and their two scale
// atoms), then the down weight rows of those 128 h columns for every output column (two
// 128-column boxes per stage, with their atoms); the gate_up stages of h block j + 1 go ahead of
// the down stages of h block j, so the ring keeps streaming while h is finished. Warp roles:
//   warp 0     TMA producer: a 5-stage ring of 33 KB stages (two boxes, two scale atoms).
//   warp 1     allocates tensor memory; one lane copies each stage's scale atoms into it and
//              issues the MMAs (M = 128, N = 16, K = 32, four per box per 128-element chunk).
//   warps 2-5  epilogue, one per tensor-memory lane quarter (32 h or output columns each).
// Tensor memory (512 columns): down accumulators [0, 256) (16 columns per 128-column output
// block, for d <= 2048); gate and up accumulators [256, 320) (two buffers, so h block j + 1's
// MMAs run while the epilogue finishes h block j); x's scale atoms [320, 384); h's scale atoms
// [384, 392) (two buffers); the stages' weight scale atoms from 392.
// The epilogue reads the gate and up accumulators of an h block (a lane holds one h column for
// the 16 tokens), computes h in fp32, rounds each token's 32 columns of a warp to MXFP8 (the
// block maximum across the warp's lanes), and writes the codes into a 16 x 128-byte B tile in
// shared memory and the scales into an atom, from which the down MMAs read them. The down
// accumulators add up the h blocks of one expert that a block owns in a row (a "run"); at the
// end of a run the epilogue writes the routing-weighted sums of the expert's rows as fp32
// partials part[first h block of the run][sorted row][d] and, when the block is done, bumps
// a counter (release).
// Summing step. Once every owner has bumped the counter, unit (token t, 128 output columns) is
// the sum over t's slots (in slot order: an expert appears once per token) and each slot's
// row's runs (ascending h block) of the partials, rounded once to bf16; units are dealt to the
// blocks from the last one down, so blocks that own nothing take them first.
// Every sum runs in an order fixed by the sizes, so repeated calls give the same bits. The
// launch is cooperative (the summing step waits for other blocks), every wait is bounded
// (2 s; on expiry the kernel records MOE_ERR_TIMEOUT, drains its own copies and MMAs, frees
// tensor memory and returns), and the counter sits in the workspace head, cleared with the
// status word before the launch. For checks, the block that writes the dispatch indices also
// writes x's MXFP8 rows, and the owners h's, into the padded layout of the multi-kernel path.

#include "decode_route.cuh"
#include "mx_tc.cuh"

namespace rdg {
namespace {

constexpr int kThreads = 192;
constexpr int kWarps = kThreads / 32;
constexpr int kProducerWarp = 0;
constexpr int kMmaWarp = 1;
constexpr int kFirstEpiWarp = 2;  // warps 2..5: TMEM lane quarter = warp % 4
constexpr int kStages = 5;
constexpr int kN = 16;                      // the MMAs' N: token columns
constexpr int kBox = 128 * 128;             // one weight box in shared memory (16 bytes / 16 codes)
constexpr uint32_t kBoxTx = 128 * 128 / 2;  // the packed bytes it reads: its transaction bytes
constexpr int kStageBytes = 2 * kBox + 2 * kAtom;
constexpr int kMaxKc = 16;                  // d <= 2048: 128-element K chunks of x
constexpr int kMaxNob = 16;                 // d <= 2048: 128-column output blocks
constexpr int kTile = kN * 128;             // a 16-row x 128-byte B tile (x chunk or h block)
constexpr int kMaxNbh = 32;                 // I <= 4096: h blocks per expert
constexpr uint64_t kWaitLimitNs = 2000000000ull;

constexpr int kOffX = kStages * kStageBytes;
constexpr int kOffH = kOffX + kMaxKc * kTile;
constexpr int kOffXsf = kOffH + 2 * kTile;
constexpr int kOffHsf = kOffXsf + kMaxKc * kAtom;
constexpr int kOffLists = kOffHsf + 2 * kAtom;
constexpr int kListInts = 3 * kMaxE + 4 * kDecodeFusedMaxRows;
constexpr int kOffBars = kOffLists + kListInts * 4;
constexpr int kNumBars = 2 * kStages + 6 + 3;
constexpr int kSmemBytes = kOffBars + kNumBars * 8 + 32 + 1024;  // + alignment slack
static_assert(kStageBytes % 1024 == 0 && kOffX % 1024 == 0 && kOffH % 1024 == 0,
              "B tiles and weight boxes must start on 1024-byte boundaries (128-byte swizzle)");
static_assert(kSmemBytes <= 232448, "exceeds the 227 KB of shared memory a block may use");

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColDown = 0;
constexpr uint32_t kColGu = kColDown + 16 * kMaxNob;
constexpr uint32_t kColXsf = kColGu + 64;
constexpr uint32_t kColHsf = kColXsf + 4 * kMaxKc;
constexpr uint32_t kColWsf = kColHsf + 8;
static_assert(kColWsf + 8 * kStages <= kTmemCols, "tensor memory columns");

struct Params {
    const __nv_bfloat16* x;  // [T, d]
    const float* logits;     // [T, E]
    const uint8_t* gu_sf;    // gate_up weight scale atoms [E][2 nbh][KCd][512]
    const uint8_t* dn_sf;    // down weight scale atoms [E][nob][KCi][512]
    int32_t* topk_ids;
    float* topk_w;
    int32_t* counts;
    int32_t* offsets;
    int32_t* s2p;
    int32_t* p2s;
    uint8_t* xq;   // padded x rows: codes [Rp][d], atoms [Rp / 128][KCd][512]
    uint8_t* xsf;
    uint8_t* hq;   // padded h rows: codes [Rp][I], atoms [Rp / 128][KCi][512]
    uint8_t* hsf;
    float* part;   // [nbh][R][d]
    __nv_bfloat16* out;  // [T, d]
    int* done;     // owners done (zero at launch)
    int* status;
    int T, d, E, k, I, R, score_fn, renorm, scale_input;
    int KCd, KCi, nbh, nob;
};

struct Bars {
    uint64_t *full, *empty, *gu_full, *gu_empty, *h_full, *dn_full, *dn_empty, *drain;
};

// Block b's h blocks [lo, hi) of NH over G blocks.
__device__ __forceinline__ void owned_range(int NH, int G, int b, int* lo, int* hi) {
    if (NH <= G) {
        *lo = b;
        *hi = b < NH ? b + 1 : b;
    } else {
        *lo = b * NH / G;
        *hi = (b + 1) * NH / G;
    }
}
// Whether h block hb of the q-th touched expert starts a run (an expert's first h block, or the
// first h block of some block's range). NH * G stays far below 2^31.
__device__ __forceinline__ bool run_start(int q, int hb, int nbh, int NH, int G) {
    if (hb == 0 || NH <= G) return true;
    const int g = q * nbh + hb;
    const int b = (g * G + NH - 1) / NH;  // first block whose range starts at or after g
    return b * NH / G == g;
}

// ================= TMA producer (one lane) =================
__device__ void produce(const CUtensorMap* tmGU, const CUtensorMap* tmD, const Params& p,
                        uint8_t* smem, const Bars& br, const int* s_eq, int lo, int n_own,
                        volatile int* abort) {
    uint32_t stage = 0, phase = 0, armed_mask = 0, armed_par = 0;
    bool ok = true;
    auto acquire = [&]() -> uint8_t* {
        if (!mbar_wait(&br.empty[stage], phase ^ 1u, abort, kWaitLimitNs)) {
            ok = false;
            return nullptr;
        }
        armed_mask |= 1u << stage;
        armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
        return smem + (size_t)stage * kStageBytes;
    };
    auto advance = [&]() {
        if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
        }
    };
    for (int i = 0; i <= n_own && ok; ++i) {
        if (i < n_own) {  // gate_up of h block lo + i: its gate and up boxes per K chunk
            const int g = lo + i, q = g / p.nbh, hb = g - q * p.nbh, e = s_eq[q];
            const uint8_t* ga = p.gu_sf + (size_t)(e * 2 * p.nbh + hb) * p.KCd * kAtom;
            const uint8_t* ua = p.gu_sf + (size_t)(e * 2 * p.nbh + p.nbh + hb) * p.KCd * kAtom;
            for (int kc = 0; kc < p.KCd; ++kc) {
                uint8_t* st = acquire();
                if (!st) break;
                uint64_t* bar = &br.full[stage];
                mbar_arrive_expect_tx(bar, 2 * kBoxTx + 2 * kAtom);
                tma_load_3d(smem_u32(st), tmGU, bar, kc * 128, hb * 128, e);
                tma_load_3d(smem_u32(st + kBox), tmGU, bar, kc * 128, p.I + hb * 128, e);
                bulk_copy(smem_u32(st + 2 * kBox), ga + (size_t)kc * kAtom, kAtom, bar);
                bulk_copy(smem_u32(st + 2 * kBox + kAtom), ua + (size_t)kc * kAtom, kAtom, bar);
                advance();
            }
        }
        if (i >= 1 && ok) {  // down of h block lo + i - 1: two output blocks per stage
            const int g = lo + i - 1, q = g / p.nbh, hb = g - q * p.nbh, e = s_eq[q];
            for (int ob = 0; ob < p.nob; ob += 2) {
                uint8_t* st = acquire();
                if (!st) break;
                uint64_t* bar = &br.full[stage];
                const int nb = p.nob - ob >= 2 ? 2 : 1;
                mbar_arrive_expect_tx(bar, (uint32_t)nb * (kBoxTx + kAtom));
                for (int x = 0; x < nb; ++x) {
                    tma_load_3d(smem_u32(st + x * kBox), tmD, bar, hb * 128, (ob + x) * 128, e);
                    bulk_copy(smem_u32(st + 2 * kBox + x * kAtom),
                              p.dn_sf + ((size_t)(e * p.nob + ob + x) * p.KCi + hb) * kAtom,
                              kAtom, bar);
                }
                advance();
            }
        }
    }
    if (!ok) {
        *abort = 1;
        set_status(p.status, MOE_ERR_TIMEOUT);
    }
    // every stage this lane filled lands before shared memory is released
    for (int s = 0; s < kStages; ++s)
        if ((armed_mask >> s) & 1u)
            mbar_wait(&br.full[s], (armed_par >> s) & 1u, nullptr, kWaitLimitNs);
}

// ================= scale copies and MMA issue (one lane) =================
__device__ void issue_mmas(const Params& p, uint8_t* smem, uint32_t tmem, const Bars& br,
                           int lo, int n_own, volatile int* abort) {
    // x's scale atoms (one per K chunk), once
    for (int kc = 0; kc < p.KCd; ++kc)
        tmem_cp_atom(tmem + kColXsf + 4 * kc, smem_desc_plain(smem_u32(smem + kOffXsf + kc * kAtom)));
    uint32_t stage = 0, phase = 0;
    bool ok = true;
    int run = 0;
    auto landed = [&]() -> bool {
        if (!mbar_wait(&br.full[stage], phase, abort, kWaitLimitNs)) return ok = false;
        tc_fence_after();
        return true;
    };
    auto release = [&]() {
        umma_commit(&br.empty[stage]);
        if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
        }
    };
    for (int i = 0; i <= n_own && ok; ++i) {
        if (i < n_own) {
            const uint32_t buf = i & 1;
            if (!mbar_wait(&br.gu_empty[buf], ((i >> 1) & 1) ^ 1u, abort, kWaitLimitNs)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t dg = tmem + kColGu + 32 * buf, du = dg + 16;
            for (int kc = 0; kc < p.KCd && landed(); ++kc) {
                const uint32_t a0 = smem_u32(smem + (size_t)stage * kStageBytes), a1 = a0 + kBox;
                const uint32_t sfw = tmem + kColWsf + 8 * stage, sfx = tmem + kColXsf + 4 * kc;
                tmem_cp_atom(sfw, smem_desc_plain(a0 + 2 * kBox));
                tmem_cp_atom(sfw + 4, smem_desc_plain(a0 + 2 * kBox + kAtom));
                const uint32_t xb = smem_u32(smem + kOffX + kc * kTile);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    // K-major, 128-byte swizzle, +32 bytes per K = 32 step on both sides
                    const uint64_t bd = smem_desc(xb + 32 * j, 16, 1024);
                    const uint32_t id = idesc_mx_w4a8(128, kN, (uint32_t)j, (uint32_t)j);
                    const uint32_t acc = (kc | j) != 0 ? 1u : 0u;
                    umma_mx(dg, smem_desc(a0 + 32 * j, 16, 1024), bd, id, sfw, sfx, acc);
                    umma_mx(du, smem_desc(a1 + 32 * j, 16, 1024), bd, id, sfw + 4, sfx, acc);
                }
                release();
            }
            if (!ok) break;
            umma_commit(&br.gu_full[buf]);
        }
        if (i >= 1) {
            const int ii = i - 1, g = lo + ii, hb = g % p.nbh;
            const uint32_t buf = ii & 1;
            const bool first = ii == 0 || hb == 0, last = ii == n_own - 1 || hb == p.nbh - 1;
            if (!mbar_wait(&br.h_full[buf], (ii >> 1) & 1, abort, kWaitLimitNs) ||
                (first && run > 0 &&
                 !mbar_wait(br.dn_empty, (run - 1) & 1, abort, kWaitLimitNs))) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t sfh = tmem + kColHsf + 4 * buf;
            tmem_cp_atom(sfh, smem_desc_plain(smem_u32(smem + kOffHsf + buf * kAtom)));
            const uint32_t hbase = smem_u32(smem + kOffH + buf * kTile);
            for (int ob = 0; ob < p.nob && landed(); ob += 2) {
                const int nb = p.nob - ob >= 2 ? 2 : 1;
                const uint32_t a0 = smem_u32(smem + (size_t)stage * kStageBytes);
                const uint32_t sfw = tmem + kColWsf + 8 * stage;
                for (int x = 0; x < nb; ++x)
                    tmem_cp_atom(sfw + 4 * x, smem_desc_plain(a0 + 2 * kBox + x * kAtom));
                for (int x = 0; x < nb; ++x) {
                    const uint32_t d = tmem + kColDown + 16 * (ob + x);
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        umma_mx(d, smem_desc(a0 + x * kBox + 32 * j, 16, 1024),
                                smem_desc(hbase + 32 * j, 16, 1024),
                                idesc_mx_w4a8(128, kN, (uint32_t)j, (uint32_t)j), sfw + 4 * x, sfh,
                                (!first || j > 0) ? 1u : 0u);
                }
                release();
            }
            if (!ok) break;
            if (last) {
                umma_commit(br.dn_full);
                ++run;
            }
        }
    }
    if (!ok) {
        *abort = 1;
        set_status(p.status, MOE_ERR_TIMEOUT);
    }
    if (*abort) {
        umma_commit(br.drain);  // completes once every copy and MMA issued above is done
        mbar_wait(br.drain, 0, nullptr, kWaitLimitNs);
    }
}

// ================= epilogue (warps 2..5) =================
// Loops over tokens, rows and output blocks stay rolled: this code runs a few times per block,
// right after the weights have flushed it from the caches, so its size is what it costs.

// The down sums of the run of h blocks that ends at owned index ii_last: weight x sum of each of
// the expert's rows, as fp32 partials.
__device__ bool down_epilogue(const Params& p, uint32_t tmem, const Bars& br, const int* s_offq,
                              const int* s_tq, const int* s_tok, const float* s_w, int lo,
                              int ii_last, int run, volatile int* abort) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, q4 = warp & 3;
    const int g = lo + ii_last, q = g / p.nbh;
    const int hb0 = run == 0 ? max(lo - q * p.nbh, 0) : 0;  // the run's first h block
    if (!mbar_wait(br.dn_full, run & 1, abort, kWaitLimitNs)) return false;
    tc_fence_after();
    const uint32_t acc = tmem + ((uint32_t)(q4 * 32) << 16) + kColDown;
    for (int r = s_offq[q]; r < s_offq[q] + s_tq[q]; ++r) {
        const int n = s_tok[r];  // the row's token: its accumulator column in each output block
        const float w = p.scale_input ? 1.0f : s_w[r];
        float* dst = p.part + ((size_t)hb0 * p.R + r) * p.d + q4 * 32 + lane;
#pragma unroll 1
        for (int ob = 0; ob < p.nob; ob += 4) {
            uint32_t v[4];
#pragma unroll
            for (int x = 0; x < 4; ++x)
                v[x] = ob + x < p.nob ? tmem_ld_32x32b_x1(acc + 16 * (ob + x) + n) : 0u;
            tmem_ld_wait();
#pragma unroll
            for (int x = 0; x < 4; ++x)
                if (ob + x < p.nob && (ob + x) * 128 + q4 * 32 + lane < p.d)
                    dst[(ob + x) * 128] = w * __uint_as_float(v[x]);
        }
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(br.dn_empty);
    return true;
}

__device__ void epilogue(const Params& p, uint8_t* smem, uint32_t tmem, const Bars& br,
                         const int* s_offq, const int* s_tq, const int* s_tok, const float* s_w,
                         int lo, int n_own, volatile int* abort) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, q4 = warp & 3;
    const uint32_t lanes = (uint32_t)(q4 * 32) << 16;
    bool ok = true;
    int run = 0;
    for (int ii = 0; ii < n_own && ok; ++ii) {
        const int g = lo + ii, q = g / p.nbh, hb = g - q * p.nbh;
        const uint32_t buf = ii & 1;
        if (!mbar_wait(&br.gu_full[buf], (ii >> 1) & 1, abort, kWaitLimitNs)) {
            ok = false;
            break;
        }
        tc_fence_after();
        // lane n < 16: token n's row of expert q (-1: not routed to it) and its input scale
        const int r0 = s_offq[q];
        int my_row = -1;
        for (int r = r0; r < r0 + s_tq[q]; ++r)
            if (s_tok[r] == lane) my_row = r;
        const float my_s = !p.scale_input ? 1.0f : my_row >= 0 ? s_w[my_row] : 0.0f;
        const int col0 = hb * 128 + q4 * 32;  // this warp's 32 h columns: one MX block
        const bool valid = col0 < p.I;
        uint8_t* ht = smem + kOffH + buf * kTile;
        const int bcol = q4 * 32 + lane;  // byte of the h tile's rows
        const uint32_t gcol = tmem + lanes + kColGu + 32 * buf;
        uint32_t my_sc = 127;
#pragma unroll 1
        for (int n0 = 0; n0 < kN; n0 += 4) {
            uint32_t gv[4], uv[4];
            tmem_ld_32x32b_x4(gcol + n0, gv);
            tmem_ld_32x32b_x4(gcol + 16 + n0, uv);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int n = n0 + i;
                const float s = __shfl_sync(0xFFFFFFFFu, my_s, n);
                const int row = __shfl_sync(0xFFFFFFFFu, my_row, n);
                const float hv = valid ? silu(__uint_as_float(gv[i]) * s) * (__uint_as_float(uv[i]) * s)
                                       : 0.0f;
                // the block maximum of |h| over the warp's 32 columns (bits of non-negative
                // floats order as integers; NaN counts as 0, as fmaxf would skip it)
                const uint32_t ab = __float_as_uint(fabsf(hv));
                const float amax = __uint_as_float(
                    __reduce_max_sync(0xFFFFFFFFu, ab > 0x7F800000u ? 0u : ab));
                const int se = mx_scale_exp(amax, 8);
                const uint32_t code = e4m3x2(hv * pow2_f32(-se), 0.0f) & 0xFFu;
                const uint32_t sc = valid ? (uint32_t)(se + 127) : 127u;
                ht[(n >> 3) * 1024 + (n & 7) * 128 + ((((bcol >> 4) ^ (n & 7)) << 4) | (bcol & 15))] =
                    (uint8_t)code;
                if (lane == n) my_sc = sc;
                if (row >= 0) {  // a routed row: into the padded h rows too
                    const int m = row - r0;
                    const size_t prow = (size_t)q * 128 + m;
                    if (valid) p.hq[prow * p.I + col0 + lane] = (uint8_t)code;
                    if (lane == 0)
                        p.hsf[((size_t)q * p.KCi + hb) * kAtom + 16 * (m & 31) + 4 * (m >> 5) +
                              q4] = (uint8_t)sc;
                }
            }
        }
        // the accumulators are read: the next-but-one h block's MMAs may overwrite them
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&br.gu_empty[buf]);
        if (lane < kN) smem[kOffHsf + buf * kAtom + 16 * lane + q4] = (uint8_t)my_sc;
        fence_proxy_async_smem();  // the MMAs read the tile through the async proxy
        __syncwarp();
        if (lane == 0) mbar_arrive(&br.h_full[buf]);
        // the run that ended with the previous h block (a new expert starts here)
        if (ii >= 1 && hb == 0) {
            if (!down_epilogue(p, tmem, br, s_offq, s_tq, s_tok, s_w, lo, ii - 1, run, abort))
                ok = false;
            ++run;
        }
    }
    if (ok && n_own > 0 &&
        !down_epilogue(p, tmem, br, s_offq, s_tq, s_tok, s_w, lo, n_own - 1, run, abort))
        ok = false;
    if (!ok) {
        *abort = 1;
        set_status(p.status, MOE_ERR_TIMEOUT);
    }
    // this block's partials are written (or given up on): tell the summing blocks
    __threadfence();
    asm volatile("bar.sync 1, 128;" ::: "memory");
    if (warp == kFirstEpiWarp && lane == 0)
        asm volatile("red.release.gpu.global.add.s32 [%0], 1;" ::"l"(p.done) : "memory");
}

// ================= x to MXFP8 (warps 1..5, beside the first weight copies) =================
// Token n's 32-element block kb: codes into row n of the B tile of chunk kb / 4, the scale into
// x's atom of that chunk (16 n + kb % 4). Rows past T and blocks past d are zero with scale 1.
__device__ void quantize_x(const Params& p, uint8_t* smem) {
    const int KB = p.d / 32, KBp = 4 * p.KCd;
    for (int it = threadIdx.x - 32; it < kN * KBp; it += kThreads - 32) {
        const int n = it / KBp, kb = it - n * KBp;
        uint32_t w[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        uint32_t sc = 127;
        if (n < p.T && kb < KB) {
            const uint4* src = reinterpret_cast<const uint4*>(p.x + (size_t)n * p.d + kb * 32);
            float v[32];
            float amax = 0.0f;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const uint4 u = __ldg(src + c);
                const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    v[8 * c + 2 * h] = __uint_as_float(w4[h] << 16);
                    v[8 * c + 2 * h + 1] = __uint_as_float(w4[h] & 0xFFFF0000u);
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
        uint8_t* row = smem + kOffX + (kb >> 2) * kTile + (n >> 3) * 1024 + (n & 7) * 128;
        const int c16 = 2 * (kb & 3);
        *reinterpret_cast<uint4*>(row + ((c16 ^ (n & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
        *reinterpret_cast<uint4*>(row + (((c16 + 1) ^ (n & 7)) << 4)) =
            make_uint4(w[4], w[5], w[6], w[7]);
        smem[kOffXsf + (kb >> 2) * kAtom + 16 * n + (kb & 3)] = (uint8_t)sc;
    }
}

// Block 0: x's codes and scales from shared memory into the padded rows of every routed slot
// (the layout of the multi-kernel path; read back by checks). One thread per (slot, K block).
__device__ void store_x_rows(const Params& p, const uint8_t* smem, const int* s_pos,
                             const int* s_rq, const int* s_offq, int tid, int nthreads) {
    const int KB = p.d / 32, KBp = 4 * p.KCd;
    for (int it = tid; it < p.R * KBp; it += nthreads) {
        const int slot = it / KBp, kb = it - slot * KBp, n = slot / p.k;
        const int r = s_pos[slot], q = s_rq[r], m = r - s_offq[q];
        const size_t prow = (size_t)q * 128 + m;
        const uint8_t* row = smem + kOffX + (kb >> 2) * kTile + (n >> 3) * 1024 + (n & 7) * 128;
        const int c16 = 2 * (kb & 3);
        if (kb < KB) {
            uint4* o = reinterpret_cast<uint4*>(p.xq + prow * p.d + kb * 32);
            o[0] = *reinterpret_cast<const uint4*>(row + ((c16 ^ (n & 7)) << 4));
            o[1] = *reinterpret_cast<const uint4*>(row + (((c16 + 1) ^ (n & 7)) << 4));
        }
        p.xsf[((size_t)q * p.KCd + (kb >> 2)) * kAtom + 16 * (m & 31) + 4 * (m >> 5) + (kb & 3)] =
            smem[kOffXsf + (kb >> 2) * kAtom + 16 * n + (kb & 3)];
    }
}

// ================= the summing step (all threads) =================
// Unit u = (token t, 128 output columns cb): the token's terms (its slots in order, then each
// slot's row's run-start h blocks ascending) summed by 6 groups of 32 threads (four columns
// each, terms grp, grp + 6, ...), then the groups in order; one rounding to bf16.
__device__ void sum_partials(const Params& p, uint8_t* smem, const int* s_pos, const int* s_rq,
                             int NH, int owners, volatile int* abort) {
    constexpr int kGroups = kThreads / 32;
    const int G = gridDim.x, b = blockIdx.x, tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int ncb = (p.d + 127) / 128, units = p.T * ncb;
    const int first = G - 1 - b;
    if (first >= units) return;
    int* terms = reinterpret_cast<int*>(smem);  // k * nbh at most
    volatile int* nterm = reinterpret_cast<volatile int*>(terms + kMaxK * kMaxNbh);
    float4* red4 = reinterpret_cast<float4*>(smem + 8 * 1024);
    if (tid == 0) {
        const uint64_t t0 = globaltimer_ns();
        while (ld_acquire(p.done) < owners) {
            if (*abort || globaltimer_ns() - t0 > kWaitLimitNs) {
                set_status(p.status, MOE_ERR_TIMEOUT);
                *abort = 1;
                break;
            }
        }
    }
    __syncthreads();
    if (*abort) return;
    const int c4 = lane, grp = warp;
    for (int u = first; u < units; u += G) {
        const int t = u / ncb, cb = u - t * ncb;
        if (warp == 0) {
            // lane j < k: slot (t, j)'s row and its run starts; positions by a prefix sum
            int r = -1, q = 0, cnt = 0;
            if (lane < p.k) {
                r = s_pos[t * p.k + lane];
                q = s_rq[r];
                for (int hb = 0; hb < p.nbh; ++hb) cnt += run_start(q, hb, p.nbh, NH, G) ? 1 : 0;
            }
            int pos = cnt;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xFFFFFFFFu, pos, o);
                if (lane >= o) pos += y;
            }
            if (lane == 31) *nterm = pos;
            pos -= cnt;
            if (lane < p.k)
                for (int hb = 0; hb < p.nbh; ++hb)
                    if (run_start(q, hb, p.nbh, NH, G)) terms[pos++] = hb * p.R + r;
        }
        __syncthreads();
        const int nt = *nterm;
        const int col = cb * 128 + 4 * c4;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (col < p.d) {
            for (int m0 = grp; m0 < nt; m0 += 4 * kGroups) {
                float4 v[4];
#pragma unroll
                for (int x = 0; x < 4; ++x) {
                    const int m = m0 + x * kGroups;
                    v[x] = m < nt ? __ldcg(reinterpret_cast<const float4*>(
                                        p.part + (size_t)terms[m] * p.d + col))
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
                }
#pragma unroll
                for (int x = 0; x < 4; ++x) {
                    acc.x += v[x].x;
                    acc.y += v[x].y;
                    acc.z += v[x].z;
                    acc.w += v[x].w;
                }
            }
        }
        red4[grp * 32 + c4] = acc;
        __syncthreads();
        if (tid < 32 && col < p.d) {
            float4 s4 = red4[c4];
            for (int gq = 1; gq < kGroups; ++gq) {
                const float4 v = red4[gq * 32 + c4];
                s4.x += v.x;
                s4.y += v.y;
                s4.z += v.z;
                s4.w += v.w;
            }
            uint2 packed;
            packed.x = pack_bf16x2(s4.x, s4.y);
            packed.y = pack_bf16x2(s4.z, s4.w);
            *reinterpret_cast<uint2*>(p.out + (size_t)t * p.d + col) = packed;
        }
        __syncthreads();  // before the next unit rewrites terms and red4
    }
}

__global__ void __launch_bounds__(kThreads, 1)
    decode_mx_tc_kernel(const __grid_constant__ CUtensorMap tmGU,
                        const __grid_constant__ CUtensorMap tmD, const Params p, int vpl) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    int* s_eq = reinterpret_cast<int*>(smem + kOffLists);
    int* s_tq = s_eq + kMaxE;
    int* s_offq = s_tq + kMaxE;
    int* s_tok = s_offq + kMaxE;
    float* s_w = reinterpret_cast<float*>(s_tok + kDecodeFusedMaxRows);
    int* s_pos = reinterpret_cast<int*>(s_w + kDecodeFusedMaxRows);
    int* s_rq = s_pos + kDecodeFusedMaxRows;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBars);
    Bars br;
    br.full = bars;
    br.empty = bars + kStages;
    br.gu_full = bars + 2 * kStages;
    br.gu_empty = br.gu_full + 2;
    br.h_full = br.gu_empty + 2;
    br.dn_full = br.h_full + 2;
    br.dn_empty = br.dn_full + 1;
    br.drain = br.dn_empty + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kNumBars);
    volatile int* flags = reinterpret_cast<volatile int*>(tmem_slot + 1);  // [0] abort, [1] nq
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    griddep_wait();
    // x is read after the dispatch: ask L2 for it now, beside the logits
    for (int i = threadIdx.x; i < p.T * p.d / 64; i += kThreads)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(p.x + (size_t)i * 64));

    // ---- router top-k and dispatch indices (scratch in the stage buffers, which no copy uses
    // yet); the set-up runs beside the routing
    const DecodeRouteIO rio{p.logits, p.T, p.E, p.k, p.R, p.score_fn, p.renorm, p.topk_ids,
                            p.topk_w, p.counts, p.offsets, p.s2p, p.p2s};
    DecodeRouteSmem rsm;
    rsm.eq = s_eq;
    rsm.tq = s_tq;
    rsm.offq = s_offq;
    rsm.tok = s_tok;
    rsm.wrow = s_w;
    rsm.pos = s_pos;
    rsm.nq = flags + 1;
    decode_route_scratch(rsm, smem);
    decode_route_tokens<kWarps>(rio, rsm, vpl);
    if (warp == kMmaWarp) tmem_alloc(tmem_slot, kTmemCols);
    if (warp == kFirstEpiWarp && lane == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&br.full[s], 1);
            mbar_init(&br.empty[s], 1);
        }
        for (int b2 = 0; b2 < 2; ++b2) {
            mbar_init(&br.gu_full[b2], 1);
            mbar_init(&br.gu_empty[b2], 4);
            mbar_init(&br.h_full[b2], 4);
        }
        mbar_init(br.dn_full, 1);
        mbar_init(br.dn_empty, 4);
        mbar_init(br.drain, 1);
        flags[0] = 0;
        fence_barrier_init();
    }
    if (warp == kProducerWarp && lane == 0) {
        tma_prefetch_desc(&tmGU);
        tma_prefetch_desc(&tmD);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const int nq = decode_dispatch(rio, rsm, blockIdx.x == 0);
    for (int q = threadIdx.x; q < nq; q += kThreads)
        for (int r = s_offq[q]; r < s_offq[q] + s_tq[q]; ++r) s_rq[r] = q;
    __syncthreads();
    const uint32_t tmem = *tmem_slot;
    const int G = gridDim.x, NH = nq * p.nbh, owners = NH < G ? NH : G;
    int lo, hi;
    owned_range(NH, G, blockIdx.x, &lo, &hi);
    const int n_own = hi - lo;

    if (n_own > 0) {
        if (warp == kProducerWarp) {
            if (lane == 0) produce(&tmGU, &tmD, p, smem, br, s_eq, lo, n_own, flags);
            __syncwarp();
        } else {
            // x to MXFP8 while the first weight copies are in flight
            quantize_x(p, smem);
            fence_proxy_async_smem();  // the MMAs and scale copies read x through the async proxy
            asm volatile("bar.sync 2, 160;" ::: "memory");
            if (warp == kMmaWarp) {
                if (lane == 0) issue_mmas(p, smem, tmem, br, lo, n_own, flags);
                __syncwarp();
            } else {
                if (blockIdx.x == 0)
                    store_x_rows(p, smem, s_pos, s_rq, s_offq, threadIdx.x - 32 * kFirstEpiWarp,
                                 128);
                epilogue(p, smem, tmem, br, s_offq, s_tq, s_tok, s_w, lo, n_own, flags);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
    sum_partials(p, smem, s_pos, s_rq, NH, owners, flags);
}

}  // namespace

bool decode_mx_tc_applies(int T, int d, int k, int I, int Is) {
    return Is == 0 && T >= 1 && T <= kN && T * k <= kDecodeFusedMaxRows && d <= 128 * kMaxNob &&
           I <= 128 * kMaxNbh;
}

size_t decode_mx_tc_part_bytes(int T, int d, int k, int I) {
    return (size_t)((I + 127) / 128) * T * k * d * 4;
}

cudaError_t launch_decode_mx_tc(const DecodeMxTcArgs& a, cudaStream_t s) {
    {
        const cudaError_t e = ensure_max_dynamic_smem(decode_mx_tc_kernel, kSmemBytes);
        if (e != cudaSuccess) return e;
    }
    const MxTcGeom gg = mx_tc_geom(true, a.d, a.I, a.E), gd = mx_tc_geom(false, a.I, a.d, a.E);
    CUtensorMap tmGU, tmD;
    // E2M1 codes [E][C][Kp] (two per byte), boxes of 128 K elements x 128 columns landing 16
    // codes per 16 bytes
    const cuuint64_t gu_dims[3] = {(cuuint64_t)gg.Kp, (cuuint64_t)gg.C, (cuuint64_t)a.E};
    const cuuint64_t gu_str[2] = {(cuuint64_t)gg.Kp / 2, (cuuint64_t)gg.C * gg.Kp / 2};
    const cuuint64_t dn_dims[3] = {(cuuint64_t)gd.Kp, (cuuint64_t)gd.C, (cuuint64_t)a.E};
    const cuuint64_t dn_str[2] = {(cuuint64_t)gd.Kp / 2, (cuuint64_t)gd.C * gd.Kp / 2};
    const cuuint32_t box[3] = {128, 128, 1};
    if (!encode_tensor_map(&tmGU, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 3, a.w_gate_up, gu_dims,
                           gu_str, box) ||
        !encode_tensor_map(&tmD, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 3, a.w_down, dn_dims,
                           dn_str, box))
        return cudaErrorInvalidValue;
    Params p;
    p.x = static_cast<const __nv_bfloat16*>(a.x);
    p.logits = a.logits;
    p.gu_sf = static_cast<const uint8_t*>(a.w_gate_up) + gg.sf_off;
    p.dn_sf = static_cast<const uint8_t*>(a.w_down) + gd.sf_off;
    p.topk_ids = a.topk_ids;
    p.topk_w = a.topk_weights;
    p.counts = a.counts;
    p.offsets = a.offsets;
    p.s2p = a.sorted_to_slot;
    p.p2s = a.slot_to_sorted;
    p.xq = static_cast<uint8_t*>(a.x_codes);
    p.xsf = static_cast<uint8_t*>(a.x_sf);
    p.hq = static_cast<uint8_t*>(a.h_codes);
    p.hsf = static_cast<uint8_t*>(a.h_sf);
    p.part = static_cast<float*>(a.partials);
    p.out = static_cast<__nv_bfloat16*>(a.out);
    p.done = a.done;
    p.status = a.status;
    p.T = a.T;
    p.d = a.d;
    p.E = a.E;
    p.k = a.k;
    p.I = a.I;
    p.R = a.T * a.k;
    p.score_fn = a.score_fn;
    p.renorm = a.renorm ? 1 : 0;
    p.scale_input = a.scale_input ? 1 : 0;
    p.KCd = gg.KC;
    p.KCi = gd.KC;
    p.nbh = gg.cbh;
    p.nob = gd.cbh;
    const int vpl = a.E <= 32 ? 1 : a.E <= 64 ? 2 : a.E <= 128 ? 4 : 8;
    int grid = device_sm_count();
    if (grid > kDecodeFusedMaxGrid) grid = kDecodeFusedMaxGrid;
    // one block per SM (its shared memory allows no more), all resident: cooperative launch
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
    return cudaLaunchKernelEx(&cfg, decode_mx_tc_kernel, tmGU, tmD, p, vpl);
}

}  // namespace rdg
