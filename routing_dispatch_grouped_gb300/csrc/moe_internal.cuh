// Internal declarations shared by the kernels and the C ABI layer of libmoe.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "moe.h"

namespace rdg {

constexpr int kMaxE = 256;
constexpr int kMaxK = 32;
constexpr int kDispatchChunk = 256;   // slots per dispatch chunk (one warp)
constexpr size_t kStatusBytes = 256;  // status word + padding at the head of a workspace

// Tile shape of the tcgen05 grouped GEMM: 128 rows x 256 accumulator columns, K step 64
// (one 128-byte swizzle span of bf16).
constexpr int kTileM = 128;
constexpr int kTileN = 256;
constexpr int kTileK = 64;

// ---------------------------------------------------------------------------------------------
// device helpers
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ void set_status(int* status, int code) {
    if (status) atomicCAS(status, 0, code);
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// SwiGLU's activation in fp32 (the GEMM epilogues and the fused decode kernel share it, so every
// path rounds h from the same value)
__device__ __forceinline__ float silu(float z) { return z * __frcp_rn(1.0f + __expf(-z)); }

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&v);
}

// Acquire load at GPU scope (a counter or flag another block releases).
__device__ __forceinline__ int ld_acquire(const int* ptr) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(ptr) : "memory");
    return v;
}

// ---- mbarrier ----
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase with parity `parity` of `bar` to complete, giving up after `limit_ns` or
// when *abort becomes non-zero. Returns false when it gave up.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 15u) == 0) {
            if (abort != nullptr && *abort) return false;
            if (globaltimer_ns() - t0 > limit_ns) return false;
        }
    }
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---- TMA (tiled bulk tensor copies, global -> shared) ----
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint64_t* bar,
                                            int c0, int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
        "l"(map), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
        : "memory");
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint64_t* bar,
                                            int c0, int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
        "l"(map), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

// The same copies with an L2 eviction-priority hint (a createpolicy value): streamed weights
// are marked evict-first, activations that every column tile re-reads evict-last.
__device__ __forceinline__ uint64_t l2_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t l2_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const CUtensorMap* map,
                                                 uint64_t* bar, int c0, int c1, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(dst),
        "l"(map), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "l"(pol)
        : "memory");
}
__device__ __forceinline__ void tma_load_3d_hint(uint32_t dst, const CUtensorMap* map,
                                                 uint64_t* bar, int c0, int c1, int c2,
                                                 uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(dst),
        "l"(map), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "l"(pol)
        : "memory");
}

// TMA store of a tile from shared memory (bulk async group; the tensor map clips at its edges).
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int c0, int c1,
                                             int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
            map),
        "r"(src), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}
__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Wait until at most N committed bulk groups of this thread still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// Wait until every committed bulk group of this thread has completed.
__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// ---- tcgen05 (5th-generation tensor cores, accumulators in tensor memory) ----
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[smem] * B[smem], bf16 inputs, fp32 accumulate (kind::f16).
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrive on `bar` once every tcgen05 operation this thread issued before has completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}
// 32 lanes x 32 consecutive 32-bit columns: thread i of the warp gets lane (base + i).
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr)
        : "memory");
}
// 32 lanes x one 32-bit column.
__device__ __forceinline__ uint32_t tmem_ld_32x32b_x1(uint32_t taddr) {
    uint32_t r;
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];" : "=r"(r) : "r"(taddr)
                 : "memory");
    return r;
}
// 32 lanes x 4 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_ld_32x32b_x4(uint32_t taddr, uint32_t (&r)[4]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(taddr)
                 : "memory");
}
// 32 lanes x 16 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Named barrier 1 among the 128 threads of the four epilogue warps of the tcgen05 GEMMs (id 0
// is __syncthreads; no other warp of those kernels uses id 1).
__device__ __forceinline__ void epilogue_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// The same barrier, returning to every epilogue thread whether any of them passed `v` true, so
// the four epilogue warps take the same branch (and none is left at a named barrier).
__device__ __forceinline__ bool epilogue_any(bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred pi, po;\n\t"
        "setp.ne.u32 pi, %1, 0;\n\t"
        "bar.red.or.pred po, 1, 128, pi;\n\t"
        "selp.u32 %0, 1, 0, po;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v)
        : "memory");
    return r != 0;
}

// Shared-memory matrix descriptor for tcgen05.mma (sm_100 family): start address, leading and
// stride byte offsets (all >> 4), descriptor version 1 (bit 46), swizzle mode in bits 61-63
// (2 = 128-byte swizzle). Tiles are 1024-byte aligned, so the base-offset field stays 0.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor, kind::f16: fp32 accumulator (bits 4-5 = 1), A and B bf16 (bits 7-9 and
// 10-12 = 1), A K-major (bit 15 = 0), B MN-major (bit 16 = 1), N >> 3 in bits 17-22,
// M >> 4 in bits 24-28.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, bool b_mn_major) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
// The same with A's major-ness chosen too (bit 15 = 1: A MN-major).
__host__ __device__ constexpr uint32_t idesc_bf16_f32_ab(int M, int N, bool a_mn_major,
                                                         bool b_mn_major) {
    return idesc_bf16_f32(M, N, b_mn_major) | ((a_mn_major ? 1u : 0u) << 15);
}

// ---------------------------------------------------------------------------------------------
// programmatic dependent launch
// ---------------------------------------------------------------------------------------------
// Every kernel calls griddep_wait() before it reads data written by the kernel launched before
// it on the stream. Launched normally this returns at once; launched with programmatic stream
// serialization (inside moe_forward's chain) it lets the kernel start, run its prologue
// (barrier set-up, TMEM allocation, descriptor prefetch) while the previous kernel drains, and
// only then wait for that kernel's results.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Launches issued while a PdlScope(true) is alive on this host thread may overlap the previous
// kernel on the stream as described above.
bool pdl_enabled();
struct PdlScope {
    explicit PdlScope(bool on);
    ~PdlScope();
    bool prev;
};

// cluster_x > 1 launches thread-block clusters of that many CTAs along x.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel_ex(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t s, int cluster_x, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    int n = 0;
    if (pdl_enabled()) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    if (cluster_x > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = cluster_x;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t s, Args&&... args) {
    return launch_kernel_ex(kernel, grid, block, smem, s, 1, std::forward<Args>(args)...);
}

// ---------------------------------------------------------------------------------------------
// launchers (one per kernel family); each returns the error of its launch
// ---------------------------------------------------------------------------------------------
cudaError_t launch_route(const float* logits, int T, int E, int k, int score_fn, bool renorm,
                         int32_t* ids, float* weights, cudaStream_t s);

// Router logits from hidden states (fp32, sequential in K) and the top-k in one kernel.
cudaError_t launch_route_hidden(const void* x, bool bf16, const float* w_router,
                                const float* bias, int T, int d, int E, int k, int score_fn,
                                bool renorm, float* logits, int32_t* ids, float* weights,
                                cudaStream_t s);

// Dispatch scratch (in a workspace after the status word): per-chunk counts/bases int32
// [nchunks * E].
size_t dispatch_scratch_bytes(int R, int E);
cudaError_t launch_dispatch(const int32_t* ids, const void* x, size_t row_bytes, int T, int E,
                            int k, int32_t* counts, int32_t* offsets, int32_t* sorted_to_slot,
                            int32_t* slot_to_sorted, void* x_sorted, int32_t* chunk_scratch,
                            int* status, cudaStream_t s);
// Number of kernels launch_dispatch enqueues.
int dispatch_kernel_count(bool copy_rows);

// Row copy of dispatch alone: x_sorted[slot_to_sorted[t*k+j]] = x[t] (grid-wide).
cudaError_t launch_dispatch_copy(const void* x, size_t row_bytes, int T, int k,
                                 const int32_t* slot_to_sorted, void* x_sorted, cudaStream_t s);

// Route and dispatch indices in one single-block kernel, for T*k <= kSmallDispatchMaxSlots.
constexpr int kSmallDispatchMaxSlots = 1024;
cudaError_t launch_route_dispatch_small(const float* logits, int T, int E, int k, int score_fn,
                                        bool renorm, int32_t* ids, float* weights,
                                        int32_t* counts, int32_t* offsets,
                                        int32_t* sorted_to_slot, int32_t* slot_to_sorted,
                                        cudaStream_t s);

// Fused decode layer (decode_fused.cu): route, dispatch, gate_up + SwiGLU, down and combine in
// one cooperative kernel, for bf16 layers without a shared expert and at most
// kDecodeFusedMaxTokens tokens.
constexpr int kDecodeFusedMaxTokens = 16;
constexpr int kDecodeFusedMaxRows = 256;  // T * k
constexpr int kDecodeFusedMaxGrid = 512;  // blocks (one per SM, at most this many)
bool decode_fused_applies(moe_dtype dt, int T, int k, int Is);
// Its scratch: counters (which must be zero at launch) and the partial sums.
struct DecodeFusedLayout {
    int nbh, nka, nbd, nkb;  // h blocks, gate_up K chunks, output blocks, down K chunks
    size_t counter_bytes;    // int counters
    size_t part_a, part_b, part_bytes;  // partial sums: offsets and total size
    size_t part_c;                      // owner-layout down partials (0: none)
};
DecodeFusedLayout decode_fused_layout(int T, int d, int k, int I, bool mx = false);
struct DecodeFusedArgs {
    const void* x;                  // [T, d] bf16
    const float* logits;            // [T, E]
    const void* w_gate_up;          // [E, d, 2I] or packed
    const void* w_down;             // [E, I, d] or packed
    bool packed;
    int score_fn;
    bool renorm;
    bool scale_input;               // router weight scales the expert input, combine weight 1
    int T, d, E, k, I;
    int32_t* topk_ids;              // outputs: router and dispatch results
    float* topk_weights;
    int32_t* counts;
    int32_t* offsets;
    int32_t* sorted_to_slot;
    int32_t* slot_to_sorted;
    void* h;                        // [R, I] bf16
    void* out;                      // [T, d] bf16
    int* counters;                  // counter_bytes, zero at launch
    void* partials;                 // part_bytes
    int* status;
    // MX layers: w_gate_up / w_down are MX buffers (packed is false); x and h are rounded to
    // MXFP8 in the kernel, h's codes [R, I] and scales [R, ceil(I / 32)] going here (and its
    // values into h)
    bool mx = false;
    void* h_codes = nullptr;
    void* h_scales = nullptr;
};
cudaError_t launch_decode_fused(const DecodeFusedArgs& a, cudaStream_t s);

// One-kernel MX decode layer on the block-scaled tensor cores (decode_mx_tc.cu), for
// moe_forward_mx_tc: weights in the MX tensor-core layout, no shared expert, at most 16 tokens,
// d <= 2048, I <= 4096. Its one counter sits in the workspace head at kDecodeMxTcCounterByte
// (cleared with the status word before the launch); its partial sums take
// decode_mx_tc_part_bytes.
constexpr size_t kDecodeMxTcCounterByte = 128;
bool decode_mx_tc_applies(int T, int d, int k, int I, int Is);
size_t decode_mx_tc_part_bytes(int T, int d, int k, int I);
struct DecodeMxTcArgs {
    const void* x;          // [T, d] bf16
    const float* logits;    // [T, E]
    const void* w_gate_up;  // MX tensor-core layout (moe_quantize_weights_mx_tc)
    const void* w_down;
    int score_fn;
    bool renorm;
    bool scale_input;
    int T, d, E, k, I;
    int32_t* topk_ids;      // outputs: router and dispatch results
    float* topk_weights;
    int32_t* counts;
    int32_t* offsets;
    int32_t* sorted_to_slot;
    int32_t* slot_to_sorted;
    void* x_codes;          // x and h rounded to MXFP8, written for the routed rows in the
    void* x_sf;             // padded layout of moe_forward_mx_tc's workspace
    void* h_codes;
    void* h_sf;
    void* partials;         // decode_mx_tc_part_bytes
    void* out;              // [T, d] bf16
    int* done;              // the counter (zero at launch)
    int* status;
};
cudaError_t launch_decode_mx_tc(const DecodeMxTcArgs& a, cudaStream_t s);

cudaError_t launch_combine(const float* y_sorted, const int32_t* slot_to_sorted,
                           const float* weights, const float* y_shared, int T, int d, int k,
                           bool out_bf16, void* out, cudaStream_t s);

// Grouped GEMMs. `which` selects gate_up (+SwiGLU, output dtype of the layer) or down (fp32).
enum GemmKind { kGateUp = 0, kDown = 1 };
// Packed weight layout (pack.cu): 64-column x 64-row blocks stored contiguously, block
// (e, nb, kb) at rows ((e * nb_total + nb) * kpad + 64 kb) of a [rows, 64] bf16 matrix. gate_up
// blocks its gate and up halves separately (nbh blocks each).
struct PackedGeom {
    int nbh;   // 64-column blocks per half (gate_up) or in all (down)
    int nb;    // blocks per expert: 2 nbh (gate_up) or nbh (down)
    int kpad;  // K rounded up to 64
};
PackedGeom packed_geom(int kind, int K, int N);  // N = I (gate_up) or d (down)
cudaError_t launch_pack_weights(int kind, const void* w, void* packed, int E, int K, int N,
                                cudaStream_t s);

struct GroupedGemmArgs {
    GemmKind kind;
    const void* a;            // [R, K] rows (x_sorted / x for gate_up, h for down)
    const void* b;            // weights: [E, K, 2I] (gate_up) or [E, K, d] (down), or packed
    bool packed;              // b is in the packed layout
    const int32_t* offsets;   // [E+1] or nullptr (one group of R rows)
    const int32_t* sorted_to_slot;
    const float* topk_weights;
    bool scale_rows;          // gate_up: scale accumulators by the row weight
    bool weight_rows;         // down: multiply output rows by the row weight
    int R, K, N, E;           // N = I for gate_up (h columns), d for down
    void* out;                // h [R, I] (layer dtype) or y_sorted [R, d] fp32
    int* status;
    void* ab = nullptr;       // gate_up for training: also store [g | u] before the row scale
                              // ([R, 2I], layer dtype); only the 128-row-tile kernel and the
                              // fp32 kernel write it
    bool mx_h = false;        // gate_up: round h to MXFP8 (blocks of 32 along I) before storing
                              // it (bf16 holds the value exactly); 128-row-tile kernel only
};
// Batches with at most this many routed rows use the small-batch (decode) GEMM configuration.
constexpr int kSmallBatchRows = 512;
// bf16 tensor-core path; picks one of the kernels below (pick_grouped_gemm_bf16).
cudaError_t launch_grouped_gemm_bf16(const GroupedGemmArgs& a, cudaStream_t s);
enum GemmPick { kPickRows = 0, kPick2sm = 1, kPickSwap = 2, kPickSwapPair = 3 };
// special_epilogue: gate_up storing the training accumulators or rounding h to MXFP8
GemmPick pick_grouped_gemm_bf16(GemmKind kind, int R, int groups, bool special_epilogue);
// tokens as the MMA M side (128-row tiles; gemm_tc.cu)
cudaError_t launch_grouped_gemm_bf16_rows(const GroupedGemmArgs& a, cudaStream_t s);
// 256-row tiles on CTA pairs with tcgen05.mma.cta_group::2 (gemm_tc_2sm.cu)
cudaError_t launch_grouped_gemm_bf16_2sm(const GroupedGemmArgs& a, cudaStream_t s);
// weights as the MMA M side, tokens as N (tiles padded to 16 tokens; gemm_tc_swap.cu)
cudaError_t launch_grouped_gemm_bf16_swap(const GroupedGemmArgs& a, cudaStream_t s);
// weights as the M = 256 side on CTA pairs, up to 256 tokens as N (gemm_tc_swap_pair.cu)
cudaError_t launch_grouped_gemm_bf16_swap_pair(const GroupedGemmArgs& a, cudaStream_t s);
// 2D/3D bf16 tensor map with 128-byte swizzle and zero fill outside the tensor.
bool encode_tensor_map_bf16(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims,
                            const cuuint64_t* strides, const cuuint32_t* box);
// The same for fp32 (used for TMA stores of fp32 tiles).
bool encode_tensor_map_f32(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims,
                           const cuuint64_t* strides, const cuuint32_t* box);
cudaError_t launch_grouped_gemm_f32(const GroupedGemmArgs& a, cudaStream_t s);

int device_sm_count();
// Lets kernel `fn` take `bytes` of dynamic shared memory on the current device. The attribute
// belongs to each device's copy of the module, so it is set the first time each device
// launches the kernel (a process-wide once would leave every other device without it).
cudaError_t ensure_max_dynamic_smem(const void* fn, int bytes);
template <typename K>
cudaError_t ensure_max_dynamic_smem(K* kernel, int bytes) {
    return ensure_max_dynamic_smem(reinterpret_cast<const void*>(kernel), bytes);
}
// Stall of the 128-row gate_up kernel's test hook (moe_debug_set_gemm_stall_ns; 0 = off).
uint32_t debug_gemm_stall_ns();

// ---------------------------------------------------------------------------------------------
// MX formats (mx.cu): MXFP4 expert weights, MXFP8 activations
// ---------------------------------------------------------------------------------------------
// MX weights are stored in blocks of 64 columns x 32 K rows (mx.cu); gate_up blocks its gate
// and up halves separately (gate blocks first), like the packed bf16 layout.
struct MxBlocks {
    int half;  // gate_up: I (columns of a half); down: 0
    int nbh;   // 64-column blocks per half (gate_up) or in all (down)
    int nb;    // column blocks per expert
    int kb;    // 32-row K blocks
    int cols;  // columns of the logical weight (2I or d)
};
struct MxGeom {
    MxBlocks blocks;
    size_t codes;       // bytes of codes: G * NB * KB * 1024
    size_t scales_off;  // offset of the scales (G * NB * KB * 64 bytes)
    size_t total;       // buffer size
};
MxBlocks mx_blocks(bool gate_up, int K, int N);  // N = I (gate_up) or d (down)
MxGeom mx_geom(bool gate_up, int K, int N, int G);
// bf16 weights [G, K, cols] -> MX buffer
cudaError_t launch_mx_quant_weights(bool gate_up, const void* w, int G, int K, int N, void* mx,
                                    cudaStream_t s);
// MX buffer -> bf16 [G, K, cols]; groups g with offsets[g + 1] == offsets[g] are skipped
// (offsets may be null)
cudaError_t launch_mx_dequant_weights(bool gate_up, const void* mx, int G, int K, int N,
                                      const int32_t* offsets, void* w, cudaStream_t s);
// bf16 rows [R, K] rounded to MXFP8 and back into out (may be in; null: not written); codes
// [R, K] and scales [R, ceil(K / 32)] written when not null
cudaError_t launch_mx_rows(const void* in, int R, int K, void* out, void* codes, void* scales,
                           cudaStream_t s);

// MX tensor-core layout (gemm_mx_tc.cu): weights as K-major E2M1 codes [G][C][Kp / 2] (Kp = K
// rounded up to 128) followed by 512-byte scale atoms [G][CB][KC]; activations as E4M3 codes
// [Rp][K] with every expert's rows starting at a multiple of 128, and scale atoms
// [Rp / 128][KC]. The block-scaled tcgen05 GEMM reads both.
struct MxTcGeom {
    int C;          // logical columns (2I or d)
    int Kp;         // K rounded up to 128
    int KC;         // Kp / 128
    int cbh;        // 128-column scale blocks of a half (gate_up) or of all columns (down)
    int CB;         // scale blocks per group
    size_t sf_off;  // byte offset of the scale atoms
    size_t total;   // buffer size
};
MxTcGeom mx_tc_geom(bool gate_up, int K, int N, int G);  // N = I (gate_up) or d (down)
cudaError_t launch_mx_tc_quant_weights(bool gate_up, const void* w, int G, int K, int N, void* mx,
                                       cudaStream_t s);
cudaError_t launch_mx_tc_dequant_weights(bool gate_up, const void* mx, int G, int K, int N,
                                         void* w, cudaStream_t s);
// x [T, d] bf16 to the padded MXFP8 layout: each token's codes and scales go to the padded row
// of each of its slots (topk_ids, slot_to_sorted, offsets of the dispatch) and, when codes_sh is
// not null, to row t of the shared expert's single group.
cudaError_t launch_mx_tc_quant_rows(const void* x, int T, int d, int k, int E,
                                    const int32_t* topk_ids, const int32_t* slot_to_sorted,
                                    const int32_t* offsets, void* codes, void* sf, void* codes_sh,
                                    void* sf_sh, cudaStream_t s);
struct MxTcGemmArgs {
    GemmKind kind;
    const void* a;     // E4M3 codes [Rp][K]
    const void* a_sf;  // their scale atoms
    const void* b;     // weights in the MX tensor-core layout
    const int32_t* offsets;  // [groups + 1] or nullptr (one group of R rows)
    const int32_t* sorted_to_slot;
    const float* topk_weights;
    bool scale_rows;   // gate_up: multiply each row's accumulators by its routing weight
    int R, Rp, K, N, groups;
    void* out;         // gate_up: h codes [Rp][N]; down: y fp32 [R][N]
    void* h_sf;        // gate_up: h scale atoms [Rp / 128][ceil(N / 128)]
    int* status;
};
cudaError_t launch_mx_tc_gemm(const MxTcGemmArgs& a, cudaStream_t s);
// Tensor map of any element type with a 128-byte swizzle (or none) and zero fill outside the
// tensor.
bool encode_tensor_map(CUtensorMap* m, CUtensorMapDataType type, int rank, const void* base,
                       const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box,
                       bool swizzle128 = true);


// ---------------------------------------------------------------------------------------------
// backward pass (gemm_bwd.cu: tensor cores; backward.cu: fp32 layers and the small kernels)
// ---------------------------------------------------------------------------------------------
// dgrad: out[p] = a[p] . W[e]^T for the rows p of expert e (a [R, K] in the layer dtype).
//   kDgradDown: a = dy_sorted [R, d], W = w_down [E, I, d] (K = d, N = I); the epilogue is the
//     SwiGLU backward: reads ab [R, 2I], writes d_ab [R, 2I] (layer dtype) and, with a row
//     scale, per-(row, 256-column tile) partial sums of d_scale into scale_part [R, n_tiles].
//   kDgradGateUp: a = d_ab [R, 2I], W = w_gate_up [E, d, 2I] (K = 2I, N = d); fp32 output
//     dx_sorted [R, d].
enum BwdKind { kDgradDown = 0, kDgradGateUp = 1 };
constexpr int kBwdTileN = 256;  // output columns per dgrad tile (scale_part has one per tile)
struct DgradArgs {
    BwdKind kind;
    const void* a;            // dy_sorted or d_ab
    const void* w;            // w_down or w_gate_up ([TP-packed] layout or packed)
    bool packed;
    const int32_t* offsets;   // [E + 1] or nullptr (one group of R rows)
    const int32_t* sorted_to_slot;
    const float* topk_weights;
    bool scale_rows;          // kDgradDown: router score scales the expert input
    const void* ab;           // kDgradDown: saved accumulators [R, 2I]
    void* out;                // d_ab (layer dtype) or dx_sorted (fp32)
    float* scale_part;        // kDgradDown with scale_rows: [R, ceil(I / 256)]
    int R, d, I, E;
    int* status;
};
cudaError_t launch_dgrad_bf16(const DgradArgs& a, cudaStream_t s);
cudaError_t launch_dgrad_f32(const DgradArgs& a, cudaStream_t s);
// wgrad: dw[e] = a[rows of e]^T . b[rows of e], a [R, M], b [R, N] (layer dtype), dw fp32
// [E, M, N]; every expert's block is written (zero for an expert without rows).
struct WgradArgs {
    const void* a;
    const void* b;
    const int32_t* offsets;   // [E + 1] or nullptr
    int R, M, N, E;
    void* dw;                 // [E, M, N]: fp32, or bf16 when dw_bf16 (bf16 layers only)
    int* status;
    bool dw_bf16 = false;
};
cudaError_t launch_wgrad_bf16(const WgradArgs& a, cudaStream_t s);
cudaError_t launch_wgrad_f32(const WgradArgs& a, cudaStream_t s);
cudaError_t launch_combine_backward(const void* dout, bool bf16, const float* y_sorted,
                                    const int32_t* slot_to_sorted, const float* weights, int T,
                                    int d, int k, void* dy_sorted, float* d_weights,
                                    cudaStream_t s);
cudaError_t launch_scale_grad(const float* scale_part, int R, int n_tiles,
                              const int32_t* sorted_to_slot, float* d_weights, cudaStream_t s);
cudaError_t launch_route_backward(const float* logits, const int32_t* ids, const float* weights,
                                  const float* d_weights, int T, int E, int k, int score_fn,
                                  bool renorm, float* d_logits, cudaStream_t s);

}  // namespace rdg
