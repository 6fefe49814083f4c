// moe_dispatch_noalloc: moe_dispatch for callers that cannot allocate device memory.
//
// Some callers have no way to obtain device scratch at the call site: a plugin inside a host
// application that owns every device allocation and exposes no allocator to it, or a service
// that forbids any device allocation once it has started. moe_dispatch needs a caller-provided
// workspace for its per-chunk expert counts; this variant keeps that scratch in a fixed
// file-scope device array instead, so the caller passes only inputs and outputs.
//
// The array holds kNoallocScratchInts int32 (1 MiB). Every GPU that loads the library keeps
// it until the process exits. All calls share it and it keeps the last call's contents; the
// dispatch kernels overwrite every entry they read before reading it, so nothing has to start
// at zero. Calls whose kernels overlap on the GPU (for instance on two streams) race on the
// array and must be serialised by the caller.
//
// Host code cannot pass the array's name to a kernel (on the host it names a stand-in, not
// device memory), so the first call in each CUDA context looks up its device address with
// cudaGetSymbolAddress while that context is current and caches it; that first call should
// come before any stream capture. The module, and so the array, is loaded once per context:
// a caller that makes its own (non-primary) context current on a device gets that context's
// copy, not the primary context's. The cache is keyed on the context's unique id (cuCtxGetId),
// which a context created after cudaDeviceReset does not share with the one it replaces, so a
// reset context is looked up again instead of reusing a stale address.
#include <mutex>

#include "moe_internal.cuh"

namespace rdg {
namespace {

constexpr size_t kNoallocScratchInts = MOE_DISPATCH_NOALLOC_MAX_SCRATCH_INTS;

static __device__ __align__(256) int32_t g_dispatch_scratch[kNoallocScratchInts];

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

struct CtxFns {
    CtxGetCurrentFn get_current = nullptr;
    CtxGetIdFn get_id = nullptr;
};

// The two driver calls, resolved through the runtime (the library links no libcuda).
const CtxFns& ctx_fns() {
    static CtxFns f;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess && q == cudaDriverEntryPointSuccess)
            f.get_current = reinterpret_cast<CtxGetCurrentFn>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            f.get_id = reinterpret_cast<CtxGetIdFn>(p);
    });
    return f;
}

// Unique id of the current context; 0 with *has == false when none is current yet.
cudaError_t current_ctx_id(unsigned long long* id, bool* has) {
    const CtxFns& f = ctx_fns();
    if (!f.get_current || !f.get_id) return cudaErrorNotSupported;
    CUcontext ctx = nullptr;
    if (f.get_current(&ctx) != CUDA_SUCCESS) return cudaErrorDeviceUninitialized;
    *has = ctx != nullptr;
    *id = 0;
    if (ctx && f.get_id(ctx, id) != CUDA_SUCCESS) return cudaErrorDeviceUninitialized;
    return cudaSuccess;
}

constexpr int kMaxContexts = 64;
std::mutex g_mu;
struct CachedAddr {
    unsigned long long ctx_id;
    int32_t* addr;
};
CachedAddr g_cache[kMaxContexts];
int g_cached = 0;

// Device address of g_dispatch_scratch in the current context (looked up once per context).
cudaError_t scratch_in_current_context(int32_t** out) {
    unsigned long long id = 0;
    bool has = false;
    cudaError_t e = current_ctx_id(&id, &has);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(g_mu);
    if (has)
        for (int i = 0; i < g_cached; ++i)
            if (g_cache[i].ctx_id == id) {
                *out = g_cache[i].addr;
                return cudaSuccess;
            }
    // not cached (or no context yet: the runtime makes the device's primary context current
    // inside this call)
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_dispatch_scratch);
    if (e != cudaSuccess) return e;
    if (!has) {
        e = current_ctx_id(&id, &has);
        if (e != cudaSuccess) return e;
        if (!has) return cudaErrorDeviceUninitialized;
        for (int i = 0; i < g_cached; ++i)
            if (g_cache[i].ctx_id == id) {
                g_cache[i].addr = static_cast<int32_t*>(p);
                *out = g_cache[i].addr;
                return cudaSuccess;
            }
    }
    // a full table drops its oldest entry (it is looked up again if that context comes back)
    if (g_cached == kMaxContexts) {
        for (int i = 1; i < kMaxContexts; ++i) g_cache[i - 1] = g_cache[i];
        --g_cached;
    }
    g_cache[g_cached++] = {id, static_cast<int32_t*>(p)};
    *out = static_cast<int32_t*>(p);
    return cudaSuccess;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace rdg

using namespace rdg;

extern "C" moe_status moe_dispatch_noalloc(const int32_t* topk_ids, const void* x, moe_dtype dt,
                                           int T, int d, int E, int k, int32_t* counts,
                                           int32_t* offsets, int32_t* sorted_to_slot,
                                           int32_t* slot_to_sorted, void* x_sorted,
                                           moe_stream_t stream) {
    if (T < 0 || E < 1 || k < 1 || k > E) return MOE_ERR_INVALID_ARG;
    if (E > kMaxE || k > kMaxK) return MOE_ERR_UNSUPPORTED;
    if ((long long)T * k >= (1ll << 31)) return MOE_ERR_UNSUPPORTED;
    if (dt != MOE_F32 && dt != MOE_BF16) return MOE_ERR_INVALID_ARG;
    if ((x == nullptr) != (x_sorted == nullptr)) return MOE_ERR_INVALID_ARG;
    const int row_mult = dt == MOE_BF16 ? 8 : 4;
    if (x != nullptr && (d < 1 || d % row_mult != 0)) return MOE_ERR_INVALID_ARG;
    if (!counts || !offsets) return MOE_ERR_INVALID_ARG;
    if (T > 0 && (!topk_ids || !sorted_to_slot || !slot_to_sorted)) return MOE_ERR_INVALID_ARG;
    const void* ptrs[] = {topk_ids, x, counts, offsets, sorted_to_slot, slot_to_sorted, x_sorted};
    for (const void* q : ptrs)
        if (q && !aligned16(q)) return MOE_ERR_INVALID_ARG;
    // the fixed scratch holds one count per (256-slot chunk, expert)
    if (dispatch_scratch_bytes(T * k, E) > kNoallocScratchInts * sizeof(int32_t))
        return MOE_ERR_UNSUPPORTED;
    int32_t* scratch = nullptr;
    if (scratch_in_current_context(&scratch) != cudaSuccess) return MOE_ERR_CUDA;
    const size_t row_bytes = (size_t)d * (dt == MOE_BF16 ? 2 : 4);
    const cudaError_t e =
        launch_dispatch(topk_ids, x, row_bytes, T, E, k, counts, offsets, sorted_to_slot,
                        slot_to_sorted, x_sorted, scratch, nullptr, (cudaStream_t)stream);
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
