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
// device memory), so the first call on each device looks up its device address with
// cudaGetSymbolAddress while that device is current and caches it; that first call on a device
// should come before any stream capture.
#include <mutex>

#include "moe_internal.cuh"

namespace rdg {
namespace {

constexpr size_t kNoallocScratchInts = MOE_DISPATCH_NOALLOC_MAX_SCRATCH_INTS;

static __device__ __align__(256) int32_t g_dispatch_scratch[kNoallocScratchInts];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int32_t* g_scratch_addr[kMaxDevices] = {nullptr};

// Device address of g_dispatch_scratch on the current device (looked up once per device).
cudaError_t scratch_on_current_device(int32_t** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_scratch_addr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_dispatch_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = static_cast<int32_t*>(p);
    }
    *out = g_scratch_addr[dev];
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
    if (scratch_on_current_device(&scratch) != cudaSuccess) return MOE_ERR_CUDA;
    const size_t row_bytes = (size_t)d * (dt == MOE_BF16 ? 2 : 4);
    const cudaError_t e =
        launch_dispatch(topk_ids, x, row_bytes, T, E, k, counts, offsets, sorted_to_slot,
                        slot_to_sorted, x_sorted, scratch, nullptr, (cudaStream_t)stream);
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
