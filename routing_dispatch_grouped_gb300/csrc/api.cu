// C ABI of libmoe: argument checks, workspace layout and the launch chain of each entry point.
// Every check runs before anything is enqueued (Expert parallelism page, "Overriding the
// plans": errors are raised before any work). No call allocates, frees or synchronises, except
// moe_read_device_status, which exists to synchronise.
#include <atomic>
#include <mutex>
#include <set>
#include <utility>

#include "moe_internal.cuh"

namespace rdg {

namespace {
thread_local bool t_pdl = false;
}
bool pdl_enabled() { return t_pdl; }
PdlScope::PdlScope(bool on) : prev(t_pdl) { t_pdl = on; }
PdlScope::~PdlScope() { t_pdl = prev; }

int device_sm_count() {
    static std::atomic<int> cache[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    int n = cache[dev].load(std::memory_order_relaxed);
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 148;
        cache[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

cudaError_t ensure_max_dynamic_smem(const void* fn, int bytes) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    static std::mutex mu;
    static std::set<std::pair<const void*, int>> done;  // (kernel, device)
    std::lock_guard<std::mutex> lock(mu);
    if (done.count({fn, dev})) return cudaSuccess;
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done.insert({fn, dev});
    return e;
}

namespace {
std::atomic<uint32_t> g_gemm_stall_ns{0};
}

uint32_t debug_gemm_stall_ns() { return g_gemm_stall_ns.load(std::memory_order_relaxed); }

}  // namespace rdg

using namespace rdg;

extern "C" void moe_debug_set_gemm_stall_ns(uint32_t ns) {
    g_gemm_stall_ns.store(ns, std::memory_order_relaxed);
}

namespace {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned256(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 255u) == 0; }
inline size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
inline size_t dtype_bytes(moe_dtype dt) { return dt == MOE_BF16 ? 2 : 4; }
inline bool dtype_ok(moe_dtype dt) { return dt == MOE_F32 || dt == MOE_BF16; }
inline int row_multiple(moe_dtype dt) { return dt == MOE_BF16 ? 8 : 4; }

// Common range checks on (T, E, k).
moe_status check_tek(int T, int E, int k) {
    if (T < 0 || E < 1 || k < 1) return MOE_ERR_INVALID_ARG;
    if (k > E) return MOE_ERR_INVALID_ARG;
    if (E > kMaxE || k > kMaxK) return MOE_ERR_UNSUPPORTED;
    if ((long long)T * k >= (1ll << 31)) return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}

moe_status launch_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

// fp32 grouped GEMM grid height is (R / 32 + E) blocks.
constexpr long long kMaxRowsF32 = 60000ll * 32;

struct ForwardLayout {
    size_t fcnt, counts, offsets, chunk, s2p, p2s, x_sorted, h, y, h_sh, y_sh, fused, ab, ab_sh,
        x_q, w_gu, w_dn, w_sgu, w_sdn, h_codes, h_scales, total;
};

// train: the layout of moe_forward_train (no one-kernel decode path; the gate/up accumulators
// of the routed rows and of the shared expert are kept for the backward pass, after the rest)
// mx: the layout of moe_forward_mx. Decode batches run the one-kernel layer on the MX weights:
// after its partial sums, h's MXFP8 codes [R, I] and scales [R, ceil(I / 32)]. Other batches:
// after the rest, x rounded to MXFP8 [T, d] and the dequantized bf16 weights of the routed and
// the shared experts.
ForwardLayout forward_layout(int T, int d, int E, int k, int I, int Is, moe_dtype dt,
                             bool train = false, bool mx = false) {
    const size_t R = (size_t)T * k, b = dtype_bytes(dt);
    ForwardLayout L;
    size_t o = kStatusBytes;
    auto take = [&](size_t bytes) {
        const size_t at = o;
        o = round_up(o + bytes, 256);
        return at;
    };
    // the fused decode kernel's counters follow the status word (one memset clears both);
    // its partial sums go last
    const bool fused = !train && decode_fused_applies(dt, T, k, Is);
    const DecodeFusedLayout F = decode_fused_layout(T, d, k, I, mx);
    L.fcnt = take(fused ? F.counter_bytes : 0);
    L.counts = take((size_t)E * 4);
    L.offsets = take((size_t)(E + 1) * 4);
    L.chunk = take(dispatch_scratch_bytes((int)R, E));
    L.s2p = take(R * 4);
    L.p2s = take(R * 4);
    L.x_sorted = take(R * d * b);
    L.h = take(R * (size_t)I * b);
    L.y = take(R * (size_t)d * 4);
    L.h_sh = take(Is > 0 ? (size_t)T * Is * b : 0);
    L.y_sh = take(Is > 0 ? (size_t)T * d * 4 : 0);
    L.fused = take(fused ? F.part_bytes : 0);
    L.ab = take(train ? R * 2 * (size_t)I * b : 0);
    L.ab_sh = take(train && Is > 0 ? (size_t)T * 2 * Is * b : 0);
    const bool mx_chain = mx && !fused;
    L.x_q = take(mx_chain ? (size_t)T * d * 2 : 0);
    L.w_gu = take(mx_chain ? (size_t)E * d * 2 * I * 2 : 0);
    L.w_dn = take(mx_chain ? (size_t)E * I * d * 2 : 0);
    L.w_sgu = take(mx_chain ? (size_t)d * 2 * Is * 2 : 0);
    L.w_sdn = take(mx_chain ? (size_t)Is * d * 2 : 0);
    L.h_codes = take(mx && fused ? R * (size_t)I : 0);
    L.h_scales = take(mx && fused ? R * (size_t)((I + 31) / 32) : 0);
    L.total = o;
    return L;
}

struct BackwardLayout {
    size_t dy, d_ab, dx_sorted, part, dw_tmp, d_ab_sh, dx_sh, total;
};

// moe_backward's workspace: status word, dy_sorted, d_ab, dx_sorted, the router-score partial
// sums, a [T, k] buffer for the routing weights' gradient (when the caller wants only the
// logits'), and the shared expert's d_ab and dx, each rounded up to 256 bytes
BackwardLayout backward_layout(int T, int d, int k, int I, int Is, moe_dtype dt) {
    const size_t R = (size_t)T * k, b = dtype_bytes(dt);
    BackwardLayout L;
    size_t o = kStatusBytes;
    auto take = [&](size_t bytes) {
        const size_t at = o;
        o = round_up(o + bytes, 256);
        return at;
    };
    L.dy = take(R * d * b);
    L.d_ab = take(R * 2 * (size_t)I * b);
    L.dx_sorted = take(R * d * 4);
    L.part = take(R * (size_t)((I + 31) / 32) * 4);
    L.dw_tmp = take(R * 4);
    L.d_ab_sh = take(Is > 0 ? (size_t)T * 2 * Is * b : 0);
    L.dx_sh = take(Is > 0 ? (size_t)T * d * 4 : 0);
    L.total = o;
    return L;
}

moe_status clear_status(void* workspace, cudaStream_t s) {
    return launch_status(cudaMemsetAsync(workspace, 0, sizeof(int), s));
}

moe_status run_gemm(GemmKind kind, const void* a, const void* b, bool packed,
                    const int32_t* offsets, const int32_t* s2p, const float* w, bool scale,
                    moe_dtype dt, int R, int K, int N, int E, void* out, int* status,
                    cudaStream_t s, void* ab = nullptr, bool mx_h = false) {
    GroupedGemmArgs g;
    g.kind = kind;
    g.a = a;
    g.b = b;
    g.packed = packed;
    g.offsets = offsets;
    g.sorted_to_slot = s2p;
    g.topk_weights = w;
    g.scale_rows = (kind == kGateUp) && scale;
    g.weight_rows = (kind == kDown) && scale;
    g.R = R;
    g.K = K;
    g.N = N;
    g.E = E;
    g.out = out;
    g.status = status;
    g.ab = ab;
    g.mx_h = mx_h;
    const cudaError_t e =
        dt == MOE_BF16 ? launch_grouped_gemm_bf16(g, s) : launch_grouped_gemm_f32(g, s);
    return launch_status(e);
}

// Checks shared by moe_gate_up / moe_down / moe_experts.
moe_status check_experts_args(const int32_t* offsets, const int32_t* s2p, const float* w,
                              bool need_w, moe_dtype dt, int R, int d, int E, int I,
                              void* workspace, size_t ws_bytes) {
    if (!dtype_ok(dt)) return MOE_ERR_INVALID_ARG;
    if (R < 0 || d < 1 || I < 1 || E < 1) return MOE_ERR_INVALID_ARG;
    if (E > kMaxE) return MOE_ERR_UNSUPPORTED;
    if (offsets == nullptr && E != 1) return MOE_ERR_INVALID_ARG;
    if (d % row_multiple(dt) != 0 || I % row_multiple(dt) != 0) return MOE_ERR_INVALID_ARG;
    if (need_w && (s2p == nullptr || w == nullptr)) return MOE_ERR_INVALID_ARG;
    if (offsets && !aligned16(offsets)) return MOE_ERR_INVALID_ARG;
    if (dt == MOE_F32 && R > kMaxRowsF32) return MOE_ERR_UNSUPPORTED;
    if (workspace == nullptr || !aligned256(workspace) || ws_bytes < kStatusBytes)
        return MOE_ERR_WORKSPACE;
    return MOE_OK;
}

}  // namespace

extern "C" {

const char* moe_status_string(moe_status st) {
    switch (st) {
        case MOE_OK: return "MOE_OK";
        case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG: invalid argument";
        case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED: shape or dtype not supported";
        case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE: workspace missing, misaligned or too small";
        case MOE_ERR_CUDA: return "MOE_ERR_CUDA: a CUDA call or kernel launch failed";
        case MOE_ERR_DEVICE_BOUNDS: return "MOE_ERR_DEVICE_BOUNDS: expert id outside [0, E)";
        case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT: a device-side wait timed out";
    }
    return "unknown moe_status";
}

moe_status moe_route(const float* logits, int T, int E, int k, moe_score_fn score_fn,
                     unsigned flags, int32_t* topk_ids, float* topk_weights,
                     moe_stream_t stream) {
    moe_status st = check_tek(T, E, k);
    if (st != MOE_OK) return st;
    if (score_fn != MOE_SCORE_SOFTMAX && score_fn != MOE_SCORE_SIGMOID) return MOE_ERR_INVALID_ARG;
    if (flags & ~(unsigned)MOE_RENORMALIZE) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    if (!logits || !topk_ids || !topk_weights) return MOE_ERR_INVALID_ARG;
    if (!aligned16(logits) || !aligned16(topk_ids) || !aligned16(topk_weights))
        return MOE_ERR_INVALID_ARG;
    return launch_status(launch_route(logits, T, E, k, (int)score_fn,
                                      (flags & MOE_RENORMALIZE) != 0, topk_ids, topk_weights,
                                      (cudaStream_t)stream));
}

moe_status moe_route_hidden(const void* x, moe_dtype dt, const float* w_router,
                            const float* bias, int T, int d, int E, int k,
                            moe_score_fn score_fn, unsigned flags, float* logits,
                            int32_t* topk_ids, float* topk_weights, moe_stream_t stream) {
    moe_status st = check_tek(T, E, k);
    if (st != MOE_OK) return st;
    if (!dtype_ok(dt) || d < 1) return MOE_ERR_INVALID_ARG;
    if (score_fn != MOE_SCORE_SOFTMAX && score_fn != MOE_SCORE_SIGMOID) return MOE_ERR_INVALID_ARG;
    if (flags & ~(unsigned)MOE_RENORMALIZE) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    if (!x || !w_router || !topk_ids || !topk_weights) return MOE_ERR_INVALID_ARG;
    const void* ptrs[] = {x, w_router, bias, logits, topk_ids, topk_weights};
    for (const void* q : ptrs)
        if (q && !aligned16(q)) return MOE_ERR_INVALID_ARG;
    return launch_status(launch_route_hidden(x, dt == MOE_BF16, w_router, bias, T, d, E, k,
                                             (int)score_fn, (flags & MOE_RENORMALIZE) != 0,
                                             logits, topk_ids, topk_weights,
                                             (cudaStream_t)stream));
}

size_t moe_dispatch_workspace_size(int T, int E, int k) {
    if (T < 0 || E < 1 || k < 1) return 0;
    return kStatusBytes + round_up(dispatch_scratch_bytes(T * k, E), 256);
}

moe_status moe_dispatch(const int32_t* topk_ids, const void* x, moe_dtype dt, int T, int d, int E,
                        int k, int32_t* counts, int32_t* offsets, int32_t* sorted_to_slot,
                        int32_t* slot_to_sorted, void* x_sorted, void* workspace,
                        size_t ws_bytes, moe_stream_t stream) {
    moe_status st = check_tek(T, E, k);
    if (st != MOE_OK) return st;
    if (!dtype_ok(dt)) return MOE_ERR_INVALID_ARG;
    if ((x == nullptr) != (x_sorted == nullptr)) return MOE_ERR_INVALID_ARG;
    if (x != nullptr && (d < 1 || d % row_multiple(dt) != 0)) return MOE_ERR_INVALID_ARG;
    if (!counts || !offsets) return MOE_ERR_INVALID_ARG;
    if (T > 0 && (!topk_ids || !sorted_to_slot || !slot_to_sorted)) return MOE_ERR_INVALID_ARG;
    const void* ptrs[] = {topk_ids, x, counts, offsets, sorted_to_slot, slot_to_sorted, x_sorted};
    for (const void* q : ptrs)
        if (q && !aligned16(q)) return MOE_ERR_INVALID_ARG;
    if (!workspace || !aligned256(workspace) || ws_bytes < moe_dispatch_workspace_size(T, E, k))
        return MOE_ERR_WORKSPACE;
    cudaStream_t s = (cudaStream_t)stream;
    st = clear_status(workspace, s);
    if (st != MOE_OK) return st;
    int32_t* chunk = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(workspace) + kStatusBytes);
    return launch_status(launch_dispatch(topk_ids, x, (size_t)d * dtype_bytes(dt), T, E, k, counts,
                                         offsets, sorted_to_slot, slot_to_sorted, x_sorted, chunk,
                                         static_cast<int*>(workspace), s));
}

size_t moe_experts_workspace_size(void) { return kStatusBytes; }

moe_status moe_gate_up(const void* x_rows, const int32_t* offsets, const int32_t* sorted_to_slot,
                       const float* topk_weights, moe_dtype dt, int R, int d, int E, int I,
                       const void* w_gate_up, unsigned flags, void* h, void* workspace,
                       size_t ws_bytes, moe_stream_t stream) {
    if (flags & ~(unsigned)(MOE_SCALE_INPUT | MOE_WEIGHTS_PACKED)) return MOE_ERR_INVALID_ARG;
    const bool scale = (flags & MOE_SCALE_INPUT) != 0;
    const bool packed = (flags & MOE_WEIGHTS_PACKED) != 0;
    if (packed && dt != MOE_BF16) return MOE_ERR_UNSUPPORTED;
    moe_status st = check_experts_args(offsets, sorted_to_slot, topk_weights, scale, dt, R, d, E,
                                       I, workspace, ws_bytes);
    if (st != MOE_OK) return st;
    if (R == 0) return MOE_OK;
    if (!x_rows || !w_gate_up || !h) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x_rows) || !aligned16(w_gate_up) || !aligned16(h)) return MOE_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    st = clear_status(workspace, s);
    if (st != MOE_OK) return st;
    return run_gemm(kGateUp, x_rows, w_gate_up, packed, offsets, sorted_to_slot, topk_weights,
                    scale, dt, R, d, I, E, h, static_cast<int*>(workspace), s);
}

moe_status moe_down(const void* h, const int32_t* offsets, const int32_t* sorted_to_slot,
                    const float* topk_weights, moe_dtype dt, int R, int d, int E, int I,
                    const void* w_down, unsigned flags, float* y_sorted, void* workspace,
                    size_t ws_bytes, moe_stream_t stream) {
    if (flags & ~(unsigned)(MOE_FUSE_COMBINE_WEIGHT | MOE_WEIGHTS_PACKED))
        return MOE_ERR_INVALID_ARG;
    const bool weight = (flags & MOE_FUSE_COMBINE_WEIGHT) != 0;
    const bool packed = (flags & MOE_WEIGHTS_PACKED) != 0;
    if (packed && dt != MOE_BF16) return MOE_ERR_UNSUPPORTED;
    moe_status st = check_experts_args(offsets, sorted_to_slot, topk_weights, weight, dt, R, d, E,
                                       I, workspace, ws_bytes);
    if (st != MOE_OK) return st;
    if (R == 0) return MOE_OK;
    if (!h || !w_down || !y_sorted) return MOE_ERR_INVALID_ARG;
    if (!aligned16(h) || !aligned16(w_down) || !aligned16(y_sorted)) return MOE_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    st = clear_status(workspace, s);
    if (st != MOE_OK) return st;
    return run_gemm(kDown, h, w_down, packed, offsets, sorted_to_slot, topk_weights, weight, dt,
                    R, I, d, E, y_sorted, static_cast<int*>(workspace), s);
}

moe_status moe_experts(const void* x_sorted, const int32_t* offsets, const int32_t* sorted_to_slot,
                       const float* topk_weights, moe_dtype dt, int R, int d, int E, int I,
                       const void* w_gate_up, const void* w_down, unsigned flags, void* h,
                       float* y_sorted, void* workspace, size_t ws_bytes, moe_stream_t stream) {
    if (flags & ~(unsigned)(MOE_SCALE_INPUT | MOE_FUSE_COMBINE_WEIGHT | MOE_WEIGHTS_PACKED))
        return MOE_ERR_INVALID_ARG;
    if ((flags & MOE_SCALE_INPUT) && (flags & MOE_FUSE_COMBINE_WEIGHT)) return MOE_ERR_INVALID_ARG;
    const bool packed = (flags & MOE_WEIGHTS_PACKED) != 0;
    if (packed && dt != MOE_BF16) return MOE_ERR_UNSUPPORTED;
    const bool any_w = (flags & (MOE_SCALE_INPUT | MOE_FUSE_COMBINE_WEIGHT)) != 0;
    moe_status st = check_experts_args(offsets, sorted_to_slot, topk_weights, any_w, dt, R, d, E,
                                       I, workspace, ws_bytes);
    if (st != MOE_OK) return st;
    if (R == 0) return MOE_OK;
    if (!x_sorted || !w_gate_up || !w_down || !h || !y_sorted) return MOE_ERR_INVALID_ARG;
    const void* ptrs[] = {x_sorted, w_gate_up, w_down, h, y_sorted};
    for (const void* q : ptrs)
        if (!aligned16(q)) return MOE_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    st = clear_status(workspace, s);
    if (st != MOE_OK) return st;
    int* status = static_cast<int*>(workspace);
    st = run_gemm(kGateUp, x_sorted, w_gate_up, packed, offsets, sorted_to_slot, topk_weights,
                  (flags & MOE_SCALE_INPUT) != 0, dt, R, d, I, E, h, status, s);
    if (st != MOE_OK) return st;
    return run_gemm(kDown, h, w_down, packed, offsets, sorted_to_slot, topk_weights,
                    (flags & MOE_FUSE_COMBINE_WEIGHT) != 0, dt, R, I, d, E, y_sorted, status, s);
}

size_t moe_packed_weights_size(moe_weight_kind kind, int E, int K, int N, moe_dtype dt) {
    if ((kind != MOE_W_GATE_UP && kind != MOE_W_DOWN) || dt != MOE_BF16) return 0;
    if (E < 1 || K < 1 || N < 1) return 0;
    const PackedGeom g = packed_geom(kind == MOE_W_GATE_UP ? kGateUp : kDown, K, N);
    return (size_t)E * g.nb * g.kpad * 64 * 2;
}

moe_status moe_pack_weights(moe_weight_kind kind, const void* w, void* packed, moe_dtype dt,
                            int E, int K, int N, moe_stream_t stream) {
    if (kind != MOE_W_GATE_UP && kind != MOE_W_DOWN) return MOE_ERR_INVALID_ARG;
    if (!dtype_ok(dt)) return MOE_ERR_INVALID_ARG;
    if (dt != MOE_BF16) return MOE_ERR_UNSUPPORTED;
    if (E < 1 || K < 1 || N < 1 || N % 8 != 0) return MOE_ERR_INVALID_ARG;
    if (!w || !packed || !aligned16(w) || !aligned16(packed)) return MOE_ERR_INVALID_ARG;
    if (moe_packed_weights_size(kind, E, K, N, dt) / 128 >= (1ull << 31))
        return MOE_ERR_UNSUPPORTED;  // packed rows are addressed with 32-bit coordinates
    return launch_status(launch_pack_weights(kind == MOE_W_GATE_UP ? kGateUp : kDown, w, packed,
                                             E, K, N, (cudaStream_t)stream));
}

moe_status moe_combine(const float* y_sorted, const int32_t* slot_to_sorted,
                       const float* topk_weights, const float* y_shared, int T, int d, int k,
                       moe_dtype out_dt, void* out, moe_stream_t stream) {
    if (T < 0 || k < 1 || d < 1) return MOE_ERR_INVALID_ARG;
    if (k > kMaxK) return MOE_ERR_UNSUPPORTED;
    if ((long long)T * k >= (1ll << 31)) return MOE_ERR_UNSUPPORTED;
    if (!dtype_ok(out_dt)) return MOE_ERR_INVALID_ARG;
    if (d % row_multiple(out_dt) != 0) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    if (!y_sorted || !slot_to_sorted || !out) return MOE_ERR_INVALID_ARG;
    const void* ptrs[] = {y_sorted, slot_to_sorted, topk_weights, y_shared, out};
    for (const void* q : ptrs)
        if (q && !aligned16(q)) return MOE_ERR_INVALID_ARG;
    return launch_status(launch_combine(y_sorted, slot_to_sorted, topk_weights, y_shared, T, d, k,
                                        out_dt == MOE_BF16, out, (cudaStream_t)stream));
}

size_t moe_forward_workspace_size(int T, int d, int E, int k, int I, int Is, moe_dtype dt) {
    if (T < 0 || d < 1 || E < 1 || k < 1 || I < 1 || Is < 0 || !dtype_ok(dt)) return 0;
    return forward_layout(T, d, E, k, I, Is, dt).total;
}

int moe_forward_kernel_count(moe_dtype dt, int T, int k, int Is) {
    if (T <= 0 || k <= 0) return 0;
    if (decode_fused_applies(dt, T, k, Is)) return 1;
    const bool small = (long long)T * k <= kSmallDispatchMaxSlots;
    const int front = small ? 2 : 1 + dispatch_kernel_count(true);
    return front + 2 + (Is > 0 ? 2 : 0) + 1;
}

const char* moe_gemm_kernel_name(moe_weight_kind kind, int R, int E, int grouped) {
    if (R <= 0 || E < 1 || (kind != MOE_W_GATE_UP && kind != MOE_W_DOWN)) return "none";
    switch (pick_grouped_gemm_bf16(kind == MOE_W_GATE_UP ? kGateUp : kDown, R,
                                   grouped ? E : 1, false)) {
        case kPickRows: return "tc_grouped_gemm";
        case kPick2sm: return "tc_grouped_gemm_2sm";
        case kPickSwapPair: return "tc_grouped_gemm_swap_pair";
        default: return "tc_grouped_gemm_swap";
    }
}

// moe_forward, and with train = true moe_forward_train
static moe_status forward_impl(const void* x, const float* logits, moe_dtype dt, int T, int d,
                               int E, int k, int I, moe_score_fn score_fn, unsigned flags,
                               const void* w_gate_up, const void* w_down,
                               const void* w_shared_gate_up, const void* w_shared_down, int Is,
                               int32_t* topk_ids, float* topk_weights, void* out,
                               void* workspace, size_t ws_bytes, moe_stream_t stream,
                               bool train, bool mx = false) {
    moe_status st = check_tek(T, E, k);
    if (st != MOE_OK) return st;
    if (!dtype_ok(dt)) return MOE_ERR_INVALID_ARG;
    if (score_fn != MOE_SCORE_SOFTMAX && score_fn != MOE_SCORE_SIGMOID) return MOE_ERR_INVALID_ARG;
    if (flags & ~(unsigned)(MOE_RENORMALIZE | MOE_SCALE_INPUT | MOE_FUSE_COMBINE_WEIGHT |
                            MOE_WEIGHTS_PACKED))
        return MOE_ERR_INVALID_ARG;
    const bool scale = (flags & MOE_SCALE_INPUT) != 0;
    const bool fuse_w = (flags & MOE_FUSE_COMBINE_WEIGHT) != 0;
    const bool packed = (flags & MOE_WEIGHTS_PACKED) != 0;
    if (packed && dt != MOE_BF16) return MOE_ERR_UNSUPPORTED;
    if (mx && (dt != MOE_BF16 || packed || train)) return MOE_ERR_UNSUPPORTED;
    if (scale && fuse_w) return MOE_ERR_INVALID_ARG;
    // training keeps y_sorted unweighted: the routing weights' gradient reads it
    if (train && fuse_w) return MOE_ERR_UNSUPPORTED;
    if (d < 1 || I < 1 || Is < 0) return MOE_ERR_INVALID_ARG;
    if (d % row_multiple(dt) != 0 || I % row_multiple(dt) != 0 || Is % row_multiple(dt) != 0)
        return MOE_ERR_INVALID_ARG;
    const bool shared = w_shared_gate_up != nullptr || w_shared_down != nullptr;
    if (shared != (Is > 0)) return MOE_ERR_INVALID_ARG;
    if (shared && (!w_shared_gate_up || !w_shared_down)) return MOE_ERR_INVALID_ARG;
    if (dt == MOE_F32 && ((long long)T * k > kMaxRowsF32)) return MOE_ERR_UNSUPPORTED;
    if (T == 0) return MOE_OK;
    if (!x || !logits || !w_gate_up || !w_down || !topk_ids || !topk_weights || !out)
        return MOE_ERR_INVALID_ARG;
    const void* ptrs[] = {x, logits, w_gate_up, w_down, w_shared_gate_up, w_shared_down,
                          topk_ids, topk_weights, out};
    for (const void* q : ptrs)
        if (q && !aligned16(q)) return MOE_ERR_INVALID_ARG;
    const ForwardLayout L = forward_layout(T, d, E, k, I, Is, dt, train, mx);
    if (!workspace || !aligned256(workspace) || ws_bytes < L.total) return MOE_ERR_WORKSPACE;

    cudaStream_t s = (cudaStream_t)stream;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    int* status = reinterpret_cast<int*>(ws);
    int32_t* counts = reinterpret_cast<int32_t*>(ws + L.counts);
    int32_t* offsets = reinterpret_cast<int32_t*>(ws + L.offsets);
    int32_t* chunk = reinterpret_cast<int32_t*>(ws + L.chunk);
    int32_t* s2p = reinterpret_cast<int32_t*>(ws + L.s2p);
    int32_t* p2s = reinterpret_cast<int32_t*>(ws + L.p2s);
    void* xs = ws + L.x_sorted;
    void* h = ws + L.h;
    float* y = reinterpret_cast<float*>(ws + L.y);
    void* h_sh = ws + L.h_sh;
    float* y_sh = reinterpret_cast<float*>(ws + L.y_sh);
    const int R = T * k;

    const bool renorm = (flags & MOE_RENORMALIZE) != 0;
    // MX layers: x rounded to MXFP8 once per token (the routed rows are copies of it); the
    // one-kernel decode layer rounds its own
    const bool fused = !train && decode_fused_applies(dt, T, k, Is);
    const void* x_in = x;
    if (mx && !fused) {
        if ((st = clear_status(workspace, s)) != MOE_OK) return st;
        if ((st = launch_status(launch_mx_rows(x, T, d, ws + L.x_q, nullptr, nullptr, s))) !=
            MOE_OK)
            return st;
        x_in = ws + L.x_q;
    }
    if (fused) {
        // decode: the whole layer in one cooperative kernel; its counters sit right after the
        // status word and are cleared with it
        if ((st = launch_status(cudaMemsetAsync(workspace, 0, L.counts, s))) != MOE_OK)
            return st;
        DecodeFusedArgs a;
        a.x = x;
        a.logits = logits;
        a.w_gate_up = w_gate_up;
        a.w_down = w_down;
        a.packed = packed;
        a.score_fn = (int)score_fn;
        a.renorm = renorm;
        a.scale_input = scale;
        a.T = T;
        a.d = d;
        a.E = E;
        a.k = k;
        a.I = I;
        a.topk_ids = topk_ids;
        a.topk_weights = topk_weights;
        a.counts = counts;
        a.offsets = offsets;
        a.sorted_to_slot = s2p;
        a.slot_to_sorted = p2s;
        a.h = h;
        a.out = out;
        a.counters = reinterpret_cast<int*>(ws + L.fcnt);
        a.partials = ws + L.fused;
        a.status = status;
        a.mx = mx;
        if (mx) {
            a.h_codes = ws + L.h_codes;
            a.h_scales = ws + L.h_scales;
        }
        return launch_status(launch_decode_fused(a, s));
    }
    if (!(mx && !fused) && (st = clear_status(workspace, s)) != MOE_OK) return st;
    if (R <= kSmallDispatchMaxSlots) {
        // few tokens: route and the dispatch indices in one launch, then the row copy
        if ((st = launch_status(launch_route_dispatch_small(logits, T, E, k, (int)score_fn,
                                                            renorm, topk_ids, topk_weights,
                                                            counts, offsets, s2p, p2s, s))) !=
            MOE_OK)
            return st;
    } else {
        if ((st = launch_status(launch_route(logits, T, E, k, (int)score_fn, renorm, topk_ids,
                                             topk_weights, s))) != MOE_OK)
            return st;
    }
    PdlScope pdl(true);
    if (R <= kSmallDispatchMaxSlots) {
        if ((st = launch_status(launch_dispatch_copy(x_in, (size_t)d * dtype_bytes(dt), T, k,
                                                     p2s, xs, s))) != MOE_OK)
            return st;
    } else {
        if ((st = launch_status(launch_dispatch(topk_ids, x_in, (size_t)d * dtype_bytes(dt), T,
                                                E, k, counts, offsets, s2p, p2s, xs, chunk,
                                                status, s))) != MOE_OK)
            return st;
    }
    // MX layers: the experts that received rows get their weights dequantized to bf16 (exact)
    const void* wgu = w_gate_up;
    const void* wdn = w_down;
    const void* wsgu = w_shared_gate_up;
    const void* wsdn = w_shared_down;
    if (mx) {
        if ((st = launch_status(launch_mx_dequant_weights(true, w_gate_up, E, d, I, offsets,
                                                          ws + L.w_gu, s))) != MOE_OK ||
            (st = launch_status(launch_mx_dequant_weights(false, w_down, E, I, d, offsets,
                                                          ws + L.w_dn, s))) != MOE_OK)
            return st;
        wgu = ws + L.w_gu;
        wdn = ws + L.w_dn;
        if (shared) {
            if ((st = launch_status(launch_mx_dequant_weights(
                     true, w_shared_gate_up, 1, d, Is, nullptr, ws + L.w_sgu, s))) != MOE_OK ||
                (st = launch_status(launch_mx_dequant_weights(false, w_shared_down, 1, Is, d,
                                                              nullptr, ws + L.w_sdn, s))) !=
                    MOE_OK)
                return st;
            wsgu = ws + L.w_sgu;
            wsdn = ws + L.w_sdn;
        }
    }
    if ((st = run_gemm(kGateUp, xs, wgu, packed, offsets, s2p, topk_weights, scale, dt, R, d, I,
                       E, h, status, s, train ? ws + L.ab : nullptr, mx)) != MOE_OK)
        return st;
    if ((st = run_gemm(kDown, h, wdn, packed, offsets, s2p, topk_weights, fuse_w, dt, R, I, d, E,
                       y, status, s)) != MOE_OK)
        return st;
    if (shared) {
        if ((st = run_gemm(kGateUp, x_in, wsgu, packed, nullptr, nullptr, nullptr, false, dt, T,
                           d, Is, 1, h_sh, status, s, train ? ws + L.ab_sh : nullptr, mx)) !=
            MOE_OK)
            return st;
        if ((st = run_gemm(kDown, h_sh, wsdn, packed, nullptr, nullptr, nullptr, false, dt, T,
                           Is, d, 1, y_sh, status, s)) != MOE_OK)
            return st;
    }
    const float* comb_w = (scale || fuse_w) ? nullptr : topk_weights;
    return launch_status(launch_combine(y, p2s, comb_w, shared ? y_sh : nullptr, T, d, k,
                                        dt == MOE_BF16, out, s));
}

moe_status moe_forward(const void* x, const float* logits, moe_dtype dt, int T, int d, int E,
                       int k, int I, moe_score_fn score_fn, unsigned flags, const void* w_gate_up,
                       const void* w_down, const void* w_shared_gate_up,
                       const void* w_shared_down, int Is, int32_t* topk_ids, float* topk_weights,
                       void* out, void* workspace, size_t ws_bytes, moe_stream_t stream) {
    return forward_impl(x, logits, dt, T, d, E, k, I, score_fn, flags, w_gate_up, w_down,
                        w_shared_gate_up, w_shared_down, Is, topk_ids, topk_weights, out,
                        workspace, ws_bytes, stream, false);
}

moe_status moe_forward_train(const void* x, const float* logits, moe_dtype dt, int T, int d,
                             int E, int k, int I, moe_score_fn score_fn, unsigned flags,
                             const void* w_gate_up, const void* w_down,
                             const void* w_shared_gate_up, const void* w_shared_down, int Is,
                             int32_t* topk_ids, float* topk_weights, void* out, void* workspace,
                             size_t ws_bytes, moe_stream_t stream) {
    return forward_impl(x, logits, dt, T, d, E, k, I, score_fn, flags, w_gate_up, w_down,
                        w_shared_gate_up, w_shared_down, Is, topk_ids, topk_weights, out,
                        workspace, ws_bytes, stream, true);
}

// moe_forward_host: the forward workspace, then device staging for x, logits, out, ids, weights
struct HostLayout {
    size_t fwd, x, logits, out, ids, w, total;
};
static HostLayout host_layout(int T, int d, int E, int k, int I, int Is, moe_dtype dt) {
    HostLayout L;
    const size_t b = dt == MOE_BF16 ? 2 : 4;
    L.fwd = forward_layout(T, d, E, k, I, Is, dt).total;
    size_t o = round_up(L.fwd, 256);
    auto take = [&](size_t n) {
        const size_t at = o;
        o += round_up(n, 256);
        return at;
    };
    L.x = take((size_t)T * d * b);
    L.logits = take((size_t)T * E * 4);
    L.out = take((size_t)T * d * b);
    L.ids = take((size_t)T * k * 4);
    L.w = take((size_t)T * k * 4);
    L.total = o;
    return L;
}

size_t moe_forward_host_workspace_size(int T, int d, int E, int k, int I, int Is, moe_dtype dt) {
    if (T < 0 || d < 1 || E < 1 || k < 1 || I < 1 || Is < 0 || !dtype_ok(dt)) return 0;
    return host_layout(T, d, E, k, I, Is, dt).total;
}

// Device address of a page-locked, mapped host buffer (one the GPU reaches over NVLink-C2C),
// or nullptr for pageable or device memory and on a failed query.
static void* mapped_host_address(const void* p) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        (void)cudaGetLastError();
        return nullptr;
    }
    return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}

moe_status moe_forward_host(const void* x_host, const float* logits_host, moe_dtype dt, int T,
                            int d, int E, int k, int I, moe_score_fn score_fn, unsigned flags,
                            const void* w_gate_up, const void* w_down,
                            const void* w_shared_gate_up, const void* w_shared_down, int Is,
                            void* out_host, void* workspace, size_t ws_bytes,
                            moe_stream_t stream) {
    moe_status st = check_tek(T, E, k);
    if (st != MOE_OK) return st;
    if (!dtype_ok(dt) || d < 1 || I < 1 || Is < 0) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    if (!x_host || !logits_host || !out_host) return MOE_ERR_INVALID_ARG;
    const HostLayout L = host_layout(T, d, E, k, I, Is, dt);
    if (!workspace || !aligned256(workspace) || ws_bytes < L.total) return MOE_ERR_WORKSPACE;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    cudaStream_t s = (cudaStream_t)stream;
    const size_t b = dt == MOE_BF16 ? 2 : 4;
    // A page-locked buffer is used in place: the route kernel reads the logits, the dispatch
    // (or the decode kernel) reads x and the combine writes out across NVLink-C2C, each once
    // and in token order, so no staging copy runs for it. x is staged whenever a shared
    // expert runs: its gate_up loads x through TMA, which is kept to device memory.
    const void* x_dev = Is == 0 ? mapped_host_address(x_host) : nullptr;
    const void* logits_dev = mapped_host_address(logits_host);
    void* out_dev = mapped_host_address(out_host);
    if (!x_dev) {
        if ((st = launch_status(cudaMemcpyAsync(ws + L.x, x_host, (size_t)T * d * b,
                                                cudaMemcpyHostToDevice, s))) != MOE_OK)
            return st;
        x_dev = ws + L.x;
    }
    if (!logits_dev) {
        if ((st = launch_status(cudaMemcpyAsync(ws + L.logits, logits_host, (size_t)T * E * 4,
                                                cudaMemcpyHostToDevice, s))) != MOE_OK)
            return st;
        logits_dev = ws + L.logits;
    }
    if ((st = forward_impl(x_dev, static_cast<const float*>(logits_dev), dt, T, d, E, k, I,
                           score_fn, flags, w_gate_up, w_down, w_shared_gate_up, w_shared_down,
                           Is, reinterpret_cast<int32_t*>(ws + L.ids),
                           reinterpret_cast<float*>(ws + L.w), out_dev ? out_dev : ws + L.out,
                           workspace, L.fwd, stream, false)) != MOE_OK)
        return st;
    if (out_dev) return MOE_OK;
    return launch_status(
        cudaMemcpyAsync(out_host, ws + L.out, (size_t)T * d * b, cudaMemcpyDeviceToHost, s));
}

size_t moe_forward_train_workspace_size(int T, int d, int E, int k, int I, int Is,
                                        moe_dtype dt) {
    if (T < 0 || d < 1 || E < 1 || k < 1 || I < 1 || Is < 0 || !dtype_ok(dt)) return 0;
    return forward_layout(T, d, E, k, I, Is, dt, true).total;
}

moe_status moe_gate_up_train(const void* x_rows, const int32_t* offsets,
                             const int32_t* sorted_to_slot, const float* topk_weights,
                             moe_dtype dt, int R, int d, int E, int I, const void* w_gate_up,
                             unsigned flags, void* h, void* ab, void* workspace,
                             size_t ws_bytes, moe_stream_t stream) {
    if (flags & ~(unsigned)(MOE_SCALE_INPUT | MOE_WEIGHTS_PACKED)) return MOE_ERR_INVALID_ARG;
    const bool scale = (flags & MOE_SCALE_INPUT) != 0;
    const bool packed = (flags & MOE_WEIGHTS_PACKED) != 0;
    if (packed && dt != MOE_BF16) return MOE_ERR_UNSUPPORTED;
    moe_status st = check_experts_args(offsets, sorted_to_slot, topk_weights, scale, dt, R, d, E,
                                       I, workspace, ws_bytes);
    if (st != MOE_OK) return st;
    if (R == 0) return MOE_OK;
    if (!x_rows || !w_gate_up || !h || !ab) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x_rows) || !aligned16(w_gate_up) || !aligned16(h) || !aligned16(ab))
        return MOE_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    if ((st = clear_status(workspace, s)) != MOE_OK) return st;
    return run_gemm(kGateUp, x_rows, w_gate_up, packed, offsets, sorted_to_slot, topk_weights,
                    scale, dt, R, d, I, E, h, static_cast<int*>(workspace), s, ab);
}

moe_status moe_combine_backward(const void* dout, const float* y_sorted,
                                const int32_t* slot_to_sorted, const float* topk_weights,
                                moe_dtype dt, int T, int d, int k, void* dy_sorted,
                                float* d_topk_weights, moe_stream_t stream) {
    if (!dtype_ok(dt) || T < 0 || d < 1 || k < 1) return MOE_ERR_INVALID_ARG;
    if (k > kMaxK || (long long)T * k >= (1ll << 31)) return MOE_ERR_UNSUPPORTED;
    if (d % row_multiple(dt) != 0) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    if (!dout || !slot_to_sorted || !dy_sorted) return MOE_ERR_INVALID_ARG;
    if ((d_topk_weights != nullptr) != (y_sorted != nullptr)) return MOE_ERR_INVALID_ARG;
    const void* ptrs[] = {dout, y_sorted, slot_to_sorted, topk_weights, dy_sorted,
                          d_topk_weights};
    for (const void* q : ptrs)
        if (q && !aligned16(q)) return MOE_ERR_INVALID_ARG;
    return launch_status(launch_combine_backward(dout, dt == MOE_BF16, y_sorted, slot_to_sorted,
                                                 topk_weights, T, d, k, dy_sorted,
                                                 d_topk_weights, (cudaStream_t)stream));
}

size_t moe_down_backward_workspace_size(int R, int I, moe_dtype dt) {
    if (R < 0 || I < 1 || !dtype_ok(dt)) return 0;
    // per-(row, column tile) partial sums of the router-score gradient: 256-column tiles on the
    // tensor cores, 32-column tiles on the fp32 path
    const int tiles = (I + 31) / 32;
    return kStatusBytes + round_up((size_t)R * tiles * 4, 256);
}

static int scale_tiles(moe_dtype dt, int I) {
    return dt == MOE_BF16 ? (I + kBwdTileN - 1) / kBwdTileN : (I + 31) / 32;
}

static moe_status run_dgrad(BwdKind kind, const void* a, const void* w, bool packed,
                            const int32_t* offsets, const int32_t* s2p, const float* tw,
                            bool scale, const void* ab, void* out, float* part, moe_dtype dt,
                            int R, int d, int I, int E, int* status, cudaStream_t s) {
    DgradArgs g;
    g.kind = kind;
    g.a = a;
    g.w = w;
    g.packed = packed;
    g.offsets = offsets;
    g.sorted_to_slot = s2p;
    g.topk_weights = tw;
    g.scale_rows = scale;
    g.ab = ab;
    g.out = out;
    g.scale_part = part;
    g.R = R;
    g.d = d;
    g.I = I;
    g.E = E;
    g.status = status;
    return launch_status(dt == MOE_BF16 ? launch_dgrad_bf16(g, s) : launch_dgrad_f32(g, s));
}

static moe_status run_wgrad(const void* a, const void* b, const int32_t* offsets, moe_dtype dt,
                            int R, int M, int N, int E, void* dw, bool dw_bf16, int* status,
                            cudaStream_t s) {
    const int groups = offsets ? E : 1;
    if (R == 0)  // no rows at all: every expert's gradient is zero
        return launch_status(
            cudaMemsetAsync(dw, 0, (size_t)groups * M * N * (dw_bf16 ? 2 : 4), s));
    WgradArgs g;
    g.a = a;
    g.b = b;
    g.offsets = offsets;
    g.R = R;
    g.M = M;
    g.N = N;
    g.E = E;
    g.dw = dw;
    g.dw_bf16 = dw_bf16;
    g.status = status;
    return launch_status(dt == MOE_BF16 ? launch_wgrad_bf16(g, s) : launch_wgrad_f32(g, s));
}

moe_status moe_down_backward(const void* dy_sorted, const void* ab, const int32_t* offsets,
                             const int32_t* sorted_to_slot, const float* topk_weights,
                             moe_dtype dt, int R, int d, int E, int I, const void* w_down,
                             unsigned flags, void* d_ab, float* d_topk_weights, void* workspace,
                             size_t ws_bytes, moe_stream_t stream) {
    if (flags & ~(unsigned)(MOE_SCALE_INPUT | MOE_WEIGHTS_PACKED)) return MOE_ERR_INVALID_ARG;
    const bool scale = (flags & MOE_SCALE_INPUT) != 0;
    const bool packed = (flags & MOE_WEIGHTS_PACKED) != 0;
    if (packed && dt != MOE_BF16) return MOE_ERR_UNSUPPORTED;
    moe_status st = check_experts_args(offsets, sorted_to_slot, topk_weights, scale, dt, R, d, E,
                                       I, workspace, ws_bytes);
    if (st != MOE_OK) return st;
    if (ws_bytes < moe_down_backward_workspace_size(R, I, dt)) return MOE_ERR_WORKSPACE;
    if (scale && !d_topk_weights) return MOE_ERR_INVALID_ARG;
    if (R == 0) return MOE_OK;
    if (!dy_sorted || !ab || !w_down || !d_ab) return MOE_ERR_INVALID_ARG;
    const void* ptrs[] = {dy_sorted, ab, sorted_to_slot, topk_weights, w_down, d_ab,
                          d_topk_weights};
    for (const void* q : ptrs)
        if (q && !aligned16(q)) return MOE_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    if ((st = clear_status(workspace, s)) != MOE_OK) return st;
    float* part = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + kStatusBytes);
    if ((st = run_dgrad(kDgradDown, dy_sorted, w_down, packed, offsets, sorted_to_slot,
                        topk_weights, scale, ab, d_ab, part, dt, R, d, I, E,
                        static_cast<int*>(workspace), s)) != MOE_OK)
        return st;
    if (!scale) return MOE_OK;
    PdlScope pdl(true);
    return launch_status(
        launch_scale_grad(part, R, scale_tiles(dt, I), sorted_to_slot, d_topk_weights, s));
}

moe_status moe_gate_up_backward(const void* d_ab, const int32_t* offsets, moe_dtype dt, int R,
                                int d, int E, int I, const void* w_gate_up, unsigned flags,
                                float* dx_sorted, void* workspace, size_t ws_bytes,
                                moe_stream_t stream) {
    if (flags & ~(unsigned)MOE_WEIGHTS_PACKED) return MOE_ERR_INVALID_ARG;
    const bool packed = (flags & MOE_WEIGHTS_PACKED) != 0;
    if (packed && dt != MOE_BF16) return MOE_ERR_UNSUPPORTED;
    moe_status st = check_experts_args(offsets, nullptr, nullptr, false, dt, R, d, E, I,
                                       workspace, ws_bytes);
    if (st != MOE_OK) return st;
    if (R == 0) return MOE_OK;
    if (!d_ab || !w_gate_up || !dx_sorted) return MOE_ERR_INVALID_ARG;
    if (!aligned16(d_ab) || !aligned16(w_gate_up) || !aligned16(dx_sorted))
        return MOE_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    if ((st = clear_status(workspace, s)) != MOE_OK) return st;
    return run_dgrad(kDgradGateUp, d_ab, w_gate_up, packed, offsets, nullptr, nullptr, false,
                     nullptr, dx_sorted, nullptr, dt, R, d, I, E, static_cast<int*>(workspace),
                     s);
}

static moe_status weight_grad(const void* a, const void* b, const int32_t* offsets,
                              moe_dtype dt, int R, int M, int N, int E, void* dw, bool dw_bf16,
                              void* workspace, size_t ws_bytes, cudaStream_t s) {
    if (!dtype_ok(dt) || R < 0 || M < 1 || N < 1 || E < 1) return MOE_ERR_INVALID_ARG;
    if (E > kMaxE) return MOE_ERR_UNSUPPORTED;
    if (offsets == nullptr && E != 1) return MOE_ERR_INVALID_ARG;
    if (M % row_multiple(dt) != 0 || N % row_multiple(dt) != 0) return MOE_ERR_INVALID_ARG;
    if (!dw || (R > 0 && (!a || !b))) return MOE_ERR_INVALID_ARG;
    const void* ptrs[] = {a, b, offsets, dw};
    for (const void* q : ptrs)
        if (q && !aligned16(q)) return MOE_ERR_INVALID_ARG;
    if (workspace == nullptr || !aligned256(workspace) || ws_bytes < kStatusBytes)
        return MOE_ERR_WORKSPACE;
    moe_status st = clear_status(workspace, s);
    if (st != MOE_OK) return st;
    return run_wgrad(a, b, offsets, dt, R, M, N, E, dw, dw_bf16, static_cast<int*>(workspace),
                     s);
}

moe_status moe_weight_grad(const void* a, const void* b, const int32_t* offsets, moe_dtype dt,
                           int R, int M, int N, int E, float* dw, void* workspace,
                           size_t ws_bytes, moe_stream_t stream) {
    return weight_grad(a, b, offsets, dt, R, M, N, E, dw, false, workspace, ws_bytes,
                       (cudaStream_t)stream);
}

moe_status moe_weight_grad_bf16(const void* a, const void* b, const int32_t* offsets, int R,
                                int M, int N, int E, void* dw, void* workspace, size_t ws_bytes,
                                moe_stream_t stream) {
    return weight_grad(a, b, offsets, MOE_BF16, R, M, N, E, dw, true, workspace, ws_bytes,
                       (cudaStream_t)stream);
}

moe_status moe_route_backward(const float* logits, const int32_t* topk_ids,
                              const float* topk_weights, const float* d_topk_weights, int T,
                              int E, int k, moe_score_fn score_fn, unsigned flags,
                              float* d_logits, moe_stream_t stream) {
    moe_status st = check_tek(T, E, k);
    if (st != MOE_OK) return st;
    if (score_fn != MOE_SCORE_SOFTMAX && score_fn != MOE_SCORE_SIGMOID) return MOE_ERR_INVALID_ARG;
    if (flags & ~(unsigned)MOE_RENORMALIZE) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    if (!logits || !topk_ids || !topk_weights || !d_topk_weights || !d_logits)
        return MOE_ERR_INVALID_ARG;
    const void* ptrs[] = {logits, topk_ids, topk_weights, d_topk_weights, d_logits};
    for (const void* q : ptrs)
        if (!aligned16(q)) return MOE_ERR_INVALID_ARG;
    return launch_status(launch_route_backward(logits, topk_ids, topk_weights, d_topk_weights, T,
                                               E, k, (int)score_fn,
                                               (flags & MOE_RENORMALIZE) != 0, d_logits,
                                               (cudaStream_t)stream));
}

size_t moe_backward_workspace_size(int T, int d, int E, int k, int I, int Is, moe_dtype dt) {
    if (T < 0 || d < 1 || E < 1 || k < 1 || I < 1 || Is < 0 || !dtype_ok(dt)) return 0;
    return backward_layout(T, d, k, I, Is, dt).total;
}

int moe_backward_kernel_count(int T, int k, int Is, unsigned flags, int want_logits) {
    if (T <= 0 || k <= 0) return 0;
    const bool scale = (flags & MOE_SCALE_INPUT) != 0;
    // combine backward, down wgrad, down dgrad (+ score gradient), gate_up wgrad and dgrad,
    // the shared expert's four, the transpose of the dispatch, the router backward
    return 1 + 2 + (scale ? 1 : 0) + 2 + (Is > 0 ? 4 : 0) + 1 + (want_logits ? 1 : 0);
}

moe_status moe_backward(const void* dout, const void* x, const float* logits, moe_dtype dt, int T,
                        int d, int E, int k, int I, moe_score_fn score_fn, unsigned flags,
                        const void* w_gate_up, const void* w_down, const void* w_shared_gate_up,
                        const void* w_shared_down, int Is, const int32_t* topk_ids,
                        const float* topk_weights, const void* fwd_workspace,
                        size_t fwd_ws_bytes, void* dx, float* d_w_gate_up, float* d_w_down,
                        float* d_w_shared_gate_up, float* d_w_shared_down,
                        float* d_topk_weights, float* d_logits, void* workspace,
                        size_t ws_bytes, moe_stream_t stream) {
    moe_status st = check_tek(T, E, k);
    if (st != MOE_OK) return st;
    if (!dtype_ok(dt)) return MOE_ERR_INVALID_ARG;
    if (score_fn != MOE_SCORE_SOFTMAX && score_fn != MOE_SCORE_SIGMOID) return MOE_ERR_INVALID_ARG;
    if (flags & ~(unsigned)(MOE_RENORMALIZE | MOE_SCALE_INPUT | MOE_WEIGHTS_PACKED |
                            MOE_WGRAD_BF16))
        return MOE_ERR_INVALID_ARG;
    const bool scale = (flags & MOE_SCALE_INPUT) != 0;
    const bool packed = (flags & MOE_WEIGHTS_PACKED) != 0;
    const bool wbf16 = (flags & MOE_WGRAD_BF16) != 0;
    if ((packed || wbf16) && dt != MOE_BF16) return MOE_ERR_UNSUPPORTED;
    if (d < 1 || I < 1 || Is < 0) return MOE_ERR_INVALID_ARG;
    if (d % row_multiple(dt) != 0 || I % row_multiple(dt) != 0 || Is % row_multiple(dt) != 0)
        return MOE_ERR_INVALID_ARG;
    const bool shared = Is > 0;
    if (shared != (w_shared_gate_up != nullptr) || shared != (w_shared_down != nullptr) ||
        shared != (d_w_shared_gate_up != nullptr) || shared != (d_w_shared_down != nullptr))
        return MOE_ERR_INVALID_ARG;
    if (dt == MOE_F32 && ((long long)T * k > kMaxRowsF32)) return MOE_ERR_UNSUPPORTED;
    if (d_logits && !logits) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    if (!dout || !x || !w_gate_up || !w_down || !topk_ids || !topk_weights || !dx ||
        !d_w_gate_up || !d_w_down || !fwd_workspace)
        return MOE_ERR_INVALID_ARG;
    const void* ptrs[] = {dout, x, logits, w_gate_up, w_down, w_shared_gate_up, w_shared_down,
                          topk_ids, topk_weights, dx, d_w_gate_up, d_w_down, d_w_shared_gate_up,
                          d_w_shared_down, d_topk_weights, d_logits};
    for (const void* q : ptrs)
        if (q && !aligned16(q)) return MOE_ERR_INVALID_ARG;
    const ForwardLayout F = forward_layout(T, d, E, k, I, Is, dt, true);
    if (!aligned256(fwd_workspace) || fwd_ws_bytes < F.total) return MOE_ERR_WORKSPACE;
    const BackwardLayout L = backward_layout(T, d, k, I, Is, dt);
    if (!workspace || !aligned256(workspace) || ws_bytes < L.total) return MOE_ERR_WORKSPACE;

    cudaStream_t s = (cudaStream_t)stream;
    const uint8_t* fw = static_cast<const uint8_t*>(fwd_workspace);
    const int32_t* offsets = reinterpret_cast<const int32_t*>(fw + F.offsets);
    const int32_t* s2p = reinterpret_cast<const int32_t*>(fw + F.s2p);
    const int32_t* p2s = reinterpret_cast<const int32_t*>(fw + F.p2s);
    const void* xs = fw + F.x_sorted;
    const void* h = fw + F.h;
    const float* y = reinterpret_cast<const float*>(fw + F.y);
    const void* ab = fw + F.ab;
    const void* h_sh = fw + F.h_sh;
    const void* ab_sh = fw + F.ab_sh;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    int* status = reinterpret_cast<int*>(ws);
    void* dy = ws + L.dy;
    void* d_ab = ws + L.d_ab;
    float* dxs = reinterpret_cast<float*>(ws + L.dx_sorted);
    float* part = reinterpret_cast<float*>(ws + L.part);
    float* dw = d_topk_weights ? d_topk_weights : reinterpret_cast<float*>(ws + L.dw_tmp);
    void* d_ab_sh = ws + L.d_ab_sh;
    float* dx_sh = reinterpret_cast<float*>(ws + L.dx_sh);
    const int R = T * k;

    if ((st = clear_status(workspace, s)) != MOE_OK) return st;
    // combine: dy = w dout (dout itself when the score scaled the input), d w = dout . y
    if ((st = launch_status(launch_combine_backward(dout, dt == MOE_BF16, scale ? nullptr : y,
                                                    p2s, scale ? nullptr : topk_weights, T, d,
                                                    k, dy, scale ? nullptr : dw, s))) != MOE_OK)
        return st;
    PdlScope pdl(true);
    // down projection: d W_down = h^T dy; dh = dy W_down^T through the SwiGLU backward
    if ((st = run_wgrad(h, dy, offsets, dt, R, I, d, E, d_w_down, wbf16, status, s)) != MOE_OK)
        return st;
    if ((st = run_dgrad(kDgradDown, dy, w_down, packed, offsets, s2p, topk_weights, scale, ab,
                        d_ab, part, dt, R, d, I, E, status, s)) != MOE_OK)
        return st;
    if (scale && (st = launch_status(launch_scale_grad(part, R, scale_tiles(dt, I), s2p, dw,
                                                       s))) != MOE_OK)
        return st;
    // gate/up projection: d W_gate_up = x_sorted^T d_ab; dx_sorted = d_ab W_gate_up^T
    if ((st = run_wgrad(xs, d_ab, offsets, dt, R, d, 2 * I, E, d_w_gate_up, wbf16, status,
                        s)) != MOE_OK)
        return st;
    if ((st = run_dgrad(kDgradGateUp, d_ab, w_gate_up, packed, offsets, nullptr, nullptr, false,
                        nullptr, dxs, nullptr, dt, R, d, I, E, status, s)) != MOE_OK)
        return st;
    if (shared) {
        // the shared expert sees the unscaled x with weight 1: its dy is dout
        if ((st = run_wgrad(h_sh, dout, nullptr, dt, T, Is, d, 1, d_w_shared_down, wbf16, status,
                            s)) != MOE_OK)
            return st;
        if ((st = run_dgrad(kDgradDown, dout, w_shared_down, packed, nullptr, nullptr, nullptr,
                            false, ab_sh, d_ab_sh, nullptr, dt, T, d, Is, 1, status, s)) !=
            MOE_OK)
            return st;
        if ((st = run_wgrad(x, d_ab_sh, nullptr, dt, T, d, 2 * Is, 1, d_w_shared_gate_up, wbf16,
                            status, s)) != MOE_OK)
            return st;
        if ((st = run_dgrad(kDgradGateUp, d_ab_sh, w_shared_gate_up, packed, nullptr, nullptr,
                            nullptr, false, nullptr, dx_sh, nullptr, dt, T, d, Is, 1, status,
                            s)) != MOE_OK)
            return st;
    }
    // the dispatch's transpose: dx[t] = sum_j dx_sorted[slot_to_sorted[t k + j]] (+ shared)
    if ((st = launch_status(launch_combine(dxs, p2s, nullptr, shared ? dx_sh : nullptr, T, d, k,
                                           dt == MOE_BF16, dx, s))) != MOE_OK)
        return st;
    if (!d_logits) return MOE_OK;
    return launch_status(launch_route_backward(logits, topk_ids, topk_weights, dw, T, E, k,
                                               (int)score_fn, (flags & MOE_RENORMALIZE) != 0,
                                               d_logits, s));
}

// ---- MX (block-scaled FP8 activations, FP4 weights) ----
size_t moe_mx_weights_size(moe_weight_kind kind, int E, int K, int N) {
    if ((kind != MOE_W_GATE_UP && kind != MOE_W_DOWN) || E < 1 || K < 1 || N < 1 || N % 8)
        return 0;
    return mx_geom(kind == MOE_W_GATE_UP, K, N, E).total;
}

static moe_status check_mx_weights(moe_weight_kind kind, const void* a, const void* b, int E,
                                   int K, int N) {
    if (kind != MOE_W_GATE_UP && kind != MOE_W_DOWN) return MOE_ERR_INVALID_ARG;
    if (E < 1 || K < 1 || N < 1 || N % 8 != 0 || K % 8 != 0) return MOE_ERR_INVALID_ARG;
    if (!a || !b || !aligned16(a) || !aligned16(b)) return MOE_ERR_INVALID_ARG;
    return MOE_OK;
}

moe_status moe_quantize_weights_mx(moe_weight_kind kind, const void* w, void* mx, int E, int K,
                                   int N, moe_stream_t stream) {
    const moe_status st = check_mx_weights(kind, w, mx, E, K, N);
    if (st != MOE_OK) return st;
    return launch_status(launch_mx_quant_weights(kind == MOE_W_GATE_UP, w, E, K, N, mx,
                                                 (cudaStream_t)stream));
}

moe_status moe_dequantize_weights_mx(moe_weight_kind kind, const void* mx, void* w, int E, int K,
                                     int N, moe_stream_t stream) {
    const moe_status st = check_mx_weights(kind, mx, w, E, K, N);
    if (st != MOE_OK) return st;
    return launch_status(launch_mx_dequant_weights(kind == MOE_W_GATE_UP, mx, E, K, N, nullptr,
                                                   w, (cudaStream_t)stream));
}

moe_status moe_quantize_rows_mx(const void* x, int R, int K, void* x_out, void* codes,
                                void* scales, moe_stream_t stream) {
    if (R < 0 || K < 1 || K % 8 != 0) return MOE_ERR_INVALID_ARG;
    if ((codes == nullptr) != (scales == nullptr)) return MOE_ERR_INVALID_ARG;
    if (R == 0) return MOE_OK;
    if (!x || (!x_out && !codes)) return MOE_ERR_INVALID_ARG;
    const void* ptrs[] = {x, x_out, codes};
    for (const void* q : ptrs)
        if (q && !aligned16(q)) return MOE_ERR_INVALID_ARG;
    return launch_status(launch_mx_rows(x, R, K, x_out, codes, scales, (cudaStream_t)stream));
}

size_t moe_forward_mx_workspace_size(int T, int d, int E, int k, int I, int Is) {
    if (T < 0 || d < 1 || E < 1 || k < 1 || I < 1 || Is < 0) return 0;
    return forward_layout(T, d, E, k, I, Is, MOE_BF16, false, true).total;
}

moe_status moe_forward_mx(const void* x, const float* logits, int T, int d, int E, int k, int I,
                          moe_score_fn score_fn, unsigned flags, const void* w_gate_up_mx,
                          const void* w_down_mx, const void* w_shared_gate_up_mx,
                          const void* w_shared_down_mx, int Is, int32_t* topk_ids,
                          float* topk_weights, void* out, void* workspace, size_t ws_bytes,
                          moe_stream_t stream) {
    if (flags & MOE_WEIGHTS_PACKED) return MOE_ERR_INVALID_ARG;
    return forward_impl(x, logits, MOE_BF16, T, d, E, k, I, score_fn, flags, w_gate_up_mx,
                        w_down_mx, w_shared_gate_up_mx, w_shared_down_mx, Is, topk_ids,
                        topk_weights, out, workspace, ws_bytes, stream, false, true);
}

// ---- MX on the block-scaled tensor cores (weights in the MX tensor-core layout) ----
size_t moe_mx_tc_weights_size(moe_weight_kind kind, int E, int K, int N) {
    if ((kind != MOE_W_GATE_UP && kind != MOE_W_DOWN) || E < 1 || K < 1 || N < 1 || N % 32 ||
        K % 32)
        return 0;
    return mx_tc_geom(kind == MOE_W_GATE_UP, K, N, E).total;
}

static moe_status check_mx_tc_weights(moe_weight_kind kind, const void* a, const void* b, int E,
                                      int K, int N) {
    if (kind != MOE_W_GATE_UP && kind != MOE_W_DOWN) return MOE_ERR_INVALID_ARG;
    if (E < 1 || K < 1 || N < 1 || N % 32 != 0 || K % 32 != 0) return MOE_ERR_INVALID_ARG;
    if (!a || !b || !aligned256(a) || !aligned256(b)) return MOE_ERR_INVALID_ARG;
    return MOE_OK;
}

moe_status moe_quantize_weights_mx_tc(moe_weight_kind kind, const void* w, void* mx, int E,
                                      int K, int N, moe_stream_t stream) {
    if (!aligned16(w)) return MOE_ERR_INVALID_ARG;
    const moe_status st = check_mx_tc_weights(kind, mx, mx, E, K, N);
    if (st != MOE_OK) return st;
    if (!w) return MOE_ERR_INVALID_ARG;
    return launch_status(launch_mx_tc_quant_weights(kind == MOE_W_GATE_UP, w, E, K, N, mx,
                                                    (cudaStream_t)stream));
}

moe_status moe_dequantize_weights_mx_tc(moe_weight_kind kind, const void* mx, void* w, int E,
                                        int K, int N, moe_stream_t stream) {
    const moe_status st = check_mx_tc_weights(kind, mx, mx, E, K, N);
    if (st != MOE_OK) return st;
    if (!w || !aligned16(w)) return MOE_ERR_INVALID_ARG;
    return launch_status(launch_mx_tc_dequant_weights(kind == MOE_W_GATE_UP, mx, E, K, N, w,
                                                      (cudaStream_t)stream));
}

namespace {
// moe_forward_mx_tc's workspace: status word, dispatch indices, then the padded MXFP8 rows
// (x codes and scale atoms, h codes and scale atoms), y_sorted, and for a shared expert its own
// x and h in the same form plus its y. Rp = R rounded up to 128 plus 128 per expert bounds the
// padded rows (every expert's rows start at a multiple of 128).
struct MxTcLayout {
    size_t counts, offsets, chunk, s2p, p2s, xq, xsf, hq, hsf, y, sxq, ssf, shq, shsf, ysh,
        part, total;
    int Rp, Tp;
};

MxTcLayout mx_tc_layout(int T, int d, int E, int k, int I, int Is) {
    const size_t R = (size_t)T * k;
    MxTcLayout L;
    L.Rp = (int)(round_up(R, 128) + 128 * (size_t)E);
    L.Tp = (int)round_up((size_t)T, 128);
    const size_t kcd = (d + 127) / 128, kci = (I + 127) / 128, kcs = (Is + 127) / 128;
    size_t o = kStatusBytes;
    auto take = [&](size_t bytes) {
        const size_t at = o;
        o = round_up(o + bytes, 256);
        return at;
    };
    L.counts = take((size_t)E * 4);
    L.offsets = take((size_t)(E + 1) * 4);
    L.chunk = take(dispatch_scratch_bytes((int)R, E));
    L.s2p = take(R * 4);
    L.p2s = take(R * 4);
    L.xq = take((size_t)L.Rp * d);
    L.xsf = take((size_t)L.Rp / 128 * kcd * 512);
    L.hq = take((size_t)L.Rp * I);
    L.hsf = take((size_t)L.Rp / 128 * kci * 512);
    L.y = take(R * (size_t)d * 4);
    L.sxq = take(Is > 0 ? (size_t)L.Tp * d : 0);
    L.ssf = take(Is > 0 ? (size_t)L.Tp / 128 * kcd * 512 : 0);
    L.shq = take(Is > 0 ? (size_t)L.Tp * Is : 0);
    L.shsf = take(Is > 0 ? (size_t)L.Tp / 128 * kcs * 512 : 0);
    L.ysh = take(Is > 0 ? (size_t)T * d * 4 : 0);
    // decode batches: the one-kernel layer's partial sums
    L.part = take(decode_mx_tc_applies(T, d, k, I, Is) ? decode_mx_tc_part_bytes(T, d, k, I) : 0);
    L.total = o;
    return L;
}

moe_status run_mx_tc_gemm(GemmKind kind, const void* a, const void* a_sf, const void* w,
                          const int32_t* offsets, const int32_t* s2p, const float* tw,
                          bool scale, int R, int Rp, int K, int N, int groups, void* out,
                          void* h_sf, int* status, cudaStream_t s) {
    MxTcGemmArgs g;
    g.kind = kind;
    g.a = a;
    g.a_sf = a_sf;
    g.b = w;
    g.offsets = offsets;
    g.sorted_to_slot = s2p;
    g.topk_weights = tw;
    g.scale_rows = scale;
    g.R = R;
    g.Rp = Rp;
    g.K = K;
    g.N = N;
    g.groups = groups;
    g.out = out;
    g.h_sf = h_sf;
    g.status = status;
    return launch_status(launch_mx_tc_gemm(g, s));
}
}  // namespace

moe_status moe_mx_tc_rows(const void* x, int T, int d, int k, int E, const int32_t* topk_ids,
                          const int32_t* slot_to_sorted, const int32_t* offsets, void* codes,
                          void* sf, void* codes_sh, void* sf_sh, moe_stream_t stream) {
    moe_status st = check_tek(T, E, k);
    if (st != MOE_OK) return st;
    if (d < 32 || d % 32) return MOE_ERR_INVALID_ARG;
    if ((codes == nullptr) != (sf == nullptr) || (codes_sh == nullptr) != (sf_sh == nullptr))
        return MOE_ERR_INVALID_ARG;
    if (codes && (!topk_ids || !slot_to_sorted || !offsets)) return MOE_ERR_INVALID_ARG;
    if (!codes && !codes_sh) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    const void* ptrs[] = {x, codes, sf, codes_sh, sf_sh};
    for (const void* q : ptrs)
        if (q && !aligned16(q)) return MOE_ERR_INVALID_ARG;
    if (!x) return MOE_ERR_INVALID_ARG;
    return launch_status(launch_mx_tc_quant_rows(x, T, d, codes ? k : 0, E, topk_ids,
                                                 slot_to_sorted, codes ? offsets : nullptr,
                                                 codes, sf, codes_sh, sf_sh,
                                                 (cudaStream_t)stream));
}

static moe_status mx_tc_gemm_entry(GemmKind kind, const void* a, const void* a_sf,
                                   const int32_t* offsets, const int32_t* s2p, const float* tw,
                                   bool scale, int R, int K, int E, int N, const void* w,
                                   void* out, void* h_sf, void* workspace, size_t ws_bytes,
                                   moe_stream_t stream) {
    if (R < 0 || E < 1 || E > kMaxE || K < 32 || N < 32 || K % 32 || N % 32)
        return MOE_ERR_INVALID_ARG;
    if (offsets == nullptr && E != 1) return MOE_ERR_INVALID_ARG;
    if (scale && (s2p == nullptr || tw == nullptr)) return MOE_ERR_INVALID_ARG;
    if ((long long)R + 128ll * (E + 1) >= (1ll << 31)) return MOE_ERR_UNSUPPORTED;
    if (workspace == nullptr || !aligned256(workspace) || ws_bytes < kStatusBytes)
        return MOE_ERR_WORKSPACE;
    if (R == 0) return MOE_OK;
    if (!a || !a_sf || !w || !out || (kind == kGateUp && !h_sf)) return MOE_ERR_INVALID_ARG;
    const void* ptrs[] = {a, a_sf, out, h_sf, offsets};
    for (const void* q : ptrs)
        if (q && !aligned16(q)) return MOE_ERR_INVALID_ARG;
    if (!aligned256(w)) return MOE_ERR_INVALID_ARG;
    const int Rp = (int)(round_up((size_t)R, 128) + (offsets ? 128 * (size_t)E : 0));
    cudaStream_t s = (cudaStream_t)stream;
    moe_status st = clear_status(workspace, s);
    if (st != MOE_OK) return st;
    return run_mx_tc_gemm(kind, a, a_sf, w, offsets, s2p, tw, scale, R, Rp, K, N, E, out, h_sf,
                          reinterpret_cast<int*>(workspace), s);
}

moe_status moe_gate_up_mx_tc(const void* x_codes, const void* x_sf, const int32_t* offsets,
                             const int32_t* sorted_to_slot, const float* topk_weights, int R,
                             int d, int E, int I, const void* w_gate_up_mx, unsigned flags,
                             void* h_codes, void* h_sf, void* workspace, size_t ws_bytes,
                             moe_stream_t stream) {
    if (flags & ~(unsigned)MOE_SCALE_INPUT) return MOE_ERR_INVALID_ARG;
    return mx_tc_gemm_entry(kGateUp, x_codes, x_sf, offsets, sorted_to_slot, topk_weights,
                            (flags & MOE_SCALE_INPUT) != 0, R, d, E, I, w_gate_up_mx, h_codes,
                            h_sf, workspace, ws_bytes, stream);
}

moe_status moe_down_mx_tc(const void* h_codes, const void* h_sf, const int32_t* offsets, int R,
                          int I, int E, int d, const void* w_down_mx, float* y_sorted,
                          void* workspace, size_t ws_bytes, moe_stream_t stream) {
    return mx_tc_gemm_entry(kDown, h_codes, h_sf, offsets, nullptr, nullptr, false, R, I, E, d,
                            w_down_mx, y_sorted, nullptr, workspace, ws_bytes, stream);
}

size_t moe_forward_mx_tc_workspace_size(int T, int d, int E, int k, int I, int Is) {
    if (T < 0 || d < 1 || E < 1 || k < 1 || I < 1 || Is < 0) return 0;
    return mx_tc_layout(T, d, E, k, I, Is).total;
}

int moe_forward_mx_tc_kernel_count(int T, int d, int k, int I, int Is) {
    if (T <= 0 || k <= 0 || d < 1 || I < 1 || Is < 0) return 0;
    if (decode_mx_tc_applies(T, d, k, I, Is)) return 1;
    const bool small = (long long)T * k <= kSmallDispatchMaxSlots;
    return (small ? 1 : 1 + dispatch_kernel_count(false)) + 3 + (Is > 0 ? 2 : 0) + 1;
}

moe_status moe_forward_mx_tc(const void* x, const float* logits, int T, int d, int E, int k,
                             int I, moe_score_fn score_fn, unsigned flags,
                             const void* w_gate_up_mx, const void* w_down_mx,
                             const void* w_shared_gate_up_mx, const void* w_shared_down_mx,
                             int Is, int32_t* topk_ids, float* topk_weights, void* out,
                             void* workspace, size_t ws_bytes, moe_stream_t stream) {
    moe_status st = check_tek(T, E, k);
    if (st != MOE_OK) return st;
    if (score_fn != MOE_SCORE_SOFTMAX && score_fn != MOE_SCORE_SIGMOID) return MOE_ERR_INVALID_ARG;
    if (flags & ~(unsigned)(MOE_RENORMALIZE | MOE_SCALE_INPUT)) return MOE_ERR_INVALID_ARG;
    if (d < 1 || I < 1 || Is < 0 || d % 32 || I % 32 || Is % 32) return MOE_ERR_INVALID_ARG;
    const bool shared = w_shared_gate_up_mx != nullptr || w_shared_down_mx != nullptr;
    if (shared != (Is > 0)) return MOE_ERR_INVALID_ARG;
    if (shared && (!w_shared_gate_up_mx || !w_shared_down_mx)) return MOE_ERR_INVALID_ARG;
    if ((long long)T * k + 128ll * (E + 1) >= (1ll << 31)) return MOE_ERR_UNSUPPORTED;
    if (T == 0) return MOE_OK;
    if (!x || !logits || !w_gate_up_mx || !w_down_mx || !topk_ids || !topk_weights || !out)
        return MOE_ERR_INVALID_ARG;
    const void* ptrs[] = {x, logits, topk_ids, topk_weights, out};
    for (const void* q : ptrs)
        if (!aligned16(q)) return MOE_ERR_INVALID_ARG;
    const void* wptrs[] = {w_gate_up_mx, w_down_mx, w_shared_gate_up_mx, w_shared_down_mx};
    for (const void* q : wptrs)
        if (q && !aligned256(q)) return MOE_ERR_INVALID_ARG;
    const MxTcLayout L = mx_tc_layout(T, d, E, k, I, Is);
    if (!workspace || !aligned256(workspace) || ws_bytes < L.total) return MOE_ERR_WORKSPACE;

    cudaStream_t s = (cudaStream_t)stream;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    int* status = reinterpret_cast<int*>(ws);
    int32_t* counts = reinterpret_cast<int32_t*>(ws + L.counts);
    int32_t* offsets = reinterpret_cast<int32_t*>(ws + L.offsets);
    int32_t* chunk = reinterpret_cast<int32_t*>(ws + L.chunk);
    int32_t* s2p = reinterpret_cast<int32_t*>(ws + L.s2p);
    int32_t* p2s = reinterpret_cast<int32_t*>(ws + L.p2s);
    float* y = reinterpret_cast<float*>(ws + L.y);
    float* ysh = reinterpret_cast<float*>(ws + L.ysh);
    const int R = T * k;
    const bool scale = (flags & MOE_SCALE_INPUT) != 0;
    const bool renorm = (flags & MOE_RENORMALIZE) != 0;

    if (decode_mx_tc_applies(T, d, k, I, Is)) {
        // decode: the whole layer in one cooperative kernel; its counter sits in the workspace
        // head and is cleared with the status word
        if ((st = launch_status(cudaMemsetAsync(workspace, 0, kStatusBytes, s))) != MOE_OK)
            return st;
        DecodeMxTcArgs a;
        a.x = x;
        a.logits = logits;
        a.w_gate_up = w_gate_up_mx;
        a.w_down = w_down_mx;
        a.score_fn = (int)score_fn;
        a.renorm = renorm;
        a.scale_input = scale;
        a.T = T;
        a.d = d;
        a.E = E;
        a.k = k;
        a.I = I;
        a.topk_ids = topk_ids;
        a.topk_weights = topk_weights;
        a.counts = counts;
        a.offsets = offsets;
        a.sorted_to_slot = s2p;
        a.slot_to_sorted = p2s;
        a.x_codes = ws + L.xq;
        a.x_sf = ws + L.xsf;
        a.h_codes = ws + L.hq;
        a.h_sf = ws + L.hsf;
        a.partials = ws + L.part;
        a.out = out;
        a.done = reinterpret_cast<int*>(ws + kDecodeMxTcCounterByte);
        a.status = status;
        return launch_status(launch_decode_mx_tc(a, s));
    }
    if ((st = clear_status(workspace, s)) != MOE_OK) return st;
    // route and the dispatch indices (no row copy: the next kernel writes the rows in MXFP8)
    if (R <= kSmallDispatchMaxSlots) {
        if ((st = launch_status(launch_route_dispatch_small(logits, T, E, k, (int)score_fn,
                                                            renorm, topk_ids, topk_weights,
                                                            counts, offsets, s2p, p2s, s))) !=
            MOE_OK)
            return st;
    } else {
        if ((st = launch_status(launch_route(logits, T, E, k, (int)score_fn, renorm, topk_ids,
                                             topk_weights, s))) != MOE_OK)
            return st;
    }
    PdlScope pdl(true);
    if (R > kSmallDispatchMaxSlots &&
        (st = launch_status(launch_dispatch(topk_ids, nullptr, 0, T, E, k, counts, offsets, s2p,
                                            p2s, nullptr, chunk, status, s))) != MOE_OK)
        return st;
    // x to MXFP8 once per token, written to every padded row it was sent to (and to the shared
    // expert's rows)
    if ((st = launch_status(launch_mx_tc_quant_rows(
             x, T, d, k, E, topk_ids, p2s, offsets, ws + L.xq, ws + L.xsf,
             shared ? ws + L.sxq : nullptr, shared ? ws + L.ssf : nullptr, s))) != MOE_OK)
        return st;
    if ((st = run_mx_tc_gemm(kGateUp, ws + L.xq, ws + L.xsf, w_gate_up_mx, offsets, s2p,
                             topk_weights, scale, R, L.Rp, d, I, E, ws + L.hq, ws + L.hsf,
                             status, s)) != MOE_OK)
        return st;
    if ((st = run_mx_tc_gemm(kDown, ws + L.hq, ws + L.hsf, w_down_mx, offsets, nullptr, nullptr,
                             false, R, L.Rp, I, d, E, y, nullptr, status, s)) != MOE_OK)
        return st;
    if (shared) {
        if ((st = run_mx_tc_gemm(kGateUp, ws + L.sxq, ws + L.ssf, w_shared_gate_up_mx, nullptr,
                                 nullptr, nullptr, false, T, L.Tp, d, Is, 1, ws + L.shq,
                                 ws + L.shsf, status, s)) != MOE_OK)
            return st;
        if ((st = run_mx_tc_gemm(kDown, ws + L.shq, ws + L.shsf, w_shared_down_mx, nullptr,
                                 nullptr, nullptr, false, T, L.Tp, Is, d, 1, ysh, nullptr, status,
                                 s)) != MOE_OK)
            return st;
    }
    return launch_status(launch_combine(y, p2s, scale ? nullptr : topk_weights,
                                        shared ? ysh : nullptr, T, d, k, true, out, s));
}

moe_status moe_read_device_status(const void* workspace, moe_stream_t stream) {
    if (!workspace) return MOE_ERR_INVALID_ARG;
    int v = 0;
    if (cudaMemcpyAsync(&v, workspace, sizeof(int), cudaMemcpyDeviceToHost,
                        (cudaStream_t)stream) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return MOE_ERR_CUDA;
    return static_cast<moe_status>(v);
}

}  // extern "C"
