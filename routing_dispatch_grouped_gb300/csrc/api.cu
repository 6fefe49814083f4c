// C ABI of libmoe: argument checks, workspace layout and the launch chain of each entry point.
// Every check runs before anything is enqueued (Expert parallelism page, "Overriding the
// plans": errors are raised before any work). No call allocates, frees or synchronises, except
// moe_read_device_status, which exists to synchronise.
#include <mutex>

#include "moe_internal.cuh"

namespace rdg {

namespace {
thread_local bool t_pdl = false;
}
bool pdl_enabled() { return t_pdl; }
PdlScope::PdlScope(bool on) : prev(t_pdl) { t_pdl = on; }
PdlScope::~PdlScope() { t_pdl = prev; }

int device_sm_count() {
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    if (cache[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 148;
        cache[dev] = n;
    }
    return cache[dev];
}

}  // namespace rdg

using namespace rdg;

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
    size_t fcnt, counts, offsets, chunk, s2p, p2s, x_sorted, h, y, h_sh, y_sh, fused, total;
};

ForwardLayout forward_layout(int T, int d, int E, int k, int I, int Is, moe_dtype dt) {
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
    const bool fused = decode_fused_applies(dt, T, k, Is);
    const DecodeFusedLayout F = decode_fused_layout(T, d, k, I);
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
    L.total = o;
    return L;
}

moe_status clear_status(void* workspace, cudaStream_t s) {
    return launch_status(cudaMemsetAsync(workspace, 0, sizeof(int), s));
}

moe_status run_gemm(GemmKind kind, const void* a, const void* b, bool packed,
                    const int32_t* offsets, const int32_t* s2p, const float* w, bool scale,
                    moe_dtype dt, int R, int K, int N, int E, void* out, int* status,
                    cudaStream_t s) {
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

moe_status moe_forward(const void* x, const float* logits, moe_dtype dt, int T, int d, int E,
                       int k, int I, moe_score_fn score_fn, unsigned flags, const void* w_gate_up,
                       const void* w_down, const void* w_shared_gate_up,
                       const void* w_shared_down, int Is, int32_t* topk_ids, float* topk_weights,
                       void* out, void* workspace, size_t ws_bytes, moe_stream_t stream) {
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
    if (scale && fuse_w) return MOE_ERR_INVALID_ARG;
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
    const ForwardLayout L = forward_layout(T, d, E, k, I, Is, dt);
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
    if (decode_fused_applies(dt, T, k, Is)) {
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
        return launch_status(launch_decode_fused(a, s));
    }
    if ((st = clear_status(workspace, s)) != MOE_OK) return st;
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
        if ((st = launch_status(launch_dispatch_copy(x, (size_t)d * dtype_bytes(dt), T, k, p2s,
                                                     xs, s))) != MOE_OK)
            return st;
    } else {
        if ((st = launch_status(launch_dispatch(topk_ids, x, (size_t)d * dtype_bytes(dt), T, E,
                                                k, counts, offsets, s2p, p2s, xs, chunk, status,
                                                s))) != MOE_OK)
            return st;
    }
    if ((st = run_gemm(kGateUp, xs, w_gate_up, packed, offsets, s2p, topk_weights, scale, dt, R,
                       d, I, E, h, status, s)) != MOE_OK)
        return st;
    if ((st = run_gemm(kDown, h, w_down, packed, offsets, s2p, topk_weights, fuse_w, dt, R, I, d,
                       E, y, status, s)) != MOE_OK)
        return st;
    if (shared) {
        if ((st = run_gemm(kGateUp, x, w_shared_gate_up, packed, nullptr, nullptr, nullptr, false,
                           dt, T, d, Is, 1, h_sh, status, s)) != MOE_OK)
            return st;
        if ((st = run_gemm(kDown, h_sh, w_shared_down, packed, nullptr, nullptr, nullptr, false,
                           dt, T, Is, d, 1, y_sh, status, s)) != MOE_OK)
            return st;
    }
    const float* comb_w = (scale || fuse_w) ? nullptr : topk_weights;
    return launch_status(launch_combine(y, p2s, comb_w, shared ? y_sh : nullptr, T, d, k,
                                        dt == MOE_BF16, out, s));
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
