/*
 * moe.h - C ABI of the GB300 (sm_103a) MoE expert-layer library (libmoe.so).
 *
 * The layer: router top-k gating over per-token expert logits, dispatch of every (token, expert)
 * pair to its expert, the per-expert gated feed-forward (gate/up projection, SwiGLU, down
 * projection) as a grouped GEMM, and the router-weighted combine back to token order.
 *
 * Sources (Transformers documentation):
 *   [EP-intro]     "Expert parallelism", introduction: a router sends tokens to the matching
 *                  experts and gathers the results; Llama-4 experts get every token already
 *                  scaled by the router score.
 *   [EP-add]       "Expert parallelism", "Adding an implementation": __call__(hidden_states,
 *                  top_k_index, top_k_weights) returns the weighted expert output for each token
 *                  of the batch; experts_forward runs on the rows, expert ids and weights routed
 *                  to the experts; an implementation may keep state such as buffers.
 *   [EP-choose]    "Expert parallelism", "Choosing an implementation": all_to_all needs a host
 *                  synchronisation per layer and so cannot be captured in a CUDA graph;
 *                  all_reduce moves no tokens, needs no host sync and is captured at decode.
 *   [EP-dispatch]  "Expert parallelism", "Token dispatch": each (token, expert) pair is sent to
 *                  the owner of that expert, the local experts run on what arrived, the results
 *                  come back and are combined with the routing weights.
 *   [EP-tp]        "Expert parallelism", "With tensor parallelism": token slices may be uneven
 *                  or empty, including single-token decoding.
 *   [EP-override]  "Expert parallelism", "Overriding the plans": a bad key raises ValueError
 *                  before anything is sharded (errors are reported before any work).
 *   [TP-packed]    "Tensor parallelism for inference", "Packed strategies": gate_up_proj is
 *                  [num_experts, hidden, 2 * expert_dim]; bmm(hidden_states, gate_up_proj) then
 *                  chunk(2, dim=-1) gives gate (first half) and up (second half).
 *
 * On one GPU the all-to-all of [EP-dispatch] becomes a local permutation (moe_dispatch) and the
 * return all-to-all plus weighted sum becomes moe_combine; no call here crosses GPUs.
 *
 * Conventions for every entry point
 *   - All device pointers are caller-owned device memory. The library never allocates, frees or
 *     synchronises inside these calls; work is enqueued on `stream` (NULL = legacy default
 *     stream) and the call returns at once. moe_route, moe_dispatch, moe_gate_up, moe_down,
 *     moe_experts, moe_combine and moe_forward need no host sync, so a sequence of them with
 *     fixed pointers can be captured in a CUDA graph (the property [EP-choose] asks of decode).
 *   - Every argument is checked before any launch ([EP-override] convention). A bad argument
 *     returns MOE_ERR_INVALID_ARG, a shape or dtype the kernels do not cover returns
 *     MOE_ERR_UNSUPPORTED, a short workspace returns MOE_ERR_WORKSPACE; in all three cases
 *     nothing is enqueued. A failed launch returns MOE_ERR_CUDA.
 *   - Faults only the device can see (an expert id outside [0, E) handed to moe_dispatch, a
 *     device-side wait that ran out of time) are written to a status word at the start of the
 *     call's workspace; the kernels stay memory-safe and finish. moe_read_device_status()
 *     reports the word (it synchronises the stream: diagnostics only).
 *   - Pointers must be 16-byte aligned. Row lengths must give 16-byte rows: d and I multiples
 *     of 8 for MOE_BF16, of 4 for MOE_F32.
 *   - Ranges: 1 <= E <= 256, 1 <= k <= min(E, 32), T >= 0, T * k < 2^31. T == 0 is a no-op
 *     returning MOE_OK ([EP-tp]: slices may be empty).
 *   - Calls are stateless and re-entrant; calls on different streams must not share outputs or
 *     workspace.
 *
 * Layouts (row-major, C order)
 *   logits         float  [T, E]
 *   topk_ids       int32  [T, k]   slot j = 0 is the best expert; slot index s = t*k + j
 *   topk_weights   float  [T, k]
 *   x              dtype  [T, d]
 *   w_gate_up      dtype  [E, d, 2I]  gate = columns [0, I), up = columns [I, 2I) ([TP-packed])
 *   w_down         dtype  [E, I, d]
 *   counts         int32  [E]
 *   offsets        int32  [E + 1]  exclusive prefix of counts; expert e owns sorted rows
 *                                  [offsets[e], offsets[e+1])
 *   sorted_to_slot int32  [R]      sorted row p came from slot sorted_to_slot[p]   (R = T*k)
 *   slot_to_sorted int32  [R]      inverse permutation (-1 for a slot whose id was invalid)
 *   x_sorted       dtype  [R, d]   x_sorted[p] = x[sorted_to_slot[p] / k]
 *   h              dtype  [R, I]   SiLU(gate) * up; stored in the layer dtype
 *   y_sorted       float  [R, d]   expert outputs in sorted order, fp32
 *   out            dtype  [T, d]
 *
 * Precision: MOE_BF16 layers take bf16 inputs and weights, accumulate in fp32 on the tensor
 * cores (tcgen05), store h as bf16 (round to nearest even), keep y_sorted in fp32 and round the
 * combined output once. MOE_F32 layers run in fp32 throughout (FFMA, no TF32).
 */
#ifndef RDG_MOE_H
#define RDG_MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; declared here so the header needs no CUDA include. */
typedef struct CUstream_st* moe_stream_t;

typedef enum moe_status {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,   /* null pointer, bad size or flag, misaligned pointer */
    MOE_ERR_UNSUPPORTED = 2,   /* valid request outside what the kernels cover (e.g. E > 256) */
    MOE_ERR_WORKSPACE = 3,     /* workspace null or smaller than the matching *_workspace_size */
    MOE_ERR_CUDA = 4,          /* a CUDA runtime/driver call or a launch failed */
    MOE_ERR_DEVICE_BOUNDS = 5, /* device saw an expert id outside [0, E); those slots skipped */
    MOE_ERR_TIMEOUT = 6        /* a device-side wait passed its time limit; kernel gave up */
} moe_status;

typedef enum moe_dtype { MOE_F32 = 0, MOE_BF16 = 1 } moe_dtype;

typedef enum moe_score_fn { MOE_SCORE_SOFTMAX = 0, MOE_SCORE_SIGMOID = 1 } moe_score_fn;

/* flags (bitwise or) */
enum {
    MOE_RENORMALIZE = 1u,          /* divide the k selected weights by their sum */
    MOE_SCALE_INPUT = 2u,          /* router weight multiplies the expert input; combine weight 1 */
    MOE_FUSE_COMBINE_WEIGHT = 4u,  /* down-projection epilogue multiplies rows by their weight */
    MOE_WEIGHTS_PACKED = 8u,       /* expert weights were repacked by moe_pack_weights */
    MOE_WGRAD_BF16 = 16u           /* moe_backward: weight gradients rounded once to bf16 */
};

/* Which expert weight a packed buffer holds. */
typedef enum moe_weight_kind { MOE_W_GATE_UP = 0, MOE_W_DOWN = 1 } moe_weight_kind;

/*
 * moe_route - router top-k gating ([EP-add]: top_k_index, top_k_weights; [EP-intro]).
 *   logits        device float [T, E], read only.
 *   topk_ids      device int32 [T, k], written: the k experts with the largest logits, in
 *                 descending logit order; equal logits go to the lower expert index; -0.0 equals
 *                 +0.0; NaN ranks below -inf. Selection compares the fp32 logits directly, so the
 *                 ids do not depend on how exp is evaluated.
 *   topk_weights  device float [T, k], written.
 *                 MOE_SCORE_SOFTMAX: exp(l_j - max) / sum over all E of exp(l_i - max); with
 *                 MOE_RENORMALIZE this is a softmax over the k selected logits.
 *                 MOE_SCORE_SIGMOID: 1 / (1 + exp(-l_j)); divided by the sum of the k selected
 *                 when MOE_RENORMALIZE is set.
 *   flags         MOE_RENORMALIZE only; other bits are MOE_ERR_INVALID_ARG.
 * Weights from a row holding NaN logits are unspecified.
 */
moe_status moe_route(const float* logits, int T, int E, int k, moe_score_fn score_fn,
                     unsigned flags, int32_t* topk_ids, float* topk_weights, moe_stream_t stream);

/*
 * moe_route_hidden - the router from hidden states: logits = x . w_router (+ bias) in fp32,
 *   then the top-k and weights of moe_route, in one kernel ([EP-intro]: a router sends each
 *   token to its experts; the workloads define the logits as x times a router weight [d, E]
 *   plus an optional per-expert bias).
 *   x             device [T, d] in dtype dt (MOE_BF16 or MOE_F32), read only.
 *   w_router      device float [d, E], row-major, read only.
 *   bias          device float [E] or NULL.
 *   logits        device float [T, E] or NULL: when given, the logits the selection used.
 *   topk_ids, topk_weights, score_fn, flags: as moe_route; for the same logits the results are
 *                 bit-identical to moe_route's.
 *   Each logit is an fp32 sum of the d products in an order fixed by the sizes (on the FP32
 *   pipes; for more than 1024 bf16 tokens on the tensor pipe with w_router split into three
 *   bf16 terms), then + bias[e]: it differs from the exact value by at most about
 *   d * 2^-22 * sum_i |x[t][i] * w_router[i][e]|, so logits closer than that may rank
 *   differently than they would under exact arithmetic. The results do not depend on timing.
 *   Constraints: 1 <= k <= E <= 256, d >= 1; pointers 16-byte aligned. T == 0 is a no-op.
 */
moe_status moe_route_hidden(const void* x, moe_dtype dt, const float* w_router,
                            const float* bias, int T, int d, int E, int k,
                            moe_score_fn score_fn, unsigned flags, float* logits,
                            int32_t* topk_ids, float* topk_weights, moe_stream_t stream);

/*
 * moe_dispatch - group the T*k routed slots by expert ([EP-dispatch]: every (token, expert)
 * pair goes to that expert; on one GPU this is a local permutation).
 *   topk_ids       device int32 [T, k], read. An id outside [0, E) sets MOE_ERR_DEVICE_BOUNDS in
 *                  the status word; that slot is left out of counts and rows and its
 *                  slot_to_sorted entry is -1.
 *   x, x_sorted    device [T, d] and [R, d] of dtype dt; both NULL = indices only.
 *   counts, offsets, sorted_to_slot, slot_to_sorted: device int32 outputs (layouts above).
 *                  Inside an expert rows keep ascending slot order, so the permutation is
 *                  deterministic (no atomics decide it).
 *   workspace      device scratch of at least moe_dispatch_workspace_size(T, E, k) bytes,
 *                  256-byte aligned; its first 4 bytes are the status word, cleared by the call.
 */
moe_status moe_dispatch(const int32_t* topk_ids, const void* x, moe_dtype dt, int T, int d, int E,
                        int k, int32_t* counts, int32_t* offsets, int32_t* sorted_to_slot,
                        int32_t* slot_to_sorted, void* x_sorted, void* workspace,
                        size_t ws_bytes, moe_stream_t stream);
size_t moe_dispatch_workspace_size(int T, int E, int k);

/*
 * moe_dispatch_noalloc - moe_dispatch without a workspace, for callers that cannot allocate
 * device memory where they call it (a plugin inside a host application that owns every device
 * allocation and hands it no allocator, or a service that forbids device allocation after
 * start-up). The pages have no counterpart to this entry point: it exists for those callers.
 *   Arguments and outputs as for moe_dispatch, minus workspace and ws_bytes. The scratch
 *   (one int32 count per (256-slot chunk, expert)) lives in a fixed device array of
 *   MOE_DISPATCH_NOALLOC_MAX_SCRATCH_INTS int32 (1 MiB) inside the library, which every GPU
 *   that loads the library holds until the process exits. Requests needing more,
 *   ceil(T*k / 256) * E > MOE_DISPATCH_NOALLOC_MAX_SCRATCH_INTS, return MOE_ERR_UNSUPPORTED
 *   before anything is enqueued; use moe_dispatch for those.
 *   No cudaMalloc, cudaFree or other allocating call is made.
 *   The first call in each CUDA context looks up the array's device address
 *   (cudaGetSymbolAddress, with that context current) and caches it per context, keyed on the
 *   context's unique id: a non-primary context on a device has its own copy of the array and
 *   gets its own address, and a context created after cudaDeviceReset is looked up afresh.
 *   Make the first call in a context before any stream capture.
 *   All calls share the array and it keeps the last call's contents (the kernels overwrite
 *   every entry before reading it). Calls whose kernels overlap on the GPU, e.g. on two
 *   streams, race on it: serialise them. There is no status word: an expert id outside [0, E)
 *   is skipped as in moe_dispatch and shows only as slot_to_sorted == -1.
 */
#define MOE_DISPATCH_NOALLOC_MAX_SCRATCH_INTS 262144
moe_status moe_dispatch_noalloc(const int32_t* topk_ids, const void* x, moe_dtype dt, int T,
                                int d, int E, int k, int32_t* counts, int32_t* offsets,
                                int32_t* sorted_to_slot, int32_t* slot_to_sorted, void* x_sorted,
                                moe_stream_t stream);

/*
 * moe_gate_up - grouped gate/up projection with SwiGLU ([TP-packed]; [EP-add] experts_forward):
 *   for each expert e and each row p in [offsets[e], offsets[e+1]):
 *     g = x_rows[p] . w_gate_up[e][:, 0:I],  u = x_rows[p] . w_gate_up[e][:, I:2I]
 *     if MOE_SCALE_INPUT: g, u *= s_p with s_p = topk_weights[sorted_to_slot[p]] (the router
 *       score applied to the expert input, [EP-intro]; applied to the fp32 accumulators, which
 *       equals scaling the input by linearity)
 *     h[p] = SiLU(g) * u, SiLU(z) = z / (1 + exp(-z)), stored in dt.
 *   x_rows     device dtype [R, d] (x_sorted, or x itself for an always-on expert).
 *   offsets    device int32 [E + 1] with offsets[0] == 0 and offsets[E] <= R, or NULL meaning one
 *              expert (E must be 1) owning all R rows. Read on the device: no host sync.
 *   sorted_to_slot, topk_weights: read only with MOE_SCALE_INPUT, else may be NULL.
 *   w_gate_up  device dtype [E, d, 2I], or packed by moe_pack_weights with MOE_WEIGHTS_PACKED.
 *   h          device dtype [R, I], written for owned rows only.
 *   flags      MOE_SCALE_INPUT, MOE_WEIGHTS_PACKED or 0.
 *   workspace  at least moe_experts_workspace_size() bytes (status word), 256-byte aligned.
 */
moe_status moe_gate_up(const void* x_rows, const int32_t* offsets, const int32_t* sorted_to_slot,
                       const float* topk_weights, moe_dtype dt, int R, int d, int E, int I,
                       const void* w_gate_up, unsigned flags, void* h, void* workspace,
                       size_t ws_bytes, moe_stream_t stream);

/*
 * moe_down - grouped down projection: y_sorted[p] = h[p] . w_down[e] (fp32), for p owned by e;
 *   with MOE_FUSE_COMBINE_WEIGHT the row is multiplied by topk_weights[sorted_to_slot[p]].
 *   h device dtype [R, I]; w_down device dtype [E, I, d] (or packed, with MOE_WEIGHTS_PACKED);
 *   y_sorted device float [R, d].
 *   offsets, sorted_to_slot, topk_weights, workspace: as for moe_gate_up.
 */
moe_status moe_down(const void* h, const int32_t* offsets, const int32_t* sorted_to_slot,
                    const float* topk_weights, moe_dtype dt, int R, int d, int E, int I,
                    const void* w_down, unsigned flags, float* y_sorted, void* workspace,
                    size_t ws_bytes, moe_stream_t stream);

/* moe_experts - moe_gate_up followed by moe_down ([EP-add] experts_forward). */
moe_status moe_experts(const void* x_sorted, const int32_t* offsets, const int32_t* sorted_to_slot,
                       const float* topk_weights, moe_dtype dt, int R, int d, int E, int I,
                       const void* w_gate_up, const void* w_down, unsigned flags, void* h,
                       float* y_sorted, void* workspace, size_t ws_bytes, moe_stream_t stream);
size_t moe_experts_workspace_size(void);

/*
 * moe_pack_weights - one-time repacking of expert weights for faster streaming (bf16 only).
 *   The pages' layout ([TP-packed]: gate_up [E, d, 2I] gate first, down [E, I, d]) makes each
 *   64 x 64 weight tile the GEMMs read a set of 64 rows of 128 bytes a full weight row apart.
 *   The packed layout stores every such tile as one contiguous 8 KB block, so the kernels read
 *   expert weights sequentially. It is a storage layout of this library, not of the pages.
 *   kind MOE_W_GATE_UP: w = [E, K=d, 2I] in the pages' layout, N = I; the gate and up halves are
 *   blocked separately. kind MOE_W_DOWN: w = [E, K=I, N=d].
 *   Layout: block (e, nb, kb) = rows [64 kb, 64 kb + 64) of the 64 columns of block nb, at rows
 *   ((e * NB + nb) * Kpad + 64 kb) of a [E * NB * Kpad, 64] bf16 matrix; Kpad = K rounded up to
 *   64; NB = ceil(N / 64) for down, 2 * ceil(I / 64) for gate_up (gate blocks first). Padding
 *   is zero. packed: device buffer of moe_packed_weights_size() bytes, 16-byte aligned.
 *   Pass MOE_WEIGHTS_PACKED to moe_gate_up / moe_down / moe_experts / moe_forward to use it
 *   (for moe_forward the shared expert's weights, if any, must be packed too, with E = 1).
 *   Results are the same as with the unpacked weights. Returns MOE_ERR_UNSUPPORTED for
 *   MOE_F32.
 */
size_t moe_packed_weights_size(moe_weight_kind kind, int E, int K, int N, moe_dtype dt);
moe_status moe_pack_weights(moe_weight_kind kind, const void* w, void* packed, moe_dtype dt,
                            int E, int K, int N, moe_stream_t stream);

/*
 * moe_combine - weighted return to token order ([EP-dispatch]: results combined with the
 * routing weights; [EP-add]: the weighted expert output for each token):
 *   out[t] = sum_{j<k} w[t, j] * y_sorted[slot_to_sorted[t*k + j]]  (+ y_shared[t])
 *   summed in fp32 in slot order, the shared row added last, rounded once to out_dt.
 *   topk_weights NULL means weight 1 (router score already applied to the input, or fused into
 *   the down projection). y_shared (device float [T, d]) may be NULL. Slots whose
 *   slot_to_sorted entry is negative contribute nothing.
 */
moe_status moe_combine(const float* y_sorted, const int32_t* slot_to_sorted,
                       const float* topk_weights, const float* y_shared, int T, int d, int k,
                       moe_dtype out_dt, void* out, moe_stream_t stream);

/*
 * moe_forward - the whole layer ([EP-add] __call__): route, dispatch, experts, combine.
 *   x, logits, weights as above; topk_ids/topk_weights/out are caller outputs.
 *   w_shared_gate_up [d, 2*Is] and w_shared_down [Is, d] (dtype dt): an always-on SwiGLU expert
 *   run on the unscaled x and added to every token before the one output rounding; both NULL
 *   (and Is == 0) for none.
 *   flags: MOE_RENORMALIZE | MOE_SCALE_INPUT | MOE_FUSE_COMBINE_WEIGHT (these two exclude
 *   each other) | MOE_WEIGHTS_PACKED (all expert weights, shared ones included, packed).
 *   workspace: at least moe_forward_workspace_size(...) bytes, 256-byte aligned. Holds counts,
 *   offsets, both permutations, x_sorted, h, y_sorted and the shared expert's h and y.
 *   Decode batches (bf16, no shared expert, T <= 16, T*k <= 256) run the whole layer as one
 *   cooperative kernel that routes in every block and streams the touched experts' weights
 *   through every SM. It leaves topk_ids/topk_weights, counts, offsets, both permutations and
 *   h as above but writes neither x_sorted nor y_sorted (the combine is folded into the down
 *   step); its counters follow the status word and its partial sums take a region at the end
 *   of the workspace (both included in moe_forward_workspace_size). MOE_FUSE_COMBINE_WEIGHT
 *   changes nothing there.
 */
moe_status moe_forward(const void* x, const float* logits, moe_dtype dt, int T, int d, int E,
                       int k, int I, moe_score_fn score_fn, unsigned flags, const void* w_gate_up,
                       const void* w_down, const void* w_shared_gate_up,
                       const void* w_shared_down, int Is, int32_t* topk_ids, float* topk_weights,
                       void* out, void* workspace, size_t ws_bytes, moe_stream_t stream);
size_t moe_forward_workspace_size(int T, int d, int E, int k, int I, int Is, moe_dtype dt);

/*
 * moe_forward_host - moe_forward for a caller whose activations live in host memory: x_host
 *   (dt [T, d]), logits_host (float [T, E]) and out_host (dt [T, d]). All work is enqueued on
 *   `stream`; the call does not wait for it, so synchronise the stream before reading out_host.
 *   A buffer that is page-locked and mapped (cudaHostAlloc, cudaMallocHost, cudaHostRegister;
 *   reached over NVLink-C2C on a Grace-Blackwell node) is used in place: the route kernel reads
 *   the logits, the dispatch (or the one-kernel decode layer) reads x and the combine writes
 *   out there, with no staging copy. Any other buffer goes through the workspace with one
 *   cudaMemcpyAsync (pageable memory makes that copy block the calling thread). With a shared
 *   expert (Is > 0) x is always staged, since its gate_up loads x with TMA. The router's ids
 *   and weights stay in the workspace. Weights, flags and errors as moe_forward; workspace:
 *   moe_forward_host_workspace_size(...) bytes, 256-byte aligned (the forward workspace
 *   followed by device room for x, logits, out, ids and weights).
 */
size_t moe_forward_host_workspace_size(int T, int d, int E, int k, int I, int Is, moe_dtype dt);
moe_status moe_forward_host(const void* x_host, const float* logits_host, moe_dtype dt, int T,
                            int d, int E, int k, int I, moe_score_fn score_fn, unsigned flags,
                            const void* w_gate_up, const void* w_down,
                            const void* w_shared_gate_up, const void* w_shared_down, int Is,
                            void* out_host, void* workspace, size_t ws_bytes,
                            moe_stream_t stream);

/*
 * Number of kernels moe_forward enqueues for these sizes (dispatch, experts and combine
 * kernels included; the status-word clear is a memset, not counted). 0 for T == 0. Batches
 * with T*k <= 1024 route and build the dispatch indices in one fused launch; decode batches
 * (see moe_forward) run one kernel in all.
 */
int moe_forward_kernel_count(moe_dtype dt, int T, int k, int Is);

/*
 * Name of the grouped GEMM kernel moe_gate_up / moe_down (and the GEMM steps of moe_forward
 * and moe_experts) launch for bf16 layers of these sizes: R routed rows over E experts
 * (grouped = 0: one group without offsets, as for a shared expert). One of
 * "tc_grouped_gemm_2sm" (256-row tiles on CTA pairs; gate_up tails of at most 128 rows with
 * the weights as the M side), "tc_grouped_gemm_swap" (weights as the MMA M side, at most 512
 * rows), "tc_grouped_gemm_swap_pair" (weights as the M side of CTA pairs: routed down);
 * "none" for R <= 0 or an unknown kind. (The training and MX forms of gate_up run the 128-row
 * kernel "tc_grouped_gemm", whose epilogue keeps the accumulators or rounds h to MXFP8.) A
 * static string; for diagnostics and benchmarks.
 */
const char* moe_gemm_kernel_name(moe_weight_kind kind, int R, int E, int grouped);

/* ============================== training: backward pass ==============================
 * [EP-intro] / [EP-dispatch]: the routing weights multiply the expert outputs, so a training
 * step differentiates the layer with respect to x, the expert weights, the routing weights and,
 * through the router's score function, the logits. Same conventions as above (caller-owned
 * memory, checks before any launch, no host sync, graph-capturable). Readings (the pages give
 * no backward formulas; each is the chain rule through the forward's steps in reverse):
 *   - a bf16 layer keeps a = x W_gate, b = x W_up (before any router scale) as bf16 for the
 *     backward pass ("ab" [R, 2I]); dy = w dout and d_ab are rounded to bf16 between kernels;
 *     weight gradients, dx_sorted and the routing gradients are fp32; dx is rounded once.
 *   - the top-k choice is piecewise constant: the logits' gradient flows only through the
 *     weights of the selected experts.
 * Layouts (row-major): dout dtype [T, d]; dy_sorted dtype [R, d]; ab, d_ab dtype [R, 2I]
 * (gate half first); dx_sorted float [R, d]; d_w_gate_up float [E, d, 2I]; d_w_down float
 * [E, I, d]; d_topk_weights float [T, k]; d_logits float [T, E]; dx dtype [T, d].
 */

/*
 * moe_gate_up_train - moe_gate_up that also stores ab[p] = [x_rows[p] . W_gate | x_rows[p] .
 *   W_up] (the fp32 accumulators before the MOE_SCALE_INPUT scale, rounded to dt) for
 *   moe_down_backward. ab device dtype [R, 2I]; other arguments as moe_gate_up.
 */
moe_status moe_gate_up_train(const void* x_rows, const int32_t* offsets,
                             const int32_t* sorted_to_slot, const float* topk_weights,
                             moe_dtype dt, int R, int d, int E, int I, const void* w_gate_up,
                             unsigned flags, void* h, void* ab, void* workspace,
                             size_t ws_bytes, moe_stream_t stream);

/*
 * moe_combine_backward - gradient of moe_combine:
 *   dy_sorted[p] = w[t, j] * dout[t] for p = slot_to_sorted[t*k + j] (w = 1 when topk_weights
 *   is NULL), computed in fp32 and stored in dt; rows of negative slot_to_sorted entries are
 *   not written.
 *   d_topk_weights[t, j] = sum_c dout[t, c] * y_sorted[p, c] (fp32, one fixed-order sum per
 *   slot; 0 for a negative entry). y_sorted is the forward's fp32 [R, d]; pass both y_sorted
 *   and d_topk_weights, or neither.
 */
moe_status moe_combine_backward(const void* dout, const float* y_sorted,
                                const int32_t* slot_to_sorted, const float* topk_weights,
                                moe_dtype dt, int T, int d, int k, void* dy_sorted,
                                float* d_topk_weights, moe_stream_t stream);

/*
 * moe_down_backward - gradient through the down projection and SwiGLU, for rows p of expert e:
 *   dh = dy_sorted[p] . w_down[e]^T (fp32); s = topk_weights[sorted_to_slot[p]] with
 *   MOE_SCALE_INPUT, else 1; a, b = ab[p] halves; g = s a, u = s b; sig = 1 / (1 + exp(-g));
 *   dg = dh u sig (1 + g (1 - sig)), du = dh g sig;
 *   d_ab[p] = [s dg | s du] stored in dt;
 *   with MOE_SCALE_INPUT also d_topk_weights[sorted_to_slot[p]] = sum_c (dg_c a_c + du_c b_c)
 *   (fp32; indexed by slot, R entries), the gradient of the score that scaled the input.
 *   flags: MOE_SCALE_INPUT, MOE_WEIGHTS_PACKED (w_down packed by moe_pack_weights).
 *   workspace: at least moe_down_backward_workspace_size(R, I, dt) bytes, 256-byte aligned.
 */
size_t moe_down_backward_workspace_size(int R, int I, moe_dtype dt);
moe_status moe_down_backward(const void* dy_sorted, const void* ab, const int32_t* offsets,
                             const int32_t* sorted_to_slot, const float* topk_weights,
                             moe_dtype dt, int R, int d, int E, int I, const void* w_down,
                             unsigned flags, void* d_ab, float* d_topk_weights, void* workspace,
                             size_t ws_bytes, moe_stream_t stream);

/*
 * moe_gate_up_backward - dx_sorted[p] = d_ab[p] . w_gate_up[e]^T (fp32 [R, d]) for rows p of
 *   expert e. flags: MOE_WEIGHTS_PACKED or 0. workspace: moe_experts_workspace_size() bytes.
 */
moe_status moe_gate_up_backward(const void* d_ab, const int32_t* offsets, moe_dtype dt, int R,
                                int d, int E, int I, const void* w_gate_up, unsigned flags,
                                float* dx_sorted, void* workspace, size_t ws_bytes,
                                moe_stream_t stream);

/*
 * moe_weight_grad - per-expert weight gradient: dw[e] = a[rows of e]^T . b[rows of e]
 *   (fp32 accumulate, fp32 out). a device dt [R, M], b device dt [R, N], dw device float
 *   [E, M, N], every expert's block written (zero for an expert with no rows). offsets as for
 *   moe_gate_up (NULL: one expert owning all R rows). M and N multiples of 8 (bf16) / 4 (fp32).
 *   (x_sorted, d_ab) gives d_w_gate_up [E, d, 2I]; (h, dy_sorted) gives d_w_down [E, I, d].
 *   workspace: moe_experts_workspace_size() bytes.
 */
moe_status moe_weight_grad(const void* a, const void* b, const int32_t* offsets, moe_dtype dt,
                           int R, int M, int N, int E, float* dw, void* workspace,
                           size_t ws_bytes, moe_stream_t stream);
/*
 * moe_weight_grad_bf16 - moe_weight_grad for bf16 a and b with dw bf16 [E, M, N]: the fp32 sum
 *   of each element rounded once to nearest even. Halves the gradient bytes written, which
 *   bind the weight gradient when experts have few rows (each dW element is M x N output for
 *   only R_e multiply-adds). Same arguments, alignment and errors as moe_weight_grad.
 */
moe_status moe_weight_grad_bf16(const void* a, const void* b, const int32_t* offsets, int R,
                                int M, int N, int E, void* dw, void* workspace, size_t ws_bytes,
                                moe_stream_t stream);

/*
 * moe_route_backward - gradient of moe_route's weights with respect to the logits, the
 *   selected ids held fixed (g = d_topk_weights[t], w = topk_weights[t], inner = sum_j w_j g_j):
 *   softmax, renormalised:   d_logits[t, ids_j] = w_j (g_j - inner), 0 for other experts;
 *   softmax over all E:      d_logits[t, m] = p_m (G_m - inner), p = softmax of the row,
 *                            G_m = g_j if m = ids_j else 0;
 *   sigmoid:                 d_logits[t, ids_j] = g_j w_j (1 - w_j);
 *   sigmoid, renormalised:   d_logits[t, ids_j] = (g_j - inner) / S * sig_j (1 - sig_j),
 *                            sig_j = 1 / (1 + exp(-l_j)), S = sum_j sig_j.
 *   flags: MOE_RENORMALIZE or 0 (as given to moe_route). d_logits device float [T, E], all of
 *   it written.
 */
moe_status moe_route_backward(const float* logits, const int32_t* topk_ids,
                              const float* topk_weights, const float* d_topk_weights, int T,
                              int E, int k, moe_score_fn score_fn, unsigned flags,
                              float* d_logits, moe_stream_t stream);

/*
 * moe_forward_train - moe_forward for a training step: the same outputs, plus what
 *   moe_backward reads, kept in its workspace (counts, offsets, both permutations, x_sorted,
 *   h, y_sorted and ab; for a shared expert its h and ab). Never takes the one-kernel decode
 *   path; MOE_FUSE_COMBINE_WEIGHT returns MOE_ERR_UNSUPPORTED (the routing weights' gradient
 *   needs the unweighted y_sorted). workspace: moe_forward_train_workspace_size(...) bytes.
 */
size_t moe_forward_train_workspace_size(int T, int d, int E, int k, int I, int Is,
                                        moe_dtype dt);
moe_status moe_forward_train(const void* x, const float* logits, moe_dtype dt, int T, int d,
                             int E, int k, int I, moe_score_fn score_fn, unsigned flags,
                             const void* w_gate_up, const void* w_down,
                             const void* w_shared_gate_up, const void* w_shared_down, int Is,
                             int32_t* topk_ids, float* topk_weights, void* out, void* workspace,
                             size_t ws_bytes, moe_stream_t stream);

/*
 * moe_backward - the whole backward pass of the layer moe_forward_train ran (same x, logits,
 *   weights, flags, topk_ids/topk_weights and its workspace `fwd_workspace`, unchanged):
 *   combine backward, the down and gate/up projections' weight and input gradients (the
 *   SwiGLU backward in between), the shared expert's (dy = dout), the transpose of the
 *   dispatch (dx[t] = sum_j dx_sorted[slot_to_sorted[t*k + j]] + the shared expert's, fp32
 *   sum, rounded once to dt), then the router backward.
 *   Outputs: dx dtype [T, d]; d_w_gate_up, d_w_down (and the shared d_w_shared_gate_up [d, 2Is],
 *   d_w_shared_down [Is, d]) fp32; d_topk_weights fp32 [T, k] (may be NULL); d_logits fp32
 *   [T, E] (may be NULL; needs logits). flags: MOE_RENORMALIZE | MOE_SCALE_INPUT |
 *   MOE_WEIGHTS_PACKED | MOE_WGRAD_BF16. With MOE_WGRAD_BF16 (bf16 layers) the four weight
 *   gradient pointers hold bf16 [same shapes] instead of fp32: each element's fp32 sum rounded
 *   once (as for bf16 parameters whose gradients keep their dtype). workspace:
 *   moe_backward_workspace_size(...) bytes, 256-byte aligned.
 */
size_t moe_backward_workspace_size(int T, int d, int E, int k, int I, int Is, moe_dtype dt);
moe_status moe_backward(const void* dout, const void* x, const float* logits, moe_dtype dt, int T,
                        int d, int E, int k, int I, moe_score_fn score_fn, unsigned flags,
                        const void* w_gate_up, const void* w_down, const void* w_shared_gate_up,
                        const void* w_shared_down, int Is, const int32_t* topk_ids,
                        const float* topk_weights, const void* fwd_workspace,
                        size_t fwd_ws_bytes, void* dx, float* d_w_gate_up, float* d_w_down,
                        float* d_w_shared_gate_up, float* d_w_shared_down,
                        float* d_topk_weights, float* d_logits, void* workspace,
                        size_t ws_bytes, moe_stream_t stream);
/* Number of kernels moe_backward enqueues (memsets not counted). */
int moe_backward_kernel_count(int T, int k, int Is, unsigned flags, int want_logits);

/* ===================== block-scaled low precision (MX formats) =====================
 * The pages name FP8 activations times FP4 weights with block scales as the low-precision
 * expert variant of the newest GPUs ("Expert parallelism", the Mega MoE paragraph) without a
 * format; these calls follow the OCP Microscaling (MX) specification v1.0:
 *   - blocks of 32 consecutive elements along the reduction axis K share one E8M0 scale 2^s,
 *     s = floor(log2(max |v|)) - emax (emax 2 for FP4 E2M1, 8 for FP8 E4M3), clamped to
 *     [-127, 127] (-127 for an all-zero block), stored as s + 127;
 *   - elements are v / 2^s rounded to nearest even and saturated at the largest finite value
 *     (6 for E2M1, 448 for E4M3).
 * The MX layer (moe_forward_mx): expert weights MXFP4 (blocks along d for gate_up, along I for
 * down); x rounded to MXFP8 (blocks along d) once per token; the SwiGLU activation h rounded
 * to MXFP8 (blocks along I) from its fp32 value, in place of the bf16 layer's bf16 rounding;
 * accumulation in fp32; y_sorted, the combine and the output as in the bf16 layer. bf16
 * layers only.
 *
 * MX weight buffer of one kind (gate_up: K = d, columns 2I, its gate and up halves blocked
 * separately; down: K = I, columns d; N as for moe_pack_weights), in blocks of 64 columns x 32
 * K rows: block (e, nb, kb) holds 1 KB of E2M1 codes at ((e * NB + nb) * KB + kb) * 1024, laid
 * out as the A fragments of mma.m16n8k16 (256 words [k-step (2)][16-column m-tile (4)][lane
 * (32)]; word byte hi + 2 kh, nibble bit holds column 16 mt + (lane >> 2) + 8 hi and row
 * 16 ks + 2 (lane & 3) + bit + 8 kh of the block), and its 64 E8M0 scales (per column) at
 * E * NB * KB * 1024 + ((e * NB + nb) * KB + kb) * 64. NB = ceil(N / 64) for down,
 * 2 ceil(I / 64) for gate_up (gate blocks first), KB = ceil(K / 32); padding holds code 0.
 * 16-byte aligned; moe_mx_weights_size(...) bytes.
 */
size_t moe_mx_weights_size(moe_weight_kind kind, int E, int K, int N);
/* bf16 weights in the pages' layout ([E, d, 2I] or [E, I, d]) -> MX buffer. */
moe_status moe_quantize_weights_mx(moe_weight_kind kind, const void* w, void* mx, int E, int K,
                                   int N, moe_stream_t stream);
/* MX buffer -> bf16 weights (exact: every MXFP4 value is a bf16 value). */
moe_status moe_dequantize_weights_mx(moe_weight_kind kind, const void* mx, void* w, int E, int K,
                                     int N, moe_stream_t stream);
/*
 * moe_quantize_rows_mx - bf16 rows [R, K] (K a multiple of 8) to MXFP8 along K: x_out (bf16
 *   [R, K], the rounded values, may equal x, may be NULL), codes (uint8 E4M3 [R, K]) and
 *   scales (uint8 E8M0 [R, ceil(K / 32)]) (both or neither).
 */
moe_status moe_quantize_rows_mx(const void* x, int R, int K, void* x_out, void* codes,
                                void* scales, moe_stream_t stream);
/*
 * moe_forward_mx - the whole layer with MX weights (moe_forward's arguments; w_gate_up_mx /
 *   w_down_mx and the shared expert's (E = 1) are MX buffers). flags: MOE_RENORMALIZE |
 *   MOE_SCALE_INPUT | MOE_FUSE_COMBINE_WEIGHT. The experts that received rows get their weights
 *   dequantized into the workspace and run on the bf16 tensor-core GEMMs (the MX values are
 *   exact in bf16). workspace: moe_forward_mx_workspace_size(...) bytes, 256-byte aligned; its
 *   head has moe_forward's layout without the decode regions.
 */
size_t moe_forward_mx_workspace_size(int T, int d, int E, int k, int I, int Is);
moe_status moe_forward_mx(const void* x, const float* logits, int T, int d, int E, int k, int I,
                          moe_score_fn score_fn, unsigned flags, const void* w_gate_up_mx,
                          const void* w_down_mx, const void* w_shared_gate_up_mx,
                          const void* w_shared_down_mx, int Is, int32_t* topk_ids,
                          float* topk_weights, void* out, void* workspace, size_t ws_bytes,
                          moe_stream_t stream);

/*
 * MX on the block-scaled tensor cores ("Expert parallelism", the Mega MoE paragraph: FP8
 * activations times FP4 weights with block scales on the newest GPUs). The same MX numerics as
 * moe_forward_mx (x and h MXFP8, weights MXFP4, fp32 accumulation), computed by
 * tcgen05.mma.kind::mxf8f6f4.block_scale: the tensor cores multiply the E4M3 and E2M1 codes and
 * apply both E8M0 block scales themselves; nothing is dequantized.
 *
 * MX tensor-core weight buffer of one kind (gate_up: K = d, logical columns C = 2I, gate
 * columns first; down: K = I, C = d), N (= I or d) and K multiples of 32, Kp = K rounded up to
 * 128:
 *   codes: for group e and logical column c, Kp / 2 bytes of E2M1 codes along K (element k in
 *     the low nibble of byte k / 2 when k is even), at (e * C + c) * Kp / 2; zero past K;
 *   scales, from sf_off = (E * C * Kp / 2) rounded up to 1024: 512-byte atoms, one per
 *     (e, 128-column block cb, 128-element K chunk kc) at sf_off + ((e * CB + cb) * (Kp / 128)
 *     + kc) * 512; byte 16 (n % 32) + 4 (n / 32) + j holds the scale (s + 127) of the block's
 *     column n at K block 4 kc + j, 127 past the end of the columns or of K. Column blocks:
 *     gate_up ceil(I / 128) for the gate half then as many for the up half (CB = 2 ceil(I/128));
 *     down ceil(d / 128).
 *   256-byte aligned; moe_mx_tc_weights_size(...) bytes (0: unsupported sizes).
 */
size_t moe_mx_tc_weights_size(moe_weight_kind kind, int E, int K, int N);
/* bf16 weights in the pages' layout ([E, d, 2I] or [E, I, d]) -> MX tensor-core buffer (the
 * same codes and scales moe_quantize_weights_mx decides, in this layout). */
moe_status moe_quantize_weights_mx_tc(moe_weight_kind kind, const void* w, void* mx, int E,
                                      int K, int N, moe_stream_t stream);
/* MX tensor-core buffer -> bf16 weights [E, K, C] (exact). */
moe_status moe_dequantize_weights_mx_tc(moe_weight_kind kind, const void* mx, void* w, int E,
                                        int K, int N, moe_stream_t stream);
/*
 * moe_forward_mx_tc - the MX layer on the block-scaled tensor cores (moe_forward_mx's
 *   arguments, weights in the MX tensor-core layout, d, I and Is multiples of 32; flags:
 *   MOE_RENORMALIZE | MOE_SCALE_INPUT). Route, dispatch indices, one kernel that rounds each
 *   token's x to MXFP8 once and writes it to every row it was sent to, the gate_up GEMM (h
 *   rounded to MXFP8 in its epilogue), the down GEMM, the combine.
 *   Decode batches (no shared expert, T <= 16, T*k <= 256, d <= 2048, I <= 4096) run the whole
 *   layer as one cooperative kernel instead (same arithmetic: the weights are the M side of the
 *   block-scaled MMAs and the tokens the N side; h's 128-column blocks are owned by one SM each;
 *   the weighted sums of each run of an expert's h blocks on one SM are fp32 partials, added
 *   per token in a fixed order and rounded once). It writes the routed rows' x and h codes and
 *   atoms as the steps do, but not y_sorted. moe_forward_mx_tc_kernel_count says which runs.
 *   workspace: moe_forward_mx_tc_workspace_size(...) bytes, 256-byte aligned: the status word
 *   (256 B; the one-kernel layer keeps a counter at byte 128 of it), then, each rounded up to
 *   256 bytes: counts [E], offsets [E+1], dispatch scratch, sorted_to_slot [R], slot_to_sorted
 *   [R], x codes [Rp][d], x scale atoms [Rp/128][ceil(d/128)], h codes [Rp][I], h scale atoms
 *   [Rp/128][ceil(I/128)], y_sorted fp32 [R][d], with a shared expert its x codes [Tp][d] and
 *   atoms, h codes [Tp][Is] and atoms, y fp32 [T][d], and for decode batches the one-kernel
 *   layer's fp32 partials [ceil(I/128)][R][d].
 *   Rp = R rounded up to 128 plus 128 E, Tp = T rounded up to 128; expert e's rows occupy padded
 *   rows from poff[e] = sum over e' < e of ceil(count[e'] / 128) * 128; an atom's byte
 *   16 (m % 32) + 4 (m / 32) + j holds the scale of row m of its 128-row block at K block j of
 *   its 128-element chunk.
 */
/*
 * The steps of moe_forward_mx_tc on their own (buffers in the layouts described above; Rp =
 * R rounded up to 128 plus 128 E with offsets, R rounded up to 128 for one group without):
 *   moe_mx_tc_rows: x [T, d] bf16 to MXFP8, written to the padded row of each routed slot
 *     (codes [Rp][d], scale atoms; needs topk_ids, slot_to_sorted and offsets from
 *     moe_dispatch) and/or to row t of one unpermuted group (codes_sh [Tp][d], atoms).
 *   moe_gate_up_mx_tc: h (codes [Rp][I] and atoms) from x codes/atoms and the gate_up weights
 *     (flags: MOE_SCALE_INPUT, which needs sorted_to_slot and topk_weights).
 *   moe_down_mx_tc: y_sorted fp32 [R][d] (unpadded sorted rows) from h codes/atoms.
 *   offsets NULL: one group (E = 1). workspace: >= 256 bytes, 256-byte aligned (status word).
 */
moe_status moe_mx_tc_rows(const void* x, int T, int d, int k, int E, const int32_t* topk_ids,
                          const int32_t* slot_to_sorted, const int32_t* offsets, void* codes,
                          void* sf, void* codes_sh, void* sf_sh, moe_stream_t stream);
moe_status moe_gate_up_mx_tc(const void* x_codes, const void* x_sf, const int32_t* offsets,
                             const int32_t* sorted_to_slot, const float* topk_weights, int R,
                             int d, int E, int I, const void* w_gate_up_mx, unsigned flags,
                             void* h_codes, void* h_sf, void* workspace, size_t ws_bytes,
                             moe_stream_t stream);
moe_status moe_down_mx_tc(const void* h_codes, const void* h_sf, const int32_t* offsets, int R,
                          int I, int E, int d, const void* w_down_mx, float* y_sorted,
                          void* workspace, size_t ws_bytes, moe_stream_t stream);
size_t moe_forward_mx_tc_workspace_size(int T, int d, int E, int k, int I, int Is);
/* Number of kernels moe_forward_mx_tc enqueues for these sizes (1: the one-kernel decode
 * layer; the status-word clear is a memset, not counted). 0 for T == 0. */
int moe_forward_mx_tc_kernel_count(int T, int d, int k, int I, int Is);
moe_status moe_forward_mx_tc(const void* x, const float* logits, int T, int d, int E, int k,
                             int I, moe_score_fn score_fn, unsigned flags,
                             const void* w_gate_up_mx, const void* w_down_mx,
                             const void* w_shared_gate_up_mx, const void* w_shared_down_mx,
                             int Is, int32_t* topk_ids, float* topk_weights, void* out,
                             void* workspace, size_t ws_bytes, moe_stream_t stream);

/*
 * moe_read_device_status - synchronise `stream`, then return the status word the kernels of
 * the last call that used `workspace` left there (MOE_OK if none). Diagnostics only.
 */
moe_status moe_read_device_status(const void* workspace, moe_stream_t stream);

/* Static text for a status code. */
const char* moe_status_string(moe_status status);

/*
 * moe_debug_set_gemm_stall_ns - test hook for the bounded-wait path of the tcgen05 kernels
 * (no counterpart on the pages: it exists to show that an expired device wait ends the kernel
 * cleanly). From the next launch on, the 128-row gate_up kernel (the one moe_gate_up_train,
 * moe_forward_train and the MX layer run) makes its MMA issuer first wait `ns` nanoseconds on
 * a barrier that nothing completes. When that wait runs out the kernel takes the path of any
 * expired wait: it records MOE_ERR_TIMEOUT in the call's status word, stops its other roles,
 * lets its own copies land, frees its tensor memory and returns; the stream goes on and the
 * context stays usable. Its outputs are then unspecified. 0 (the default) turns the hook off.
 * Process-wide and read at launch: set it only while no other thread launches these kernels.
 */
void moe_debug_set_gemm_stall_ns(uint32_t ns);

#ifdef __cplusplus
}
#endif

#endif /* RDG_MOE_H */
