"""Python binding of libmoe (ctypes). Argument marshalling only: every step runs in the library's
CUDA kernels. Tensors are PyTorch CUDA tensors (PyTorch provides device memory and streams);
outputs and workspaces not passed in are allocated here with torch.

The functions keep the C names: moe_route, moe_dispatch, moe_gate_up, moe_down, moe_experts,
moe_combine, moe_forward. A non-zero status raises MoEError. There is no CPU fallback: if the
library is missing, loading raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe.so")

SOFTMAX, SIGMOID = 0, 1
RENORMALIZE, SCALE_INPUT, FUSE_COMBINE_WEIGHT, WEIGHTS_PACKED, WGRAD_BF16 = 1, 2, 4, 8, 16
W_GATE_UP, W_DOWN = 0, 1
F32, BF16 = 0, 1
STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED",
          3: "MOE_ERR_WORKSPACE", 4: "MOE_ERR_CUDA", 5: "MOE_ERR_DEVICE_BOUNDS",
          6: "MOE_ERR_TIMEOUT"}

# name -> (restype, argtypes)
_P, _I, _U, _S = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint, ctypes.c_size_t
SIGNATURES = {
    "moe_route": (_I, [_P, _I, _I, _I, _I, _U, _P, _P, _P]),
    "moe_route_hidden": (_I, [_P, _I, _P, _P, _I, _I, _I, _I, _I, _U, _P, _P, _P, _P]),
    "moe_dispatch": (_I, [_P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _S, _P]),
    "moe_dispatch_workspace_size": (_S, [_I, _I, _I]),
    "moe_dispatch_noalloc": (_I, [_P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P]),
    "moe_gate_up": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _U, _P, _P, _S, _P]),
    "moe_down": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _U, _P, _P, _S, _P]),
    "moe_experts": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _U, _P, _P, _P, _S, _P]),
    "moe_experts_workspace_size": (_S, []),
    "moe_combine": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _P, _P]),
    "moe_packed_weights_size": (_S, [_I, _I, _I, _I, _I]),
    "moe_pack_weights": (_I, [_I, _P, _P, _I, _I, _I, _I, _P]),
    "moe_forward": (_I, [_P, _P, _I, _I, _I, _I, _I, _I, _I, _U, _P, _P, _P, _P, _I, _P, _P,
                         _P, _P, _S, _P]),
    "moe_forward_workspace_size": (_S, [_I, _I, _I, _I, _I, _I, _I]),
    "moe_forward_host": (_I, [_P, _P, _I, _I, _I, _I, _I, _I, _I, _U, _P, _P, _P, _P, _I, _P,
                              _P, _S, _P]),
    "moe_forward_host_workspace_size": (_S, [_I, _I, _I, _I, _I, _I, _I]),
    "moe_forward_kernel_count": (_I, [_I, _I, _I, _I]),
    "moe_gemm_kernel_name": (ctypes.c_char_p, [_I, _I, _I, _I]),
    "moe_gate_up_train": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _U, _P, _P, _P, _S,
                               _P]),
    "moe_combine_backward": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _P]),
    "moe_down_backward_workspace_size": (_S, [_I, _I, _I]),
    "moe_down_backward": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _U, _P, _P, _P, _S,
                               _P]),
    "moe_gate_up_backward": (_I, [_P, _P, _I, _I, _I, _I, _I, _P, _U, _P, _P, _S, _P]),
    "moe_weight_grad": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _S, _P]),
    "moe_weight_grad_bf16": (_I, [_P, _P, _P, _I, _I, _I, _I, _P, _P, _S, _P]),
    "moe_route_backward": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _U, _P, _P]),
    "moe_forward_train_workspace_size": (_S, [_I, _I, _I, _I, _I, _I, _I]),
    "moe_forward_train": (_I, [_P, _P, _I, _I, _I, _I, _I, _I, _I, _U, _P, _P, _P, _P, _I, _P,
                               _P, _P, _P, _S, _P]),
    "moe_backward_workspace_size": (_S, [_I, _I, _I, _I, _I, _I, _I]),
    "moe_backward": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _U, _P, _P, _P, _P, _I, _P,
                          _P, _P, _S, _P, _P, _P, _P, _P, _P, _P, _P, _S, _P]),
    "moe_backward_kernel_count": (_I, [_I, _I, _I, _U, _I]),
    "moe_mx_weights_size": (_S, [_I, _I, _I, _I]),
    "moe_quantize_weights_mx": (_I, [_I, _P, _P, _I, _I, _I, _P]),
    "moe_dequantize_weights_mx": (_I, [_I, _P, _P, _I, _I, _I, _P]),
    "moe_quantize_rows_mx": (_I, [_P, _I, _I, _P, _P, _P, _P]),
    "moe_forward_mx_workspace_size": (_S, [_I, _I, _I, _I, _I, _I]),
    "moe_forward_mx": (_I, [_P, _P, _I, _I, _I, _I, _I, _I, _U, _P, _P, _P, _P, _I, _P, _P, _P,
                            _P, _S, _P]),
    "moe_mx_tc_weights_size": (_S, [_I, _I, _I, _I]),
    "moe_quantize_weights_mx_tc": (_I, [_I, _P, _P, _I, _I, _I, _P]),
    "moe_dequantize_weights_mx_tc": (_I, [_I, _P, _P, _I, _I, _I, _P]),
    "moe_mx_tc_rows": (_I, [_P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P]),
    "moe_gate_up_mx_tc": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _U, _P, _P, _P, _S,
                               _P]),
    "moe_down_mx_tc": (_I, [_P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _S, _P]),
    "moe_forward_mx_tc_workspace_size": (_S, [_I, _I, _I, _I, _I, _I]),
    "moe_forward_mx_tc_kernel_count": (_I, [_I, _I, _I, _I, _I]),
    "moe_forward_mx_tc": (_I, [_P, _P, _I, _I, _I, _I, _I, _I, _U, _P, _P, _P, _P, _I, _P, _P,
                               _P, _P, _S, _P]),
    "moe_read_device_status": (_I, [_P, _P]),
    "moe_status_string": (ctypes.c_char_p, [_I]),
    "moe_debug_set_gemm_stall_ns": (None, [ctypes.c_uint32]),
}

_lib = None


class MoEError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {STATUS.get(status, status)}")


def lib() -> ctypes.CDLL:
    """Load libmoe.so (built in-tree by routing_dispatch_grouped_gb300.build)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with "
                              "`python -m routing_dispatch_grouped_gb300.build`")
        cdll = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(cdll, name)
            f.restype, f.argtypes = res, args
        _lib = cdll
    return _lib


def _check(fn: str, st: int):
    if st != 0:
        raise MoEError(fn, st)


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _need(t: torch.Tensor, name: str):
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor")
    return t


class PackedWeights:
    """Expert weights repacked by moe_pack_weights (bf16): `data` is the packed buffer, kind is
    W_GATE_UP (logical [E, K=d, 2I], N = I) or W_DOWN (logical [E, K=I, N=d])."""

    def __init__(self, data: torch.Tensor, kind: int, E: int, K: int, N: int, tc=False):
        self.data, self.kind, self.E, self.K, self.N = data, kind, E, K, N
        self.tc = tc  # True: the MX tensor-core layout (moe_quantize_weights_mx_tc)

    def data_ptr(self):
        return self.data.data_ptr()


def moe_packed_weights_size(kind, E, K, N) -> int:
    return lib().moe_packed_weights_size(kind, E, K, N, BF16)


def pack_weights(w: torch.Tensor, kind: int, stream=None) -> PackedWeights:
    """Repack gate_up ([E, d, 2I] or [d, 2I]) or down ([E, I, d] or [I, d]) bf16 weights."""
    _need(w, "w")
    w3 = w.unsqueeze(0) if w.dim() == 2 else w
    E, K, C = w3.shape
    N = C // 2 if kind == W_GATE_UP else C
    out = torch.empty(moe_packed_weights_size(kind, E, K, N), dtype=torch.uint8,
                      device=w.device)
    _check("moe_pack_weights", lib().moe_pack_weights(kind, _p(w3), _p(out), _dt(w3), E, K, N,
                                                      _stream(stream)))
    return PackedWeights(out, kind, E, K, N)


def _w_dims(w, kind):
    """(E, K, N, flag) of a weight argument, packed or not."""
    if isinstance(w, PackedWeights):
        assert w.kind == kind, "packed weights of the other kind"
        return w.E, w.K, w.N, WEIGHTS_PACKED
    E, K, C = w.shape
    return E, K, (C // 2 if kind == W_GATE_UP else C), 0


def _workspace(nbytes: int, device) -> torch.Tensor:
    # torch's caching allocator returns blocks aligned to at least 512 bytes
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


# ------------------------------------------------------------------------------------------------
def moe_route(logits, k, score_fn=SOFTMAX, renormalize=True, topk_ids=None, topk_weights=None,
              stream=None):
    _need(logits, "logits")
    T, E = logits.shape
    dev = logits.device
    ids = topk_ids if topk_ids is not None else torch.empty(T, k, dtype=torch.int32, device=dev)
    w = topk_weights if topk_weights is not None else torch.empty(T, k, dtype=torch.float32,
                                                                  device=dev)
    _check("moe_route", lib().moe_route(_p(logits), T, E, k, score_fn,
                                        RENORMALIZE if renormalize else 0, _p(ids), _p(w),
                                        _stream(stream)))
    return ids, w


def moe_route_hidden(x, w_router, k, score_fn=SOFTMAX, renormalize=True, bias=None,
                     logits=None, topk_ids=None, topk_weights=None, want_logits=True,
                     stream=None):
    """Router logits x @ w_router (+ bias) and the top-k in one kernel. Returns
    (topk_ids, topk_weights, logits or None)."""
    _need(x, "x")
    _need(w_router, "w_router")
    T, d = x.shape
    E = w_router.shape[1]
    dev = x.device
    ids = topk_ids if topk_ids is not None else torch.empty(T, k, dtype=torch.int32, device=dev)
    w = topk_weights if topk_weights is not None else torch.empty(T, k, dtype=torch.float32,
                                                                  device=dev)
    if logits is None and want_logits:
        logits = torch.empty(T, E, dtype=torch.float32, device=dev)
    _check("moe_route_hidden", lib().moe_route_hidden(
        _p(x), _dt(x), _p(w_router), _p(bias), T, d, E, k, score_fn,
        RENORMALIZE if renormalize else 0, _p(logits), _p(ids), _p(w), _stream(stream)))
    return ids, w, logits


def moe_dispatch_workspace_size(T, E, k) -> int:
    return lib().moe_dispatch_workspace_size(T, E, k)


def moe_dispatch(topk_ids, E, x=None, workspace=None, out=None, stream=None):
    """Returns dict(counts, offsets, sorted_to_slot, slot_to_sorted, x_sorted, workspace)."""
    _need(topk_ids, "topk_ids")
    T, k = topk_ids.shape
    R = T * k
    dev = topk_ids.device
    o = dict(out or {})
    o.setdefault("counts", torch.empty(E, dtype=torch.int32, device=dev))
    o.setdefault("offsets", torch.empty(E + 1, dtype=torch.int32, device=dev))
    o.setdefault("sorted_to_slot", torch.empty(R, dtype=torch.int32, device=dev))
    o.setdefault("slot_to_sorted", torch.empty(R, dtype=torch.int32, device=dev))
    d, dt = 0, BF16
    if x is not None:
        _need(x, "x")
        d, dt = x.shape[1], _dt(x)
        o.setdefault("x_sorted", torch.empty(R, d, dtype=x.dtype, device=dev))
    else:
        o["x_sorted"] = None
    ws = workspace if workspace is not None else _workspace(moe_dispatch_workspace_size(T, E, k),
                                                            dev)
    _check("moe_dispatch", lib().moe_dispatch(
        _p(topk_ids), _p(x), dt, T, d, E, k, _p(o["counts"]), _p(o["offsets"]),
        _p(o["sorted_to_slot"]), _p(o["slot_to_sorted"]), _p(o["x_sorted"]), _p(ws),
        ws.numel(), _stream(stream)))
    o["workspace"] = ws
    return o


def moe_experts_workspace_size() -> int:
    return lib().moe_experts_workspace_size()


def moe_gate_up(x_rows, offsets, w_gate_up, sorted_to_slot=None, topk_weights=None,
                scale_input=False, h=None, workspace=None, stream=None):
    _need(x_rows, "x_rows")
    R, d = x_rows.shape
    E, _, I, pk = _w_dims(w_gate_up, W_GATE_UP)
    dev = x_rows.device
    h = h if h is not None else torch.empty(R, I, dtype=x_rows.dtype, device=dev)
    ws = workspace if workspace is not None else _workspace(moe_experts_workspace_size(), dev)
    _check("moe_gate_up", lib().moe_gate_up(
        _p(x_rows), _p(offsets), _p(sorted_to_slot), _p(topk_weights), _dt(x_rows), R, d, E, I,
        _p(w_gate_up), (SCALE_INPUT if scale_input else 0) | pk, _p(h), _p(ws), ws.numel(),
        _stream(stream)))
    return h


def moe_down(h, offsets, w_down, sorted_to_slot=None, topk_weights=None, fuse_weight=False,
             y_sorted=None, workspace=None, stream=None):
    _need(h, "h")
    R, I = h.shape
    E, _, d, pk = _w_dims(w_down, W_DOWN)
    dev = h.device
    y = y_sorted if y_sorted is not None else torch.empty(R, d, dtype=torch.float32, device=dev)
    ws = workspace if workspace is not None else _workspace(moe_experts_workspace_size(), dev)
    _check("moe_down", lib().moe_down(
        _p(h), _p(offsets), _p(sorted_to_slot), _p(topk_weights), _dt(h), R, d, E, I,
        _p(w_down), (FUSE_COMBINE_WEIGHT if fuse_weight else 0) | pk, _p(y), _p(ws), ws.numel(),
        _stream(stream)))
    return y


def moe_experts(x_sorted, offsets, w_gate_up, w_down, sorted_to_slot=None, topk_weights=None,
                flags=0, h=None, y_sorted=None, workspace=None, stream=None):
    _need(x_sorted, "x_sorted")
    R, d = x_sorted.shape
    E, _, I, pk = _w_dims(w_gate_up, W_GATE_UP)
    flags |= pk
    dev = x_sorted.device
    h = h if h is not None else torch.empty(R, I, dtype=x_sorted.dtype, device=dev)
    y = y_sorted if y_sorted is not None else torch.empty(R, d, dtype=torch.float32, device=dev)
    ws = workspace if workspace is not None else _workspace(moe_experts_workspace_size(), dev)
    _check("moe_experts", lib().moe_experts(
        _p(x_sorted), _p(offsets), _p(sorted_to_slot), _p(topk_weights), _dt(x_sorted), R, d, E,
        I, _p(w_gate_up), _p(w_down), flags, _p(h), _p(y), _p(ws), ws.numel(), _stream(stream)))
    return h, y


def moe_combine(y_sorted, slot_to_sorted, k, out_dtype, topk_weights=None, y_shared=None,
                out=None, stream=None):
    _need(y_sorted, "y_sorted")
    R, d = y_sorted.shape
    T = slot_to_sorted.numel() // k
    out = out if out is not None else torch.empty(T, d, dtype=out_dtype, device=y_sorted.device)
    _check("moe_combine", lib().moe_combine(
        _p(y_sorted), _p(slot_to_sorted), _p(topk_weights), _p(y_shared), T, d, k, _dt(out),
        _p(out), _stream(stream)))
    return out


def moe_forward_workspace_size(T, d, E, k, I, Is, dtype) -> int:
    return lib().moe_forward_workspace_size(T, d, E, k, I, Is, BF16 if dtype == torch.bfloat16
                                            else F32)


def moe_forward_kernel_count(T, k, Is, dtype=torch.bfloat16) -> int:
    return lib().moe_forward_kernel_count(BF16 if dtype == torch.bfloat16 else F32, T, k, Is)


def moe_gemm_kernel_name(kind, R, E, grouped=True) -> str:
    """The grouped GEMM kernel a bf16 gate_up (kind W_GATE_UP) or down (W_DOWN) call of R rows
    over E experts launches."""
    return lib().moe_gemm_kernel_name(kind, R, E, 1 if grouped else 0).decode()


def moe_forward(x, logits, w_gate_up, w_down, k, score_fn=SOFTMAX, flags=RENORMALIZE,
                w_shared_gate_up=None, w_shared_down=None, out=None, topk_ids=None,
                topk_weights=None, workspace=None, stream=None):
    """The whole layer. Returns (out, topk_ids, topk_weights, workspace)."""
    _need(x, "x")
    _need(logits, "logits")
    T, d = x.shape
    E, _, I, pk = _w_dims(w_gate_up, W_GATE_UP)
    flags |= pk
    Is = 0
    if w_shared_gate_up is not None:
        Is = (w_shared_gate_up.N if isinstance(w_shared_gate_up, PackedWeights)
              else w_shared_gate_up.shape[-1] // 2)
    dev = x.device
    out = out if out is not None else torch.empty(T, d, dtype=x.dtype, device=dev)
    ids = topk_ids if topk_ids is not None else torch.empty(T, k, dtype=torch.int32, device=dev)
    w = topk_weights if topk_weights is not None else torch.empty(T, k, dtype=torch.float32,
                                                                  device=dev)
    ws = workspace if workspace is not None else _workspace(
        moe_forward_workspace_size(T, d, E, k, I, Is, x.dtype), dev)
    _check("moe_forward", lib().moe_forward(
        _p(x), _p(logits), _dt(x), T, d, E, k, I, score_fn, flags, _p(w_gate_up), _p(w_down),
        _p(w_shared_gate_up), _p(w_shared_down), Is, _p(ids), _p(w), _p(out), _p(ws), ws.numel(),
        _stream(stream)))
    return out, ids, w, ws


def moe_forward_host_workspace_size(T, d, E, k, I, Is, dtype) -> int:
    return lib().moe_forward_host_workspace_size(T, d, E, k, I, Is,
                                                 BF16 if dtype == torch.bfloat16 else F32)


def moe_forward_host(x_host, logits_host, w_gate_up, w_down, k, score_fn=SOFTMAX,
                     flags=RENORMALIZE, w_shared_gate_up=None, w_shared_down=None, out=None,
                     workspace=None, stream=None, device=None):
    """The whole layer on host activations (CPU tensors): pinned ones are read and written in
    place by the kernels, pageable ones copied in and out by the library on `stream`. Returns
    (out_host, workspace); synchronise the stream before reading out_host."""
    if x_host.is_cuda or logits_host.is_cuda:
        raise ValueError("moe_forward_host takes host tensors")
    x_host, logits_host = x_host.contiguous(), logits_host.contiguous()
    T, d = x_host.shape
    E, _, I, pk = _w_dims(w_gate_up, W_GATE_UP)
    flags |= pk
    Is = 0
    if w_shared_gate_up is not None:
        Is = (w_shared_gate_up.N if isinstance(w_shared_gate_up, PackedWeights)
              else w_shared_gate_up.shape[-1] // 2)
    dev = device if device is not None else torch.device("cuda", torch.cuda.current_device())
    out = out if out is not None else torch.empty(T, d, dtype=x_host.dtype).pin_memory()
    ws = workspace if workspace is not None else _workspace(
        moe_forward_host_workspace_size(T, d, E, k, I, Is, x_host.dtype), dev)
    _check("moe_forward_host", lib().moe_forward_host(
        _p(x_host), _p(logits_host), _dt(x_host), T, d, E, k, I, score_fn, flags,
        _p(w_gate_up), _p(w_down), _p(w_shared_gate_up), _p(w_shared_down), Is, _p(out), _p(ws),
        ws.numel(), _stream(stream)))
    return out, ws


def moe_read_device_status(workspace, stream=None) -> int:
    return lib().moe_read_device_status(_p(workspace), _stream(stream))


def forward_workspace_views(ws: torch.Tensor, T, d, E, k, I, Is, dtype, mx=False):
    """Views of the intermediates moe_forward (moe_forward_mx with mx=True) leaves in its
    workspace (for tests and tools);
    the offsets follow the library's layout rule: 256-byte status word, then (decode batches
    only) the one-kernel layer's counters, counts, offsets,
    dispatch scratch, sorted_to_slot, slot_to_sorted, x_sorted, h, y_sorted, shared h, shared y,
    each rounded up to 256 bytes."""
    R = T * k
    b = 2 if dtype == torch.bfloat16 else 4
    nchunks = (R + 255) // 256
    # decode batches run the one-kernel layer, whose counters follow the status word
    fused = dtype == torch.bfloat16 and Is == 0 and 1 <= T <= 16 and R <= 256
    nbd = (d + 63) // 64
    fcnt = (2 * R * ((I + 63) // 64) + nbd + (nbd + 3) // 4) * 4 if fused else 0
    sizes = [("fused_counters", fcnt), ("counts", E * 4), ("offsets", (E + 1) * 4), ("chunk", nchunks * E * 4),
             ("sorted_to_slot", R * 4), ("slot_to_sorted", R * 4), ("x_sorted", R * d * b),
             ("h", R * I * b), ("y_sorted", R * d * 4), ("h_shared", T * Is * b),
             ("y_shared", T * d * 4 if Is else 0)]
    views, o = {}, 256
    for name, nbytes in sizes:
        views[name] = ws[o:o + nbytes]
        o = (o + nbytes + 255) // 256 * 256
    v = views
    if mx and fused:
        # the one-kernel layer on MX weights: its partial sums, then h's MXFP8 codes and scales
        nbh = (I + 63) // 64
        part_b = ((512 + R * nbh) * T * 128 * 4 + 255) // 256 * 256
        part = part_b + ((512 + nbd) * T * 64 * 4 + 255) // 256 * 256
        if nbh < 512 and nbd * T <= 1024:  # the owner layout's down partials [nbh][R][d]
            part += (nbh * R * d * 4 + 255) // 256 * 256
        o = (o + part + 255) // 256 * 256
        views["h_codes"] = ws[o:o + R * I]
        o = (o + R * I + 255) // 256 * 256
        views["h_scales"] = ws[o:o + R * ((I + 31) // 32)]
    out = {
        "counts": v["counts"].view(torch.int32),
        "offsets": v["offsets"].view(torch.int32),
        "sorted_to_slot": v["sorted_to_slot"].view(torch.int32),
        "slot_to_sorted": v["slot_to_sorted"].view(torch.int32),
        "x_sorted": v["x_sorted"].view(dtype).view(R, d),
        "h": v["h"].view(dtype).view(R, I),
        "y_sorted": v["y_sorted"].view(torch.float32).view(R, d),
    }
    if Is:
        out["h_shared"] = v["h_shared"].view(dtype).view(T, Is)
        out["y_shared"] = v["y_shared"].view(torch.float32).view(T, d)
    if "h_codes" in v:
        out["h_codes"] = v["h_codes"].view(R, I)
        out["h_scales"] = v["h_scales"].view(R, (I + 31) // 32)
    return out


# ------------------------------------------------------------------------------------------------
# training: the forward that keeps what the backward reads, and the backward pass
# ------------------------------------------------------------------------------------------------
def _code(dtype):
    return BF16 if dtype == torch.bfloat16 else F32


def moe_gate_up_train(x_rows, offsets, w_gate_up, sorted_to_slot=None, topk_weights=None,
                      scale_input=False, h=None, ab=None, workspace=None, stream=None):
    """moe_gate_up that also returns ab = [x W_gate | x W_up] (unscaled, layer dtype)."""
    _need(x_rows, "x_rows")
    R, d = x_rows.shape
    E, _, I, pk = _w_dims(w_gate_up, W_GATE_UP)
    dev = x_rows.device
    h = h if h is not None else torch.empty(R, I, dtype=x_rows.dtype, device=dev)
    ab = ab if ab is not None else torch.empty(R, 2 * I, dtype=x_rows.dtype, device=dev)
    ws = workspace if workspace is not None else _workspace(moe_experts_workspace_size(), dev)
    _check("moe_gate_up_train", lib().moe_gate_up_train(
        _p(x_rows), _p(offsets), _p(sorted_to_slot), _p(topk_weights), _dt(x_rows), R, d, E, I,
        _p(w_gate_up), (SCALE_INPUT if scale_input else 0) | pk, _p(h), _p(ab), _p(ws),
        ws.numel(), _stream(stream)))
    return h, ab


def moe_combine_backward(dout, slot_to_sorted, k, topk_weights=None, y_sorted=None,
                         want_weight_grad=True, dy_sorted=None, d_topk_weights=None,
                         stream=None):
    """Returns (dy_sorted [R, d] in dout's dtype, d_topk_weights [T, k] fp32 or None)."""
    _need(dout, "dout")
    T, d = dout.shape
    R = slot_to_sorted.numel()
    dev = dout.device
    dy = dy_sorted if dy_sorted is not None else torch.empty(R, d, dtype=dout.dtype, device=dev)
    dw = None
    if want_weight_grad:
        dw = d_topk_weights if d_topk_weights is not None else torch.empty(
            T, k, dtype=torch.float32, device=dev)
    _check("moe_combine_backward", lib().moe_combine_backward(
        _p(dout), _p(y_sorted if want_weight_grad else None), _p(slot_to_sorted),
        _p(topk_weights), _dt(dout), T, d, k, _p(dy), _p(dw), _stream(stream)))
    return dy, dw


def moe_down_backward(dy_sorted, ab, offsets, w_down, sorted_to_slot=None, topk_weights=None,
                      scale_input=False, d_ab=None, d_topk_weights=None, workspace=None,
                      stream=None):
    """Returns (d_ab [R, 2I], d_topk_weights by slot [R] fp32 or None)."""
    _need(dy_sorted, "dy_sorted")
    R, d = dy_sorted.shape
    E, I, _, pk = _w_dims(w_down, W_DOWN)
    dev = dy_sorted.device
    d_ab = d_ab if d_ab is not None else torch.empty(R, 2 * I, dtype=dy_sorted.dtype, device=dev)
    dw = None
    if scale_input:
        dw = d_topk_weights if d_topk_weights is not None else torch.empty(
            R, dtype=torch.float32, device=dev)
    ws = workspace if workspace is not None else _workspace(
        lib().moe_down_backward_workspace_size(R, I, _dt(dy_sorted)), dev)
    _check("moe_down_backward", lib().moe_down_backward(
        _p(dy_sorted), _p(ab), _p(offsets), _p(sorted_to_slot), _p(topk_weights), _dt(dy_sorted),
        R, d, E, I, _p(w_down), (SCALE_INPUT if scale_input else 0) | pk, _p(d_ab), _p(dw),
        _p(ws), ws.numel(), _stream(stream)))
    return d_ab, dw


def moe_gate_up_backward(d_ab, offsets, w_gate_up, dx_sorted=None, workspace=None, stream=None):
    """Returns dx_sorted [R, d] fp32."""
    _need(d_ab, "d_ab")
    R = d_ab.shape[0]
    E, d, I, pk = _w_dims(w_gate_up, W_GATE_UP)
    dev = d_ab.device
    dx = dx_sorted if dx_sorted is not None else torch.empty(R, d, dtype=torch.float32, device=dev)
    ws = workspace if workspace is not None else _workspace(moe_experts_workspace_size(), dev)
    _check("moe_gate_up_backward", lib().moe_gate_up_backward(
        _p(d_ab), _p(offsets), _dt(d_ab), R, d, E, I, _p(w_gate_up), pk, _p(dx), _p(ws),
        ws.numel(), _stream(stream)))
    return dx


def moe_weight_grad(a, b, offsets, E, dw=None, workspace=None, stream=None,
                    out_dtype=torch.float32):
    """dw[e] = a[rows of e]^T b[rows of e]: [E, M, N] fp32, or bf16 (bf16 a, b) with
    out_dtype=torch.bfloat16 (moe_weight_grad_bf16)."""
    _need(a, "a")
    _need(b, "b")
    R, M = a.shape
    N = b.shape[1]
    dev = a.device
    dw = dw if dw is not None else torch.empty(E, M, N, dtype=out_dtype, device=dev)
    ws = workspace if workspace is not None else _workspace(moe_experts_workspace_size(), dev)
    if dw.dtype == torch.bfloat16:
        _check("moe_weight_grad_bf16", lib().moe_weight_grad_bf16(
            _p(a), _p(b), _p(offsets), R, M, N, E, _p(dw), _p(ws), ws.numel(), _stream(stream)))
    else:
        _check("moe_weight_grad", lib().moe_weight_grad(
            _p(a), _p(b), _p(offsets), _dt(a), R, M, N, E, _p(dw), _p(ws), ws.numel(),
            _stream(stream)))
    return dw


def moe_route_backward(logits, topk_ids, topk_weights, d_topk_weights, score_fn=SOFTMAX,
                       renormalize=True, d_logits=None, stream=None):
    _need(logits, "logits")
    T, E = logits.shape
    k = topk_ids.shape[1]
    dl = d_logits if d_logits is not None else torch.empty(T, E, dtype=torch.float32,
                                                           device=logits.device)
    _check("moe_route_backward", lib().moe_route_backward(
        _p(logits), _p(topk_ids), _p(topk_weights), _p(d_topk_weights), T, E, k, score_fn,
        RENORMALIZE if renormalize else 0, _p(dl), _stream(stream)))
    return dl


def moe_forward_train_workspace_size(T, d, E, k, I, Is, dtype) -> int:
    return lib().moe_forward_train_workspace_size(T, d, E, k, I, Is, _code(dtype))


def moe_forward_train(x, logits, w_gate_up, w_down, k, score_fn=SOFTMAX, flags=RENORMALIZE,
                      w_shared_gate_up=None, w_shared_down=None, out=None, topk_ids=None,
                      topk_weights=None, workspace=None, stream=None):
    """moe_forward for training. Returns (out, topk_ids, topk_weights, workspace); the
    workspace holds what moe_backward reads."""
    _need(x, "x")
    _need(logits, "logits")
    T, d = x.shape
    E, _, I, pk = _w_dims(w_gate_up, W_GATE_UP)
    flags |= pk
    Is = _shared_width(w_shared_gate_up)
    dev = x.device
    out = out if out is not None else torch.empty(T, d, dtype=x.dtype, device=dev)
    ids = topk_ids if topk_ids is not None else torch.empty(T, k, dtype=torch.int32, device=dev)
    w = topk_weights if topk_weights is not None else torch.empty(T, k, dtype=torch.float32,
                                                                  device=dev)
    ws = workspace if workspace is not None else _workspace(
        moe_forward_train_workspace_size(T, d, E, k, I, Is, x.dtype), dev)
    _check("moe_forward_train", lib().moe_forward_train(
        _p(x), _p(logits), _dt(x), T, d, E, k, I, score_fn, flags, _p(w_gate_up), _p(w_down),
        _p(w_shared_gate_up), _p(w_shared_down), Is, _p(ids), _p(w), _p(out), _p(ws), ws.numel(),
        _stream(stream)))
    return out, ids, w, ws


def _shared_width(w_shared_gate_up):
    if w_shared_gate_up is None:
        return 0
    return (w_shared_gate_up.N if isinstance(w_shared_gate_up, PackedWeights)
            else w_shared_gate_up.shape[-1] // 2)


def moe_backward_workspace_size(T, d, E, k, I, Is, dtype) -> int:
    return lib().moe_backward_workspace_size(T, d, E, k, I, Is, _code(dtype))


def moe_backward_kernel_count(T, k, Is, flags, want_logits=True) -> int:
    return lib().moe_backward_kernel_count(T, k, Is, flags, 1 if want_logits else 0)


def moe_backward(dout, x, logits, w_gate_up, w_down, k, topk_ids, topk_weights, fwd_workspace,
                 score_fn=SOFTMAX, flags=RENORMALIZE, w_shared_gate_up=None, w_shared_down=None,
                 want_logits=True, out=None, workspace=None, stream=None):
    """The whole backward pass for a moe_forward_train call with the same arguments.
    Returns a dict: dx, d_w_gate_up, d_w_down, d_topk_weights, d_logits (None unless
    want_logits) and, with a shared expert, d_w_shared_gate_up, d_w_shared_down. `out` may
    pass preallocated tensors under those names. flags may include WGRAD_BF16: the weight
    gradients are then bf16."""
    _need(dout, "dout")
    T, d = dout.shape
    E, _, I, pk = _w_dims(w_gate_up, W_GATE_UP)
    flags |= pk
    Is = _shared_width(w_shared_gate_up)
    dev = dout.device
    o = dict(out or {})
    f32 = torch.float32

    def get(name, shape, dtype):
        if o.get(name) is None:
            o[name] = torch.empty(*shape, dtype=dtype, device=dev)
        return o[name]

    wdt = torch.bfloat16 if flags & WGRAD_BF16 else f32
    dx = get("dx", (T, d), dout.dtype)
    dwgu = get("d_w_gate_up", (E, d, 2 * I), wdt)
    dwd = get("d_w_down", (E, I, d), wdt)
    dtw = get("d_topk_weights", (T, k), f32)
    dl = get("d_logits", (T, E), f32) if want_logits else None
    o.setdefault("d_logits", dl)
    dsgu = get("d_w_shared_gate_up", (d, 2 * Is), wdt) if Is else None
    dsd = get("d_w_shared_down", (Is, d), wdt) if Is else None
    ws = workspace if workspace is not None else _workspace(
        moe_backward_workspace_size(T, d, E, k, I, Is, dout.dtype), dev)
    _check("moe_backward", lib().moe_backward(
        _p(dout), _p(x), _p(logits), _dt(dout), T, d, E, k, I, score_fn, flags, _p(w_gate_up),
        _p(w_down), _p(w_shared_gate_up), _p(w_shared_down), Is, _p(topk_ids), _p(topk_weights),
        _p(fwd_workspace), fwd_workspace.numel(), _p(dx), _p(dwgu), _p(dwd), _p(dsgu), _p(dsd),
        _p(dtw), _p(dl), _p(ws), ws.numel(), _stream(stream)))
    o["workspace"] = ws
    return o


def backward_workspace_views(ws: torch.Tensor, T, d, k, I, dtype):
    """Views of the intermediates moe_backward leaves in its workspace (for tests): dy_sorted
    [R, d], d_ab [R, 2I] (layer dtype) and dx_sorted [R, d] fp32, after the 256-byte status word,
    each rounded up to 256 bytes."""
    R = T * k
    b = 2 if dtype == torch.bfloat16 else 4
    views, o = {}, 256
    for name, nbytes in [("dy_sorted", R * d * b), ("d_ab", R * 2 * I * b),
                         ("dx_sorted", R * d * 4)]:
        views[name] = ws[o:o + nbytes]
        o = (o + nbytes + 255) // 256 * 256
    return {"dy_sorted": views["dy_sorted"].view(dtype).view(R, d),
            "d_ab": views["d_ab"].view(dtype).view(R, 2 * I),
            "dx_sorted": views["dx_sorted"].view(torch.float32).view(R, d)}


def forward_train_workspace_views(ws: torch.Tensor, T, d, E, k, I, Is, dtype):
    """forward_workspace_views for moe_forward_train's workspace, plus "ab" [R, 2I] and (shared
    expert) "ab_shared" [T, 2Is]."""
    R = T * k
    b = 2 if dtype == torch.bfloat16 else 4
    nchunks = (R + 255) // 256
    sizes = [("counts", E * 4), ("offsets", (E + 1) * 4), ("chunk", nchunks * E * 4),
             ("sorted_to_slot", R * 4), ("slot_to_sorted", R * 4), ("x_sorted", R * d * b),
             ("h", R * I * b), ("y_sorted", R * d * 4), ("h_shared", T * Is * b),
             ("y_shared", T * d * 4 if Is else 0), ("fused", 0), ("ab", R * 2 * I * b),
             ("ab_shared", T * 2 * Is * b)]
    views, o = {}, 256
    for name, nbytes in sizes:
        views[name] = ws[o:o + nbytes]
        o = (o + nbytes + 255) // 256 * 256
    v = views
    out = {
        "counts": v["counts"].view(torch.int32),
        "offsets": v["offsets"].view(torch.int32),
        "sorted_to_slot": v["sorted_to_slot"].view(torch.int32),
        "slot_to_sorted": v["slot_to_sorted"].view(torch.int32),
        "x_sorted": v["x_sorted"].view(dtype).view(R, d),
        "h": v["h"].view(dtype).view(R, I),
        "y_sorted": v["y_sorted"].view(torch.float32).view(R, d),
        "ab": v["ab"].view(dtype).view(R, 2 * I),
    }
    if Is:
        out["h_shared"] = v["h_shared"].view(dtype).view(T, Is)
        out["y_shared"] = v["y_shared"].view(torch.float32).view(T, d)
        out["ab_shared"] = v["ab_shared"].view(dtype).view(T, 2 * Is)
    return out


# ------------------------------------------------------------------------------------------------
# MX formats: MXFP4 expert weights, MXFP8 activations
# ------------------------------------------------------------------------------------------------
class MxWeights:
    """Expert weights in the MX buffer layout (moe_quantize_weights_mx): `data` holds the E2M1
    codes then the E8M0 scales; kind W_GATE_UP (logical [E, K=d, 2I], N = I) or W_DOWN
    ([E, K=I, N=d])."""

    def __init__(self, data: torch.Tensor, kind: int, E: int, K: int, N: int, tc=False):
        self.data, self.kind, self.E, self.K, self.N = data, kind, E, K, N
        self.tc = tc  # True: the MX tensor-core layout (moe_quantize_weights_mx_tc)

    def data_ptr(self):
        return self.data.data_ptr()


def quantize_weights_mx(w: torch.Tensor, kind: int, stream=None) -> MxWeights:
    """bf16 gate_up ([E, d, 2I] or [d, 2I]) or down ([E, I, d] or [I, d]) weights to MXFP4."""
    _need(w, "w")
    w3 = w.unsqueeze(0) if w.dim() == 2 else w
    E, K, C = w3.shape
    N = C // 2 if kind == W_GATE_UP else C
    out = torch.empty(lib().moe_mx_weights_size(kind, E, K, N), dtype=torch.uint8,
                      device=w.device)
    _check("moe_quantize_weights_mx", lib().moe_quantize_weights_mx(
        kind, _p(w3), _p(out), E, K, N, _stream(stream)))
    return MxWeights(out, kind, E, K, N)


def dequantize_weights_mx(mx: MxWeights, stream=None) -> torch.Tensor:
    cols = 2 * mx.N if mx.kind == W_GATE_UP else mx.N
    w = torch.empty(mx.E, mx.K, cols, dtype=torch.bfloat16, device=mx.data.device)
    _check("moe_dequantize_weights_mx", lib().moe_dequantize_weights_mx(
        mx.kind, _p(mx.data), _p(w), mx.E, mx.K, mx.N, _stream(stream)))
    return w


def quantize_weights_mx_tc(w: torch.Tensor, kind: int, stream=None) -> MxWeights:
    """bf16 gate_up ([E, d, 2I] or [d, 2I]) or down ([E, I, d] or [I, d]) weights to MXFP4 in
    the MX tensor-core layout (the block-scaled GEMMs of moe_forward_mx_tc read it)."""
    _need(w, "w")
    w3 = w.unsqueeze(0) if w.dim() == 2 else w
    E, K, C = w3.shape
    N = C // 2 if kind == W_GATE_UP else C
    n = lib().moe_mx_tc_weights_size(kind, E, K, N)
    if n == 0:
        raise MoEError("moe_mx_tc_weights_size", 1)
    out = torch.empty(n, dtype=torch.uint8, device=w.device)
    _check("moe_quantize_weights_mx_tc", lib().moe_quantize_weights_mx_tc(
        kind, _p(w3), _p(out), E, K, N, _stream(stream)))
    return MxWeights(out, kind, E, K, N, tc=True)


def dequantize_weights_mx_tc(mx: MxWeights, stream=None) -> torch.Tensor:
    cols = 2 * mx.N if mx.kind == W_GATE_UP else mx.N
    w = torch.empty(mx.E, mx.K, cols, dtype=torch.bfloat16, device=mx.data.device)
    _check("moe_dequantize_weights_mx_tc", lib().moe_dequantize_weights_mx_tc(
        mx.kind, _p(mx.data), _p(w), mx.E, mx.K, mx.N, _stream(stream)))
    return w


def quantize_rows_mx(x: torch.Tensor, want_codes=True, stream=None):
    """bf16 rows [R, K] to MXFP8 along K: (rounded bf16 rows, codes uint8 [R, K] or None,
    scales uint8 [R, ceil(K/32)] or None)."""
    _need(x, "x")
    R, K = x.shape
    xo = torch.empty_like(x)
    codes = torch.empty(R, K, dtype=torch.uint8, device=x.device) if want_codes else None
    scales = (torch.empty(R, (K + 31) // 32, dtype=torch.uint8, device=x.device)
              if want_codes else None)
    _check("moe_quantize_rows_mx", lib().moe_quantize_rows_mx(
        _p(x), R, K, _p(xo), _p(codes), _p(scales), _stream(stream)))
    return xo, codes, scales


def moe_forward_mx_workspace_size(T, d, E, k, I, Is) -> int:
    return lib().moe_forward_mx_workspace_size(T, d, E, k, I, Is)


def moe_forward_mx(x, logits, w_gate_up: MxWeights, w_down: MxWeights, k, score_fn=SOFTMAX,
                   flags=RENORMALIZE, w_shared_gate_up=None, w_shared_down=None, out=None,
                   topk_ids=None, topk_weights=None, workspace=None, stream=None):
    """The MX layer. Returns (out, topk_ids, topk_weights, workspace)."""
    _need(x, "x")
    _need(logits, "logits")
    T, d = x.shape
    E, I = w_gate_up.E, w_gate_up.N
    Is = w_shared_gate_up.N if w_shared_gate_up is not None else 0
    dev = x.device
    out = out if out is not None else torch.empty(T, d, dtype=x.dtype, device=dev)
    ids = topk_ids if topk_ids is not None else torch.empty(T, k, dtype=torch.int32, device=dev)
    w = topk_weights if topk_weights is not None else torch.empty(T, k, dtype=torch.float32,
                                                                  device=dev)
    ws = workspace if workspace is not None else _workspace(
        moe_forward_mx_workspace_size(T, d, E, k, I, Is), dev)
    _check("moe_forward_mx", lib().moe_forward_mx(
        _p(x), _p(logits), T, d, E, k, I, score_fn, flags, _p(w_gate_up), _p(w_down),
        _p(w_shared_gate_up), _p(w_shared_down), Is, _p(ids), _p(w), _p(out), _p(ws), ws.numel(),
        _stream(stream)))
    return out, ids, w, ws


def moe_forward_mx_tc_workspace_size(T, d, E, k, I, Is) -> int:
    return lib().moe_forward_mx_tc_workspace_size(T, d, E, k, I, Is)


def moe_forward_mx_tc_kernel_count(T, d, k, I, Is=0) -> int:
    """Kernels moe_forward_mx_tc launches for these sizes (1: the one-kernel decode layer)."""
    return lib().moe_forward_mx_tc_kernel_count(T, d, k, I, Is)


def moe_forward_mx_tc(x, logits, w_gate_up: MxWeights, w_down: MxWeights, k, score_fn=SOFTMAX,
                      flags=RENORMALIZE, w_shared_gate_up=None, w_shared_down=None, out=None,
                      topk_ids=None, topk_weights=None, workspace=None, stream=None):
    """The MX layer on the block-scaled tensor cores (weights from quantize_weights_mx_tc).
    Returns (out, topk_ids, topk_weights, workspace)."""
    _need(x, "x")
    _need(logits, "logits")
    T, d = x.shape
    E, I = w_gate_up.E, w_gate_up.N
    Is = w_shared_gate_up.N if w_shared_gate_up is not None else 0
    dev = x.device
    out = out if out is not None else torch.empty(T, d, dtype=x.dtype, device=dev)
    ids = topk_ids if topk_ids is not None else torch.empty(T, k, dtype=torch.int32, device=dev)
    w = topk_weights if topk_weights is not None else torch.empty(T, k, dtype=torch.float32,
                                                                  device=dev)
    ws = workspace if workspace is not None else _workspace(
        moe_forward_mx_tc_workspace_size(T, d, E, k, I, Is), dev)
    _check("moe_forward_mx_tc", lib().moe_forward_mx_tc(
        _p(x), _p(logits), T, d, E, k, I, score_fn, flags, _p(w_gate_up), _p(w_down),
        _p(w_shared_gate_up), _p(w_shared_down), Is, _p(ids), _p(w), _p(out), _p(ws), ws.numel(),
        _stream(stream)))
    return out, ids, w, ws


def mx_tc_workspace_views(ws: torch.Tensor, T, d, E, k, I, Is):
    """Views of what moe_forward_mx_tc leaves in its workspace (layout of include/moe.h):
    indices, the padded MXFP8 rows of x and h (codes [Rp, K] uint8, scale atoms
    [Rp / 128, ceil(K / 128), 512] uint8), y_sorted and the shared expert's."""
    R = T * k
    Rp = (R + 127) // 128 * 128 + 128 * E
    Tp = (T + 127) // 128 * 128
    kc = lambda K: (K + 127) // 128
    sizes = [("counts", E * 4), ("offsets", (E + 1) * 4), ("chunk", (R + 255) // 256 * E * 4),
             ("sorted_to_slot", R * 4), ("slot_to_sorted", R * 4), ("x_codes", Rp * d),
             ("x_sf", Rp // 128 * kc(d) * 512), ("h_codes", Rp * I),
             ("h_sf", Rp // 128 * kc(I) * 512), ("y_sorted", R * d * 4),
             ("sx_codes", Tp * d if Is else 0), ("sx_sf", Tp // 128 * kc(d) * 512 if Is else 0),
             ("sh_codes", Tp * Is if Is else 0), ("sh_sf", Tp // 128 * kc(Is) * 512 if Is else 0),
             ("y_shared", T * d * 4 if Is else 0)]
    v, o = {}, 256
    for name, nbytes in sizes:
        v[name] = ws[o:o + nbytes]
        o = (o + nbytes + 255) // 256 * 256
    out = {"counts": v["counts"].view(torch.int32), "offsets": v["offsets"].view(torch.int32),
           "sorted_to_slot": v["sorted_to_slot"].view(torch.int32),
           "slot_to_sorted": v["slot_to_sorted"].view(torch.int32),
           "x_codes": v["x_codes"].view(Rp, d), "x_sf": v["x_sf"].view(Rp // 128, kc(d), 512),
           "h_codes": v["h_codes"].view(Rp, I), "h_sf": v["h_sf"].view(Rp // 128, kc(I), 512),
           "y_sorted": v["y_sorted"].view(torch.float32).view(R, d), "Rp": Rp, "Tp": Tp}
    if Is:
        out.update({"sx_codes": v["sx_codes"].view(Tp, d),
                    "sx_sf": v["sx_sf"].view(Tp // 128, kc(d), 512),
                    "sh_codes": v["sh_codes"].view(Tp, Is),
                    "sh_sf": v["sh_sf"].view(Tp // 128, kc(Is), 512),
                    "y_shared": v["y_shared"].view(torch.float32).view(T, d)})
    return out


def mx_tc_rows(x, topk_ids, slot_to_sorted, offsets, E, codes, sf, codes_sh=None, sf_sh=None,
               stream=None):
    """x [T, d] bf16 to MXFP8 in the padded tensor-core layout (see moe_mx_tc_rows)."""
    T, d = x.shape
    k = topk_ids.shape[1] if topk_ids is not None else 1
    _check("moe_mx_tc_rows", lib().moe_mx_tc_rows(
        _p(x), T, d, k, E, _p(topk_ids), _p(slot_to_sorted), _p(offsets), _p(codes), _p(sf),
        _p(codes_sh), _p(sf_sh), _stream(stream)))


def moe_gate_up_mx_tc(x_codes, x_sf, offsets, w_gate_up: MxWeights, R, h_codes, h_sf,
                      sorted_to_slot=None, topk_weights=None, scale_input=False,
                      workspace=None, stream=None):
    d, E, I = w_gate_up.K, w_gate_up.E, w_gate_up.N
    ws = workspace if workspace is not None else _workspace(256, x_codes.device)
    _check("moe_gate_up_mx_tc", lib().moe_gate_up_mx_tc(
        _p(x_codes), _p(x_sf), _p(offsets), _p(sorted_to_slot), _p(topk_weights), R, d, E, I,
        _p(w_gate_up), SCALE_INPUT if scale_input else 0, _p(h_codes), _p(h_sf), _p(ws),
        ws.numel(), _stream(stream)))
    return ws


def moe_down_mx_tc(h_codes, h_sf, offsets, w_down: MxWeights, R, y_sorted, workspace=None,
                   stream=None):
    I, E, d = w_down.K, w_down.E, w_down.N
    ws = workspace if workspace is not None else _workspace(256, h_codes.device)
    _check("moe_down_mx_tc", lib().moe_down_mx_tc(
        _p(h_codes), _p(h_sf), _p(offsets), R, I, E, d, _p(w_down), _p(y_sorted), _p(ws),
        ws.numel(), _stream(stream)))
    return ws
