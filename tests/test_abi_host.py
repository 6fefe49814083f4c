"""The C ABI on a machine without a GPU: the library loads, exports every entry point the header
declares, and rejects bad arguments before enqueueing anything (no CUDA call is reached)."""
import ctypes
import os
import re

import pytest

from routing_dispatch_grouped_gb300 import moe

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")


@pytest.fixture(scope="module")
def L():
    if not os.path.exists(moe.LIB_PATH):
        from routing_dispatch_grouped_gb300 import build
        build.build()
    return moe.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_five_steps():
    names = declared_functions()
    for n in ("moe_route", "moe_dispatch", "moe_experts", "moe_combine", "moe_forward"):
        assert n in names


def test_every_declared_symbol_is_exported(L):
    names = declared_functions()
    assert names, "no declarations parsed"
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(moe.SIGNATURES), "binding and header disagree"


FAKE = 0x10000  # 16-byte aligned, never dereferenced: every call below fails validation first
MIS = 0x10004   # misaligned
NULL = None


def test_route_validation(L):
    r = L.moe_route
    assert r(FAKE, 4, 8, 9, 0, 1, FAKE, FAKE, NULL) == 1          # k > E
    assert r(FAKE, 4, 300, 2, 0, 1, FAKE, FAKE, NULL) == 2        # E > 256
    assert r(FAKE, 4, 8, 0, 0, 1, FAKE, FAKE, NULL) == 1          # k = 0
    assert r(FAKE, -1, 8, 2, 0, 1, FAKE, FAKE, NULL) == 1         # T < 0
    assert r(FAKE, 4, 8, 2, 7, 1, FAKE, FAKE, NULL) == 1          # bad score fn
    assert r(FAKE, 4, 8, 2, 0, 8, FAKE, FAKE, NULL) == 1          # unknown flag
    assert r(NULL, 4, 8, 2, 0, 1, FAKE, FAKE, NULL) == 1          # null logits
    assert r(MIS, 4, 8, 2, 0, 1, FAKE, FAKE, NULL) == 1           # misaligned
    assert r(NULL, 0, 8, 2, 0, 1, NULL, NULL, NULL) == 0          # T = 0: no-op
    assert r(FAKE, 1 << 28, 8, 8, 0, 1, FAKE, FAKE, NULL) == 2    # T*k >= 2^31


def test_route_hidden_validation(L):
    r = L.moe_route_hidden
    # (x, dt, w_router, bias, T, d, E, k, fn, flags, logits, ids, weights, stream)
    assert r(FAKE, 1, FAKE, NULL, 4, 64, 8, 9, 0, 1, NULL, FAKE, FAKE, NULL) == 1   # k > E
    assert r(FAKE, 1, FAKE, NULL, 4, 64, 300, 2, 0, 1, NULL, FAKE, FAKE, NULL) == 2  # E > 256
    assert r(FAKE, 1, FAKE, NULL, 4, 0, 8, 2, 0, 1, NULL, FAKE, FAKE, NULL) == 1    # d = 0
    assert r(FAKE, 5, FAKE, NULL, 4, 64, 8, 2, 0, 1, NULL, FAKE, FAKE, NULL) == 1   # bad dtype
    assert r(FAKE, 1, FAKE, NULL, 4, 64, 8, 2, 7, 1, NULL, FAKE, FAKE, NULL) == 1   # bad fn
    assert r(FAKE, 1, FAKE, NULL, 4, 64, 8, 2, 0, 2, NULL, FAKE, FAKE, NULL) == 1   # bad flag
    assert r(FAKE, 1, NULL, NULL, 4, 64, 8, 2, 0, 1, NULL, FAKE, FAKE, NULL) == 1   # no weight
    assert r(FAKE, 1, FAKE, MIS, 4, 64, 8, 2, 0, 1, NULL, FAKE, FAKE, NULL) == 1    # misaligned
    assert r(NULL, 1, NULL, NULL, 0, 64, 8, 2, 0, 1, NULL, NULL, NULL, NULL) == 0   # T = 0


def test_dispatch_validation(L):
    d = L.moe_dispatch
    ws_need = L.moe_dispatch_workspace_size(100, 8, 2)
    assert ws_need >= 256 and ws_need % 256 == 0
    ok = dict(ids=FAKE, x=FAKE, dt=1, T=100, d=64, E=8, k=2)

    def call(**kw):
        a = {**ok, **kw}
        return d(a["ids"], a["x"], a["dt"], a["T"], a["d"], a["E"], a["k"], FAKE, FAKE, FAKE,
                 FAKE, FAKE if a["x"] else None, a.get("ws", 0x100000), a.get("wsb", ws_need),
                 NULL)
    assert call(d=60) == 1                    # bf16 rows must be a multiple of 8 elements
    assert call(dt=5) == 1
    assert call(wsb=ws_need - 1) == 3         # short workspace
    assert call(ws=0x100010) == 3             # workspace not 256-byte aligned
    assert call(k=9) == 1
    assert d(FAKE, FAKE, 1, 100, 64, 8, 2, FAKE, FAKE, FAKE, FAKE, None, 0x100000, ws_need,
             NULL) == 1                       # x without x_sorted


def test_experts_validation(L):
    g = L.moe_gate_up
    ws = 0x100000
    # offsets NULL needs E == 1
    assert g(FAKE, None, None, None, 1, 128, 64, 4, 64, FAKE, 0, FAKE, ws, 256, NULL) == 1
    # scale needs sorted_to_slot and weights
    assert g(FAKE, FAKE, None, None, 1, 128, 64, 4, 64, FAKE, 2, FAKE, ws, 256, NULL) == 1
    # bad flag for gate_up
    assert g(FAKE, FAKE, FAKE, FAKE, 1, 128, 64, 4, 64, FAKE, 4, FAKE, ws, 256, NULL) == 1
    # I not a multiple of 8
    assert g(FAKE, FAKE, None, None, 1, 128, 64, 4, 60, FAKE, 0, FAKE, ws, 256, NULL) == 1
    # workspace too small
    assert g(FAKE, FAKE, None, None, 1, 128, 64, 4, 64, FAKE, 0, FAKE, ws, 16, NULL) == 3
    # R == 0 is a no-op
    assert g(FAKE, FAKE, None, None, 1, 0, 64, 4, 64, FAKE, 0, FAKE, ws, 256, NULL) == 0
    e = L.moe_experts
    assert e(FAKE, FAKE, FAKE, FAKE, 1, 128, 64, 4, 64, FAKE, FAKE, 6, FAKE, FAKE, ws, 256,
             NULL) == 1                         # scale + fused weight exclude each other
    assert L.moe_experts_workspace_size() == 256


def test_combine_and_forward_validation(L):
    c = L.moe_combine
    assert c(FAKE, FAKE, None, None, 10, 64, 33, 1, FAKE, NULL) == 2   # k > 32
    assert c(FAKE, FAKE, None, None, 10, 60, 2, 1, FAKE, NULL) == 1    # bf16 d % 8
    assert c(MIS, FAKE, None, None, 10, 64, 2, 1, FAKE, NULL) == 1
    assert c(None, None, None, None, 0, 64, 2, 1, None, NULL) == 0
    f = L.moe_forward
    sz = L.moe_forward_workspace_size(64, 128, 8, 2, 256, 0, 1)
    args = [FAKE, FAKE, 1, 64, 128, 8, 2, 256, 0, 1, FAKE, FAKE, None, None, 0, FAKE, FAKE, FAKE,
            0x100000, sz, NULL]
    bad = list(args); bad[9] = 1 | 2 | 4
    assert f(*bad) == 1                                            # scale + fuse
    bad = list(args); bad[12] = FAKE
    assert f(*bad) == 1                                            # shared weights without Is
    bad = list(args); bad[19] = sz - 256
    assert f(*bad) == 3
    bad = list(args); bad[3] = 0
    assert f(*bad) == 0


def test_workspace_size_matches_binding_layout(L):
    import torch
    for (T, d, E, k, I, Is, dt) in [(256, 128, 8, 2, 256, 0, torch.float32),
                                    (4096, 4096, 8, 2, 14336, 0, torch.bfloat16),
                                    (16384, 5120, 16, 1, 8192, 8192, torch.bfloat16),
                                    (1, 2048, 128, 8, 768, 0, torch.bfloat16)]:
        sz = moe.moe_forward_workspace_size(T, d, E, k, I, Is, dt)
        ws = torch.empty(sz, dtype=torch.uint8)
        v = moe.forward_workspace_views(ws, T, d, E, k, I, Is, dt)
        assert v["y_sorted"].numel() == T * k * d
        last = v["y_shared"] if Is else v["y_sorted"]
        end = last.untyped_storage().data_ptr()
        assert sz >= (last.data_ptr() - ws.data_ptr()) + last.numel() * last.element_size()


def test_pack_validation_and_sizes(L):
    P = L.moe_pack_weights
    assert P(0, FAKE, FAKE, 0, 2, 64, 64, NULL) == 2     # fp32 packing is not supported
    assert P(7, FAKE, FAKE, 1, 2, 64, 64, NULL) == 1     # unknown kind
    assert P(0, FAKE, FAKE, 1, 2, 64, 60, NULL) == 1     # N not a multiple of 8
    assert P(1, MIS, FAKE, 1, 2, 64, 64, NULL) == 1      # misaligned
    S = L.moe_packed_weights_size
    # gate_up [E=8, d=4096, 2I=2*14336]: 2 * 224 blocks of 64 columns, Kpad 4096
    assert S(0, 8, 4096, 14336, 1) == 8 * 448 * 4096 * 64 * 2
    # down [E=128, I=2880, d=2880]: 45 blocks, Kpad 2880
    assert S(1, 128, 2880, 2880, 1) == 128 * 45 * 2880 * 128
    # padding: K=200 -> 256, N=200 -> 4 blocks per half
    assert S(0, 1, 200, 200, 1) == 8 * 256 * 128
    assert S(0, 1, 200, 200, 0) == 0
    f = L.moe_forward
    sz = L.moe_forward_workspace_size(64, 128, 8, 2, 256, 0, 0)
    assert f(FAKE, FAKE, 0, 64, 128, 8, 2, 256, 0, 1 | 8, FAKE, FAKE, None, None, 0, FAKE, FAKE,
             FAKE, 0x100000, sz, NULL) == 2           # packed weights need bf16


def test_kernel_count_and_strings(L):
    bf16, f32 = moe.BF16, moe.F32
    assert L.moe_forward_kernel_count(bf16, 0, 2, 0) == 0
    assert L.moe_forward_kernel_count(bf16, 10, 2, 0) == 1      # one-kernel decode layer
    assert L.moe_forward_kernel_count(bf16, 16, 16, 0) == 1
    assert L.moe_forward_kernel_count(bf16, 17, 2, 0) == 5      # fused small-batch front end
    assert L.moe_forward_kernel_count(bf16, 16, 17, 0) == 5     # T*k above the decode limit
    assert L.moe_forward_kernel_count(f32, 10, 2, 0) == 5       # fp32 layers: no decode kernel
    assert L.moe_forward_kernel_count(bf16, 10, 2, 128) == 7    # shared expert: no decode kernel
    assert L.moe_forward_kernel_count(bf16, 4096, 2, 0) == 8
    assert L.moe_forward_kernel_count(bf16, 16384, 1, 8192) == 10
    # the MX tensor-core layer: (T, d, k, I, Is)
    mc = L.moe_forward_mx_tc_kernel_count
    assert mc(0, 2048, 8, 768, 0) == 0
    assert mc(1, 2048, 8, 768, 0) == 1          # one-kernel decode layer
    assert mc(16, 2048, 16, 768, 0) == 1
    assert mc(17, 2048, 8, 768, 0) == 5         # route+dispatch, rows, gate_up, down, combine
    assert mc(16, 2048, 17, 768, 0) == 5        # T*k above the decode limit
    assert mc(8, 2176, 8, 768, 0) == 5          # d above the one-kernel layer's 2048
    assert mc(8, 2048, 8, 4128, 0) == 5         # I above its 4096
    assert mc(8, 2048, 8, 768, 256) == 7        # shared expert: no one-kernel layer
    assert mc(4096, 4096, 2, 14336, 0) == 8     # dispatch in 3 kernels above 1024 slots
    for code in range(7):
        assert L.moe_status_string(code).decode().startswith(moe.STATUS[code])


def test_mx_validation_and_sizes(L):
    # blocks of 64 columns x 32 rows: 1 KB of codes + 64 B of scales each. gate_up [E=2, K=64,
    # I=64]: 2 column blocks (gate, up) x 2 K blocks per expert; down [E=1, K=200, d=96]: 2 x 7
    assert L.moe_mx_weights_size(0, 2, 64, 64) == 2 * 2 * 2 * (1024 + 64)
    assert L.moe_mx_weights_size(1, 1, 200, 96) == 2 * 7 * (1024 + 64)
    assert L.moe_mx_weights_size(0, 1, 64, 60) == 0                     # N % 8
    q = L.moe_quantize_weights_mx
    assert q(7, FAKE, FAKE, 1, 64, 64, NULL) == 1                          # unknown kind
    assert q(0, FAKE, FAKE, 1, 60, 64, NULL) == 1                          # K % 8
    assert q(0, MIS, FAKE, 1, 64, 64, NULL) == 1                           # misaligned
    r = L.moe_quantize_rows_mx
    assert r(FAKE, 4, 60, FAKE, None, None, NULL) == 1                     # K % 8
    assert r(FAKE, 4, 64, FAKE, FAKE, None, NULL) == 1                     # codes without scales
    assert r(None, 0, 64, None, None, None, NULL) == 0                     # R = 0
    f = L.moe_forward_mx
    sz = L.moe_forward_mx_workspace_size(64, 128, 8, 2, 256, 0)
    assert sz > L.moe_forward_workspace_size(64, 128, 8, 2, 256, 0, 1)
    args = [FAKE, FAKE, 64, 128, 8, 2, 256, 0, 1, FAKE, FAKE, None, None, 0, FAKE, FAKE, FAKE,
            0x100000, sz, NULL]
    bad = list(args); bad[8] = 1 | 8
    assert f(*bad) == 1                                                    # packed: not MX
    bad = list(args); bad[18] = sz - 256
    assert f(*bad) == 3                                                    # short workspace
    bad = list(args); bad[2] = 0
    assert f(*bad) == 0                                                    # T = 0


def test_weight_grad_validation(L):
    w = L.moe_weight_grad_bf16
    ws = 0x100000
    assert w(FAKE, FAKE, FAKE, 10, 64, 60, 4, FAKE, ws, 256, NULL) == 1     # N % 8
    assert w(FAKE, FAKE, None, 10, 64, 64, 4, FAKE, ws, 256, NULL) == 1     # NULL offsets, E > 1
    assert w(FAKE, FAKE, FAKE, 10, 64, 64, 4, MIS, ws, 256, NULL) == 1      # misaligned dw
    assert w(FAKE, FAKE, FAKE, 10, 64, 64, 4, FAKE, ws, 16, NULL) == 3      # workspace
    assert w(FAKE, FAKE, FAKE, 10, 64, 64, 300, FAKE, ws, 256, NULL) == 2   # E > 256
    b = L.moe_backward
    args = [FAKE, FAKE, FAKE, 1, 64, 128, 8, 2, 256, 0, 1, FAKE, FAKE, None, None, 0, FAKE, FAKE,
            FAKE, 1 << 30, FAKE, FAKE, FAKE, None, None, FAKE, FAKE, 0x100000, 1 << 30, NULL]
    bad = list(args); bad[3] = 0; bad[10] = 1 | 16
    assert b(*bad) == 2                                      # bf16 weight gradients of fp32 layers
    bad = list(args); bad[10] = 1 | 32
    assert b(*bad) == 1                                      # unknown flag


def test_gemm_kernel_choice(L):
    name = moe.moe_gemm_kernel_name
    # routed gate_up above the small-batch size: 256-row CTA pairs (tails swapped)
    for R, E in ((8192, 8), (16384, 16), (32768, 128), (1024, 128)):
        assert name(moe.W_GATE_UP, R, E) == "tc_grouped_gemm_2sm"
    # routed down above the small-batch size: weights as the M side of CTA pairs
    for R, E in ((8192, 8), (32768, 128), (1024, 128)):
        assert name(moe.W_DOWN, R, E) == "tc_grouped_gemm_swap_pair"
    # one dense group (shared expert): 256-row CTA pairs for both
    assert name(moe.W_GATE_UP, 16384, 1, False) == "tc_grouped_gemm_2sm"
    assert name(moe.W_DOWN, 16384, 1, False) == "tc_grouped_gemm_2sm"
    # at most 512 routed rows (decode chain): swapped operands
    assert name(moe.W_GATE_UP, 512, 128) == "tc_grouped_gemm_swap"
    assert name(moe.W_DOWN, 8, 128) == "tc_grouped_gemm_swap"
    assert name(moe.W_DOWN, 0, 8) == "none" and name(7, 100, 8) == "none"
    # the small-batch boundary: at most 512 routed rows stay on the swapped-operand kernel
    assert name(moe.W_GATE_UP, 512, 8) == "tc_grouped_gemm_swap"
    assert name(moe.W_GATE_UP, 513, 8) == "tc_grouped_gemm_2sm"
    assert name(moe.W_DOWN, 512, 8) == "tc_grouped_gemm_swap"
    assert name(moe.W_DOWN, 513, 8) == "tc_grouped_gemm_swap_pair"


def test_forward_host_validation(L):
    f = L.moe_forward_host
    sz = L.moe_forward_host_workspace_size(64, 128, 8, 2, 256, 0, 1)
    assert sz > L.moe_forward_workspace_size(64, 128, 8, 2, 256, 0, 1)
    args = [FAKE, FAKE, 1, 64, 128, 8, 2, 256, 0, 1, FAKE, FAKE, None, None, 0, FAKE, 0x100000,
            sz, NULL]
    bad = list(args); bad[0] = None
    assert f(*bad) == 1                                            # no host x
    bad = list(args); bad[15] = None
    assert f(*bad) == 1                                            # no host out
    bad = list(args); bad[17] = sz - 256
    assert f(*bad) == 3                                            # short workspace
    bad = list(args); bad[3] = 0
    assert f(*bad) == 0                                            # T = 0: nothing enqueued
    bad = list(args); bad[6] = 9
    assert f(*bad) == 1                                            # k > E


def test_mx_tc_weights_size_follows_the_layout(L):
    """moe_mx_tc_weights_size: codes (K padded to 128, two per byte) then 512-byte scale atoms
    from a 1024-byte boundary, as include/moe.h states; 0 for sizes the layout cannot hold."""
    for kind, E, K, N in ((0, 3, 256, 160), (1, 2, 288, 96), (0, 128, 2880, 2880),
                          (1, 8, 14336, 4096)):
        C = 2 * N if kind == 0 else N
        Kp = (K + 127) // 128 * 128
        cbh = (N + 127) // 128
        CB = 2 * cbh if kind == 0 else cbh
        sf_off = (E * C * Kp // 2 + 1023) // 1024 * 1024
        assert L.moe_mx_tc_weights_size(kind, E, K, N) == sf_off + E * CB * (Kp // 128) * 512
    assert L.moe_mx_tc_weights_size(0, 2, 256, 48) == 0      # N not a multiple of 32
    assert L.moe_mx_tc_weights_size(1, 2, 200, 64) == 0      # K not a multiple of 32
    assert L.moe_mx_tc_weights_size(5, 2, 256, 64) == 0      # unknown kind


def test_mx_tc_validation(L):
    q = L.moe_quantize_weights_mx_tc
    assert q(0, FAKE, FAKE, 2, 200, 64, NULL) == 1            # K % 32
    assert q(0, FAKE, FAKE + 16, 2, 256, 64, NULL) == 1       # buffer not 256-byte aligned
    assert q(0, NULL, FAKE, 2, 256, 64, NULL) == 1            # no weights
    f = L.moe_forward_mx_tc
    need = L.moe_forward_mx_tc_workspace_size(100, 256, 8, 2, 128, 0)
    ok = [FAKE, FAKE, 100, 256, 8, 2, 128, 0, 1, FAKE, FAKE, NULL, NULL, 0, FAKE, FAKE, FAKE,
          FAKE, need, NULL]

    def call(**ch):
        a = list(ok)
        names = ["x", "logits", "T", "d", "E", "k", "I", "fn", "flags", "wgu", "wdn", "wsgu",
                 "wsdn", "Is", "ids", "w", "out", "ws", "ws_bytes", "stream"]
        for k_, v in ch.items():
            a[names.index(k_)] = v
        return f(*a)

    assert call(d=240) == 1                  # d % 32
    assert call(I=100) == 1                  # I % 32
    assert call(flags=4) == 1                # the combine weight is not fused on this path
    assert call(fn=3) == 1                   # bad score function
    assert call(k=9) == 1                    # k > E
    assert call(E=300, k=2) == 2             # E > 256
    assert call(wsgu=FAKE) == 1              # a shared expert without Is
    assert call(Is=64) == 1                  # Is without shared weights
    assert call(wgu=FAKE + 16) == 1          # weights not 256-byte aligned
    assert call(x=MIS) == 1                  # misaligned activations
    assert call(ws_bytes=need - 1) == 3      # workspace too small
    assert call(T=0, x=NULL, logits=NULL) == 0   # empty batch: nothing to do
    g = L.moe_gate_up_mx_tc
    # (x_codes, x_sf, offsets, s2p, w, R, d, E, I, w_gate_up, flags, h_codes, h_sf, ws, bytes, st)
    assert g(FAKE, FAKE, NULL, NULL, NULL, 100, 256, 4, 128, FAKE, 0, FAKE, FAKE, FAKE, 256,
             NULL) == 1                      # no offsets with E > 1
    assert g(FAKE, FAKE, FAKE, NULL, NULL, 100, 256, 4, 128, FAKE, 2, FAKE, FAKE, FAKE, 256,
             NULL) == 1                      # scaled input without the routing weights
    assert g(FAKE, FAKE, FAKE, NULL, NULL, 100, 256, 4, 128, FAKE, 0, FAKE, FAKE, FAKE, 255,
             NULL) == 3                      # no room for the status word
    assert g(FAKE, FAKE, FAKE, NULL, NULL, 0, 256, 4, 128, FAKE, 0, FAKE, FAKE, FAKE, 256,
             NULL) == 0                      # no rows
    r = L.moe_mx_tc_rows
    # (x, T, d, k, E, ids, s2p, offsets, codes, sf, codes_sh, sf_sh, stream)
    assert r(FAKE, 10, 200, 2, 8, FAKE, FAKE, FAKE, FAKE, FAKE, NULL, NULL, NULL) == 1  # d % 32
    assert r(FAKE, 10, 256, 2, 8, FAKE, FAKE, FAKE, FAKE, NULL, NULL, NULL, NULL) == 1  # no sf
    assert r(FAKE, 10, 256, 2, 8, NULL, FAKE, FAKE, FAKE, FAKE, NULL, NULL, NULL) == 1  # no ids
    assert r(NULL, 0, 256, 2, 8, FAKE, FAKE, FAKE, FAKE, FAKE, NULL, NULL, NULL) == 0   # T = 0


def test_mx_tc_workspace_views_fit_the_workspace(L):
    """The binding's views of moe_forward_mx_tc's workspace follow the library's layout: every
    view ends inside the size the library asks for."""
    import torch
    for (T, d, E, k, I, Is) in ((100, 256, 8, 2, 128, 0), (4096, 4096, 8, 2, 14336, 0),
                                (96, 256, 4, 1, 384, 192), (1, 1024, 32, 8, 384, 0)):
        n = L.moe_forward_mx_tc_workspace_size(T, d, E, k, I, Is)
        ws = torch.empty(n, dtype=torch.uint8)
        v = moe.mx_tc_workspace_views(ws, T, d, E, k, I, Is)
        for name, t in v.items():
            if isinstance(t, torch.Tensor):
                end = t.data_ptr() + t.numel() * t.element_size() - ws.data_ptr()
                assert end <= n, (name, end, n)
