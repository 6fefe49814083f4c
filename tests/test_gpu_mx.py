"""Parity of the MX (block-scaled FP8/FP4) kernels and layer with the MX oracle.

Bit-exact: MXFP4 weight codes and scales, their dequantized bf16 values, MXFP8 row codes and
scales and the rounded rows (the quantisation decisions are taken on the same bf16 values on
both sides), router ids. Within the bar: the layer output (2e-2 rms); the SwiGLU activation h,
which the GPU rounds to MXFP8 from its fp32 value and the oracle from its float64 value, may
land one E4M3 step apart where the two sit on either side of a rounding midpoint (rare), and is
checked elementwise against that.
"""
import numpy as np
import pytest
import torch

from oracle import moe_mx as M
from routing_dispatch_grouped_gb300 import moe, synth
from tests.helpers import HostMX, err_rms, f64, mx_weight_views

pytestmark = pytest.mark.gpu
DEV = "cuda"
bf16 = torch.bfloat16


@pytest.fixture(scope="module", autouse=True)
def _loaded():
    assert torch.cuda.is_available(), "GPU tests need a GPU"
    moe.lib()


def _special_columns(w):
    """Plant blocks that exercise the corners: an all-zero block, a block whose largest value
    saturates (amax / 2^s in (6, 8)), and E2M1 ties (midpoints at the block's scale)."""
    w = w.clone()
    w[0, 0:32, 0] = 0
    w[0, 0:32, 1] = 0.01
    w[0, 5, 1] = 7.0 * 2 ** -6   # s = floor(log2 0.109) - 2 = -6: 7 saturates to 6
    w[0, 32:64, 2] = torch.tensor([1.0, 0.25 * 1, 0.75 * 0.25, 1.25 * 0.25, 1.75 * 0.25,
                                   2.5 * 0.25, 3.5 * 0.25, 5.0 * 0.25] * 4, dtype=bf16)
    return w


@pytest.mark.parametrize("kind,E,K,N", [(moe.W_GATE_UP, 3, 200, 136), (moe.W_DOWN, 2, 264, 96),
                                        (moe.W_GATE_UP, 1, 64, 64)])
def test_weight_quantisation_bit_exact(kind, E, K, N):
    cols = 2 * N if kind == moe.W_GATE_UP else N
    w = synth.normal((E, K, cols), bf16, 0, f"mxw{kind}{K}", 0.02, device=DEV)
    w = _special_columns(w)
    mx = moe.quantize_weights_mx(w, kind)
    deq = moe.dequantize_weights_mx(mx)
    torch.cuda.synchronize()
    got, scales = mx_weight_views(mx)
    rc, rs = M.quantize_mx(f64(w), M.E2M1, axis=1)
    assert np.array_equal(scales, rs)
    assert np.array_equal(got, rc)
    assert np.array_equal(f64(deq), M.dequantize_mx(rc, rs, M.E2M1, axis=1))


@pytest.mark.parametrize("R,K", [(77, 200), (256, 2048), (3, 64)])
def test_row_quantisation_bit_exact(R, K):
    x = synth.normal((R, K), bf16, 0, f"mxr{K}", 1.0, device=DEV)
    x[0, :32] = 0                       # zero block
    x[1, :32] = 2.0 ** -3               # amax 2^-3: s = -11, values 256 exactly
    # E4M3 ties at scale s = 0 (amax 256): 1.0625 (1 / 1.125), 17 (16 / 18), 300 (288 / 320)
    x[2, 32:64] = torch.tensor([256.0, 1.0625, 17.0, 300.0] * 8, dtype=bf16)
    xo, codes, scales = moe.quantize_rows_mx(x)
    torch.cuda.synchronize()
    rc, rs = M.quantize_mx(f64(x), M.E4M3, axis=1)
    assert np.array_equal(scales.cpu().numpy(), rs)
    assert np.array_equal(codes.cpu().numpy(), rc)
    assert np.array_equal(f64(xo), M.dequantize_mx(rc, rs, M.E4M3, axis=1))


CASES = [  # (name, T, d, E, k, I, score fn, renorm, scaled input, shared I, bias)
    ("mixtral_like", 200, 512, 8, 2, 640, M.fwd.SOFTMAX, True, False, 0, "none"),
    ("gptoss_like", 150, 264, 16, 4, 200, M.fwd.SOFTMAX, True, False, 0, "normal0.5"),
    ("scout_like", 96, 256, 4, 1, 384, M.fwd.SIGMOID, False, True, 192, "zipf1.2"),
    # decode batches: the one-kernel layer on the MX weights (x and h rounded in the kernel)
    ("decode_T1", 1, 1024, 32, 8, 384, M.fwd.SOFTMAX, True, False, 0, "none"),
    ("decode_T8", 8, 1024, 32, 8, 384, M.fwd.SOFTMAX, True, False, 0, "none"),
    ("decode_T16", 16, 2048, 128, 8, 768, M.fwd.SOFTMAX, True, False, 0, "none"),
    ("decode_ragged", 5, 264, 16, 4, 200, M.fwd.SOFTMAX, False, False, 0, "normal0.5"),
    ("decode_sigmoid_scaled", 6, 512, 8, 1, 136, M.fwd.SIGMOID, False, True, 0, "none"),
    ("decode_one_expert", 3, 256, 4, 4, 64, M.fwd.SOFTMAX, True, False, 0, "none"),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_mx_layer_matches_oracle(case):
    name, T, d, E, k, I, fn, renorm, scale, Is, bias = case
    cfg = synth.MoEConfig(name, T, d, E, k, I, bf16, score_fn=fn, renormalize=renorm,
                          scale_input=scale, I_shared=Is, bias=bias)
    inp = synth.make_inputs(cfg, DEV)
    mgu = moe.quantize_weights_mx(inp["w_gate_up"], moe.W_GATE_UP)
    mdn = moe.quantize_weights_mx(inp["w_down"], moe.W_DOWN)
    msgu = moe.quantize_weights_mx(inp["w_shared_gate_up"], moe.W_GATE_UP) if Is else None
    msdn = moe.quantize_weights_mx(inp["w_shared_down"], moe.W_DOWN) if Is else None
    flags = (moe.RENORMALIZE if renorm else 0) | (moe.SCALE_INPUT if scale else 0)
    out, ids, w, ws = moe.moe_forward_mx(inp["x"], inp["logits"], mgu, mdn, k, fn, flags,
                                         msgu, msdn)
    torch.cuda.synchronize()
    assert moe.moe_read_device_status(ws) == 0
    # the oracle's weights are quantised on the host from the bf16 weights, one expert at a
    # time; the device quantiser is checked against them separately (bit for bit, below)
    hgu, hdn = HostMX(inp["w_gate_up"]), HostMX(inp["w_down"])
    sh = {}
    if Is:
        sh = dict(wsgu_deq=HostMX(inp["w_shared_gate_up"][None])[0],
                  wsd_deq=HostMX(inp["w_shared_down"][None])[0])
    ref = M.mx_forward(f64(inp["x"]), inp["logits"].cpu().numpy(), hgu, hdn, k, fn, renorm,
                       scale, **sh)
    assert np.array_equal(ids.cpu().numpy(), ref["topk_ids"])
    v = moe.forward_workspace_views(ws, T, d, E, k, I, Is, bf16, mx=True)
    fused = moe.moe_forward_kernel_count(T, k, Is) == 1
    if not fused:  # x_sorted: the MXFP8 rounding of x, permuted (bit-exact)
        assert np.array_equal(f64(v["x_sorted"]), ref["x_sorted"])
    else:  # the kernel keeps h's codes for its down items: they encode the h it wrote
        hc = v["h_codes"].cpu().numpy()
        hs = v["h_scales"].cpu().numpy()
        assert np.array_equal(M.dequantize_mx(hc, hs, M.E4M3, axis=1), f64(v["h"]))
    # h: MXFP8 values; where the GPU's fp32 h and the oracle's float64 h round apart it is by
    # one E4M3 step (2^-3 of the value) or, when the block's largest value crosses a power of
    # two, by the scale step; such places are rare
    hg, hr = f64(v["h"]), ref["hq"]
    off = np.abs(hg - hr) > 0
    assert off.mean() <= 2e-3, off.mean()
    assert np.all(np.abs(hg - hr)[off] <= 2.0 ** -3 * np.maximum(np.abs(hg), np.abs(hr))[off]
                  + 2.0 ** -9 * np.abs(hr).max())
    e = err_rms(f64(out), ref["out"])
    assert e <= 2e-2, e
    # the weights the layer ran on: the device's dequantized MXFP4 values equal the host
    # quantisation of this workload's own bf16 weights
    pairs = [(mgu, hgu), (mdn, hdn)]
    if Is:
        pairs += [(msgu, HostMX(inp["w_shared_gate_up"][None])),
                  (msdn, HostMX(inp["w_shared_down"][None]))]
    for mx_w, host in pairs:
        deq = moe.dequantize_weights_mx(mx_w)
        for ex in range(len(host)):
            assert np.array_equal(f64(deq[ex]), host[ex]), ex
