"""Parity of the one-kernel decode path of moe_forward (bf16, no shared expert, T <= 16,
T*k <= 256: one cooperative kernel routes, dispatches, runs gate_up + SwiGLU and down and
combines) with the CPU oracle.

Bit-exact: router ids, counts, offsets, both permutations. Within the stated tolerance: h (one
bf16 ulp) and the layer output (the fused path folds the combine into the down step and leaves
no y_sorted). The cases cover ragged d and I (tails of the 64-column
blocks and of the 128/256-row K chunks), more than 8 rows per expert (two reduction passes),
one expert, the largest T*k, the sigmoid/scale-input router, the fused combine weight, both
weight layouts, determinism and graph replay.
"""
import dataclasses

import numpy as np
import pytest
import torch

from oracle import moe_oracle as o
from routing_dispatch_grouped_gb300 import moe, synth
from tests.helpers import TOL, W_REL_TOL, Expertwise, err_rms, f64, within_one_bf16_ulp

pytestmark = pytest.mark.gpu
DEV = "cuda"

_BASE = synth.CONFIGS["decode"]
CASES = {
    "decode_T1": _BASE.with_T(1),
    "decode_T8": _BASE.with_T(8),
    "decode_T16": _BASE.with_T(16),
    # d, I not multiples of 64; sigmoid score applied to the input, no renormalisation
    "ragged_sigmoid": dataclasses.replace(_BASE, name="ragged_sigmoid", T=5, d=200, E=16, k=4,
                                          I=136, score_fn=synth.SIGMOID, renormalize=False,
                                          scale_input=True),
    # T*k = 256, the largest batch the fused kernel takes; fewer work items than SMs in the
    # one_expert case below (empty per-block ranges)
    "max_rows": dataclasses.replace(_BASE, name="max_rows", T=16, d=640, E=40, k=16, I=320),
    # up to 16 rows per expert: two 8-row reduction passes
    "crowded": dataclasses.replace(_BASE, name="crowded", T=16, d=1024, E=4, k=2, I=1024),
    "one_expert": dataclasses.replace(_BASE, name="one_expert", T=16, d=384, E=1, k=1, I=448),
}


def _flags(cfg, fuse=False):
    f = moe.RENORMALIZE if cfg.renormalize else 0
    f |= moe.SCALE_INPUT if cfg.scale_input else 0
    f |= moe.FUSE_COMBINE_WEIGHT if fuse else 0
    return f


def _weights(inp, packed):
    if not packed:
        return inp["w_gate_up"], inp["w_down"]
    return (moe.pack_weights(inp["w_gate_up"], moe.W_GATE_UP),
            moe.pack_weights(inp["w_down"], moe.W_DOWN))


def _h_ref(cfg, inp, ref):
    """h of every sorted row from the oracle's dispatch, rounded to bf16 as both sides store it."""
    xs, offsets = ref["x_sorted"], ref["offsets"]
    w = ref["topk_weights"].reshape(-1)[ref["sorted_to_slot"]]
    wgu = Expertwise(inp["w_gate_up"])
    h = np.zeros((xs.shape[0], cfg.I))
    for e in range(cfg.E):
        a, b = offsets[e], offsets[e + 1]
        if b > a:
            g = xs[a:b] @ wgu[e][:, :cfg.I]
            u = xs[a:b] @ wgu[e][:, cfg.I:]
            if cfg.scale_input:
                g, u = g * w[a:b, None], u * w[a:b, None]
            h[a:b] = g / (1 + np.exp(-g)) * u
    return o.round_bf16(h)


@pytest.mark.parametrize("packed", [False, True])
@pytest.mark.parametrize("name", list(CASES))
def test_decode_fused_matches_oracle(name, packed):
    cfg = CASES[name]
    assert moe.moe_forward_kernel_count(cfg.T, cfg.k, 0, cfg.dtype) == 1
    inp = synth.make_inputs(cfg, DEV)
    wgu, wd = _weights(inp, packed)
    out, ids, w, ws = moe.moe_forward(inp["x"], inp["logits"], wgu, wd, cfg.k, cfg.score_fn,
                                      _flags(cfg))
    assert moe.moe_read_device_status(ws) == 0
    ref = o.forward(f64(inp["x"]), inp["logits"].cpu().numpy(), Expertwise(inp["w_gate_up"]),
                    Expertwise(inp["w_down"]), cfg.k, cfg.score_fn, cfg.renormalize,
                    cfg.scale_input, True)
    assert np.array_equal(ids.cpu().numpy(), ref["topk_ids"])
    assert (np.abs(w.cpu().numpy() - ref["topk_weights"]) / ref["topk_weights"]).max() <= W_REL_TOL
    v = moe.forward_workspace_views(ws, cfg.T, cfg.d, cfg.E, cfg.k, cfg.I, 0, cfg.dtype)
    for key in ("counts", "offsets", "sorted_to_slot", "slot_to_sorted"):
        assert np.array_equal(v[key].cpu().numpy(), ref[key]), key
    assert within_one_bf16_ulp(f64(v["h"]), _h_ref(cfg, inp, ref))
    tol = TOL[cfg.dtype]
    e = err_rms(f64(out), ref["out"])
    assert e <= tol, e


def test_decode_fused_combine_weight_flag():
    cfg = CASES["max_rows"]
    inp = synth.make_inputs(cfg, DEV)
    out, _, w, ws = moe.moe_forward(inp["x"], inp["logits"], inp["w_gate_up"], inp["w_down"],
                                    cfg.k, cfg.score_fn, _flags(cfg, fuse=True))
    assert moe.moe_read_device_status(ws) == 0
    ref = o.forward(f64(inp["x"]), inp["logits"].cpu().numpy(), Expertwise(inp["w_gate_up"]),
                    Expertwise(inp["w_down"]), cfg.k, cfg.score_fn, cfg.renormalize, False, True)
    assert err_rms(f64(out), ref["out"]) <= TOL[cfg.dtype]


@pytest.mark.parametrize("name", ["decode_T8", "decode_T1", "crowded"])
def test_decode_fused_is_deterministic_and_replays_in_a_graph(name):
    """Every partial sum is reduced in a fixed order, so repeated calls give the same bits, and
    the launch captures into a CUDA graph. T=1 and the crowded case run the layout where each
    touched h block has a block of its own; T=8 the stream-K layout."""
    cfg = CASES[name]
    inp = synth.make_inputs(cfg, DEV)
    wgu, wd = _weights(inp, True)
    out, ids, w, ws = moe.moe_forward(inp["x"], inp["logits"], wgu, wd, cfg.k)
    first = out.clone()
    for _ in range(3):
        moe.moe_forward(inp["x"], inp["logits"], wgu, wd, cfg.k, out=out, topk_ids=ids,
                        topk_weights=w, workspace=ws)
        assert torch.equal(out, first)
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            moe.moe_forward(inp["x"], inp["logits"], wgu, wd, cfg.k, out=out, topk_ids=ids,
                            topk_weights=w, workspace=ws, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(3):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, first)
    assert moe.moe_read_device_status(ws) == 0
