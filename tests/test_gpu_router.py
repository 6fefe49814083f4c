"""Parity of the router from hidden states (moe_route_hidden: fp32 logits x @ W_r + b and the
top-k in one kernel) with the CPU oracle.

- logits: within d * 2^-22 * sum_i |x_i w_ie| (plus the fp32 roundings of the bias add and of
  the result) of the exact value: the error bound of an fp32 sum of d products, with room for
  the tensor pipe's fp32 accumulation and the three-term bf16 split of W_r on the large-batch
  bf16 path;
- ids and weights: bit-identical to moe_route run on the kernel's own logits (same warp
  router), and ids bit-exact against the oracle's route on those fp32 logits;
- both launch shapes: clusters of 8 blocks splitting K (up to 1024 tokens) and 64 tokens per
  block (above);
- against the oracle's exact logits the ids may differ only where two experts' exact logits
  are closer than twice that bound (a near tie the fp32 sum cannot order); every such case is
  checked to be one.
"""
import numpy as np
import pytest
import torch

from oracle import moe_oracle as o
from routing_dispatch_grouped_gb300 import moe, synth
from tests.helpers import W_REL_TOL

pytestmark = pytest.mark.gpu
DEV = "cuda"

# (name, T, d, E, k, dtype, score_fn, renormalize, bias)
CASES = [
    ("gpt_oss_like", 300, 2880, 128, 4, torch.bfloat16, o.SOFTMAX, True, "normal0.5"),
    ("mixtral_like", 200, 4096, 8, 2, torch.bfloat16, o.SOFTMAX, True, None),
    ("scout_like", 130, 5120, 16, 1, torch.bfloat16, o.SIGMOID, False, "zipf1.2"),
    ("decode_T1", 1, 2048, 128, 8, torch.bfloat16, o.SOFTMAX, True, None),
    ("decode_T5", 5, 2048, 128, 8, torch.bfloat16, o.SOFTMAX, True, None),
    ("tiny_fp32", 256, 128, 8, 2, torch.float32, o.SOFTMAX, True, None),
    ("ragged", 67, 100, 37, 5, torch.bfloat16, o.SOFTMAX, False, "normal0.5"),
    ("e256", 70, 64, 256, 8, torch.float32, o.SIGMOID, True, None),
    # above 1024 tokens: 64 tokens per block, all of K in one block (a ragged last block); bf16
    # x takes the tensor-pipe kernel
    ("large_T", 1100, 2880, 128, 4, torch.bfloat16, o.SOFTMAX, True, "normal0.5"),
    ("large_T_e256", 1090, 96, 256, 8, torch.bfloat16, o.SOFTMAX, True, None),
]


def _inputs(name, T, d, E, dtype, bias):
    x = synth.normal((T, d), dtype, 0, "rh_x_" + name, 1.0, device=DEV)
    w = synth.normal((d, E), torch.float32, 0, "rh_w_" + name, 0.02, device=DEV)
    b = None
    if bias == "normal0.5":
        b = synth.normal((E,), torch.float32, 0, "rh_b_" + name, 0.5, device=DEV)
    elif bias == "zipf1.2":
        b = synth.zipf_bias(E).to(torch.float32).to(DEV)
    return x, w, b


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_route_hidden_matches_oracle(case):
    name, T, d, E, k, dtype, fn, renorm, bias = case
    x, w, b = _inputs(name, T, d, E, dtype, bias)
    ids, wt, logits = moe.moe_route_hidden(x, w, k, fn, renorm, bias=b)
    torch.cuda.synchronize()
    x64 = x.double().cpu().numpy()
    w64 = w.double().cpu().numpy()
    b64 = None if b is None else b.double().cpu().numpy()
    exact = o.router_logits(x64, w64, b64)
    bound = (d * 2.0 ** -22 * (np.abs(x64) @ np.abs(w64))
             + 2.0 ** -23 * np.abs(exact) + (0 if b64 is None else 2.0 ** -24 * np.abs(b64)))
    got = logits.double().cpu().numpy()
    assert np.all(np.abs(got - exact) <= bound), np.max(np.abs(got - exact) / bound)

    # the same warp router as moe_route: identical ids and weights on the kernel's logits
    ids_r, wt_r = moe.moe_route(logits, k, fn, renorm)
    assert torch.equal(ids, ids_r) and torch.equal(wt, wt_r)
    # and the oracle's route on those fp32 logits
    ref_ids, ref_w = o.route(logits.cpu().numpy(), k, fn, renorm)
    assert np.array_equal(ids.cpu().numpy(), ref_ids)
    assert (np.abs(wt.cpu().numpy() - ref_w) / ref_w).max() <= W_REL_TOL

    # against the exact logits: any different id must be a near tie
    ex_ids, _ = o.route(exact, k, fn, renorm)
    gi = ids.cpu().numpy()
    for t, j in zip(*np.nonzero(gi != ex_ids)):
        a, c = gi[t, j], ex_ids[t, j]
        assert abs(exact[t, a] - exact[t, c]) <= bound[t, a] + bound[t, c], (t, j, a, c)


def test_route_hidden_without_logits_output():
    name, T, d, E, k, dtype, fn, renorm, bias = CASES[0]
    x, w, b = _inputs(name, T, d, E, dtype, bias)
    ids, wt, logits = moe.moe_route_hidden(x, w, k, fn, renorm, bias=b)
    ids2, wt2, none = moe.moe_route_hidden(x, w, k, fn, renorm, bias=b, want_logits=False)
    assert none is None
    assert torch.equal(ids, ids2) and torch.equal(wt, wt2)


def test_route_hidden_empty_batch():
    x = torch.empty(0, 64, dtype=torch.bfloat16, device=DEV)
    w = torch.zeros(64, 8, dtype=torch.float32, device=DEV)
    ids, wt, logits = moe.moe_route_hidden(x, w, 2)
    assert ids.shape == (0, 2) and logits.shape == (0, 8)
