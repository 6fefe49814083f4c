"""Full-size parity of the whole layer in the launch configuration the benchmark times.

Routing, counts, offsets, permutations and x_sorted are compared over every token; the layer
output is compared on a sample of tokens that the oracle computes one at a time (every expert
the sample routes to is covered, including the heaviest and the lightest)."""
import numpy as np
import pytest
import torch

from oracle import moe_oracle as o
from routing_dispatch_grouped_gb300 import moe, synth
from tests.helpers import TOL, W_REL_TOL, Expertwise, bits, err_rms, f64

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _flags(cfg):
    return (moe.RENORMALIZE if cfg.renormalize else 0) | (moe.SCALE_INPUT if cfg.scale_input else 0)


def _sample_tokens(ids, E, n=40, seed=0):
    rng = np.random.default_rng(seed)
    T = ids.shape[0]
    pick = set(rng.choice(T, size=min(n, T), replace=False).tolist()) | {0, T - 1}
    counts = np.bincount(ids.reshape(-1), minlength=E)
    for e in (int(np.argmax(counts)), int(np.argmin(np.where(counts > 0, counts, 1 << 30)))):
        rows = np.nonzero((ids == e).any(axis=1))[0]
        pick |= set(rows[:2].tolist())
    return sorted(pick)


@pytest.mark.parametrize("name", ["mixtral_8x7b", "gpt_oss_120b", "llama4_scout"])
def test_forward_full_size(name):
    cfg = synth.CONFIGS[name]
    inp = synth.make_inputs(cfg, DEV)
    # the benchmark's configuration: expert weights packed once, then the layer
    pk = {n: moe.pack_weights(inp[n], moe.W_GATE_UP if "gate_up" in n else moe.W_DOWN)
          if inp[n] is not None else None
          for n in ("w_gate_up", "w_down", "w_shared_gate_up", "w_shared_down")}
    out, ids, w, ws = moe.moe_forward(inp["x"], inp["logits"], pk["w_gate_up"], pk["w_down"],
                                      cfg.k, cfg.score_fn, _flags(cfg), pk["w_shared_gate_up"],
                                      pk["w_shared_down"])
    del pk
    assert moe.moe_read_device_status(ws) == 0
    rid, rw = o.route(inp["logits"].cpu().numpy(), cfg.k, cfg.score_fn, cfg.renormalize)
    assert np.array_equal(ids.cpu().numpy(), rid)
    assert (np.abs(w.cpu().numpy() - rw) / rw).max() <= W_REL_TOL
    counts, offsets, s2p, p2s = o.dispatch(rid, cfg.E)
    v = moe.forward_workspace_views(ws, cfg.T, cfg.d, cfg.E, cfg.k, cfg.I, cfg.I_shared, cfg.dtype)
    assert np.array_equal(v["counts"].cpu().numpy(), counts)
    assert np.array_equal(v["offsets"].cpu().numpy(), offsets)
    assert np.array_equal(v["sorted_to_slot"].cpu().numpy(), s2p)
    assert np.array_equal(v["slot_to_sorted"].cpu().numpy(), p2s)
    assert np.array_equal(bits(v["x_sorted"]), o.permute_rows(bits(inp["x"]), s2p, cfg.k))

    toks = _sample_tokens(rid, cfg.E)
    sh = inp["w_shared_gate_up"]
    ref = o.token_outputs(range(len(toks)), f64(inp["x"][toks]), rid[toks], rw[toks],
                          Expertwise(inp["w_gate_up"]), Expertwise(inp["w_down"]),
                          cfg.scale_input, True,
                          None if sh is None else f64(sh),
                          None if sh is None else f64(inp["w_shared_down"]))
    e = err_rms(f64(out[toks]), ref)
    assert e <= TOL[cfg.dtype], e
