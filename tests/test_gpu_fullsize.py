"""Full-size parity of the whole layer in the launch configuration the benchmark times.

Every tensor of the layer is compared with the oracle over every token: routing, counts,
offsets, permutations and x_sorted bit for bit; the SwiGLU activation h (and the shared
expert's) within one bf16 ulp; y_sorted, the shared expert's y and the layer output within the
workload's bar. The oracle runs the whole layer in float64 (seconds to tens of seconds on the
host cores)."""
import numpy as np
import pytest
import torch

from oracle import moe_oracle as o
from routing_dispatch_grouped_gb300 import moe, synth
from tests.helpers import TOL, W_REL_TOL, Expertwise, bits, err_rms, f64, within_one_bf16_ulp

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _flags(cfg):
    return (moe.RENORMALIZE if cfg.renormalize else 0) | (moe.SCALE_INPUT if cfg.scale_input else 0)


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
    sh = inp["w_shared_gate_up"]
    ref = o.forward(f64(inp["x"]), inp["logits"].cpu().numpy(), Expertwise(inp["w_gate_up"]),
                    Expertwise(inp["w_down"]), cfg.k, cfg.score_fn, cfg.renormalize,
                    cfg.scale_input, True, None if sh is None else f64(sh),
                    None if sh is None else f64(inp["w_shared_down"]))
    assert np.array_equal(ids.cpu().numpy(), ref["topk_ids"])
    rw = ref["topk_weights"]
    assert (np.abs(w.cpu().numpy() - rw) / rw).max() <= W_REL_TOL
    v = moe.forward_workspace_views(ws, cfg.T, cfg.d, cfg.E, cfg.k, cfg.I, cfg.I_shared, cfg.dtype)
    for n in ("counts", "offsets", "sorted_to_slot", "slot_to_sorted"):
        assert np.array_equal(v[n].cpu().numpy(), ref[n]), n
    assert np.array_equal(bits(v["x_sorted"]), o.permute_rows(bits(inp["x"]), ref["sorted_to_slot"],
                                                              cfg.k))
    tol = TOL[cfg.dtype]
    # every row of every expert tile the timed kernels produce
    assert within_one_bf16_ulp(f64(v["h"]), ref["h"])
    assert err_rms(f64(v["y_sorted"]), ref["y_sorted"]) <= tol
    if cfg.I_shared:
        assert within_one_bf16_ulp(f64(v["h_shared"]), ref["h_shared"])
        assert err_rms(f64(v["y_shared"]), ref["y_shared"]) <= tol
    e = err_rms(f64(out), ref["out"])
    assert e <= tol, e
