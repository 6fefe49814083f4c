"""The seeded input generator: slice independence, prefix consistency, moments, and the
workload statistics the configurations ask for."""
import numpy as np
import pytest
import torch

from routing_dispatch_grouped_gb300 import synth


def test_slices_and_prefixes_are_consistent():
    full = synth.normal_f64(3, "w", 0, 10_000, 1.0)
    assert torch.equal(full[1234:5678], synth.normal_f64(3, "w", 1234, 5678 - 1234, 1.0))
    a = synth.normal((64, 32), torch.bfloat16, 0, "x", 1.0)
    b = synth.normal((8, 32), torch.bfloat16, 0, "x", 1.0)
    assert torch.equal(a[:8], b)


def test_streams_and_seeds_differ():
    a = synth.normal_f64(0, "x", 0, 1000, 1.0)
    assert not torch.equal(a, synth.normal_f64(1, "x", 0, 1000, 1.0))
    assert not torch.equal(a, synth.normal_f64(0, "y", 0, 1000, 1.0))


def test_moments_are_normal_like():
    v = synth.normal_f64(0, "m", 0, 1 << 20, 0.02).numpy()
    assert abs(v.mean()) < 0.02 * 0.01
    assert abs(v.std() / 0.02 - 1) < 0.01
    kurt = ((v - v.mean()) ** 4).mean() / v.var() ** 2
    assert abs(kurt - (3 - 1.2 / 8)) < 0.03          # Irwin-Hall(8) kurtosis


def test_chunked_fill_equals_direct():
    out = torch.empty(3 * (1 << 10) + 7, dtype=torch.float32)
    old = synth._CHUNK
    try:
        synth._CHUNK = 1 << 10
        synth.fill_normal(out, 0, "c", 1.0)
    finally:
        synth._CHUNK = old
    ref = synth.normal_f64(0, "c", 0, out.numel(), 1.0).to(torch.float32)
    assert torch.equal(out, ref)


def test_mix32_matches_uint64_arithmetic():
    """The int64 hash equals the same hash in numpy uint32 wrap-around arithmetic."""
    x = np.random.default_rng(0).integers(0, 1 << 32, 100_000, dtype=np.uint64)
    ref = x.astype(np.uint32)
    for _ in range(2):
        ref = (((ref >> np.uint32(16)) ^ ref) * np.uint32(0x45D9F3B)).astype(np.uint32)
    ref = (ref >> np.uint32(16)) ^ ref
    got = synth._mix32(torch.from_numpy(x.astype(np.int64)))
    assert np.array_equal(got.numpy().astype(np.uint32), ref)


@pytest.mark.slow
def test_scout_top_expert_share_near_30_percent():
    from oracle import moe_oracle as o
    cfg = synth.CONFIGS["llama4_scout"]
    inp = synth.make_inputs(cfg, weights=False)
    ids, _ = o.route(inp["logits"].numpy(), 1, o.SIGMOID, False)
    share = np.bincount(ids[:, 0], minlength=cfg.E).max() / cfg.T
    assert 0.28 <= share <= 0.32
