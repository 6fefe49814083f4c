"""Parity of the CUDA path (called through the C ABI) with the CPU oracle.

Bit-exact: router ids, counts, offsets, both permutations, x_sorted. Within the stated tolerance:
router weights, h, y_sorted and the layer output. Sizes span several tiles with ragged tails;
the workloads' own shapes run at reduced token counts here (the whole oracle finishes in
seconds) and at full size in test_gpu_fullsize.py.
"""
import dataclasses

import numpy as np
import pytest
import torch

from oracle import moe_oracle as o
from routing_dispatch_grouped_gb300 import moe, synth
from tests.helpers import TOL, W_REL_TOL, Expertwise, bits, err_rms, f64, within_one_bf16_ulp

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _loaded():
    assert torch.cuda.is_available(), "GPU tests need a GPU"
    moe.lib()


def _cfg(name, T=None):
    cfg = synth.CONFIGS[name]
    return cfg if T is None else cfg.with_T(T)


# ------------------------------------------------------------------------------------------------
# generator: device and host produce the same bits
# ------------------------------------------------------------------------------------------------
def test_generator_cpu_equals_cuda():
    a = synth.normal((1000, 37), torch.bfloat16, 0, "x", 1.0, device=DEV)
    b = synth.normal((1000, 37), torch.bfloat16, 0, "x", 1.0, device="cpu")
    assert np.array_equal(bits(a), bits(b))
    a = synth.normal_f64(5, "w", 123456, 100000, 0.02, device=DEV).cpu()
    b = synth.normal_f64(5, "w", 123456, 100000, 0.02, device="cpu")
    assert torch.equal(a, b)


# ------------------------------------------------------------------------------------------------
# route
# ------------------------------------------------------------------------------------------------
ROUTE_CASES = [("tiny_fp32", None), ("mixtral_8x7b", None), ("gpt_oss_120b", None),
               ("decode", 1), ("decode", 8), ("decode", 64), ("llama4_scout", None)]


@pytest.mark.parametrize("name,T", ROUTE_CASES)
def test_route_matches_oracle(name, T):
    cfg = _cfg(name, T)
    inp = synth.make_inputs(cfg, DEV, weights=False)
    ids, w = moe.moe_route(inp["logits"], cfg.k, cfg.score_fn, cfg.renormalize)
    rid, rw = o.route(inp["logits"].cpu().numpy(), cfg.k, cfg.score_fn, cfg.renormalize)
    assert np.array_equal(ids.cpu().numpy(), rid)
    rel = np.abs(w.cpu().numpy() - rw) / np.abs(rw)
    assert rel.max() <= W_REL_TOL, rel.max()


@pytest.mark.parametrize("E,k", [(8, 2), (37, 5), (128, 8), (256, 8), (16, 1), (32, 32), (5, 5)])
def test_route_ties_inf_nan(E, k):
    rng = np.random.default_rng(E + 100 * k)
    z = rng.integers(-3, 4, size=(300, E)).astype(np.float32) * np.float32(0.5)
    z[rng.random(z.shape) < 0.05] = -np.inf
    z[rng.random(z.shape) < 0.05] = -0.0
    z[rng.random(z.shape) < 0.03] = np.nan
    z[0, :] = 1.0    # a row of all ties
    ids, _ = moe.moe_route(torch.from_numpy(z).to(DEV), k)
    rid, _ = o.route(z, k)
    assert np.array_equal(ids.cpu().numpy(), rid)


@pytest.mark.parametrize("fn,renorm", [(o.SOFTMAX, False), (o.SIGMOID, True), (o.SIGMOID, False)])
def test_route_score_variants(fn, renorm):
    rng = np.random.default_rng(3)
    z = (rng.standard_normal((777, 64)) * 1.7).astype(np.float32)
    ids, w = moe.moe_route(torch.from_numpy(z).to(DEV), 6, fn, renorm)
    rid, rw = o.route(z, 6, fn, renorm)
    assert np.array_equal(ids.cpu().numpy(), rid)
    assert (np.abs(w.cpu().numpy() - rw) / rw).max() <= W_REL_TOL


# ------------------------------------------------------------------------------------------------
# dispatch
# ------------------------------------------------------------------------------------------------
def _check_dispatch(ids_np, E, x):
    T, k = ids_np.shape
    ids = torch.from_numpy(ids_np.astype(np.int32)).to(DEV)
    r = moe.moe_dispatch(ids, E, x=x)
    counts, offsets, s2p, p2s = o.dispatch(ids_np, E)
    assert np.array_equal(r["counts"].cpu().numpy(), counts)
    assert np.array_equal(r["offsets"].cpu().numpy(), offsets)
    assert np.array_equal(r["sorted_to_slot"].cpu().numpy(), s2p)
    assert np.array_equal(r["slot_to_sorted"].cpu().numpy(), p2s)
    if x is not None:
        assert np.array_equal(bits(r["x_sorted"]), o.permute_rows(bits(x), s2p, k))
    assert moe.moe_read_device_status(r["workspace"]) == 0


@pytest.mark.parametrize("name,T", ROUTE_CASES)
def test_dispatch_matches_oracle(name, T):
    cfg = _cfg(name, T)
    inp = synth.make_inputs(cfg, DEV, weights=False)
    rid, _ = o.route(inp["logits"].cpu().numpy(), cfg.k, cfg.score_fn, cfg.renormalize)
    _check_dispatch(rid, cfg.E, inp["x"])


@pytest.mark.parametrize("case", ["all_experts", "one_expert", "sparse", "ragged", "single",
                                  "E1", "big_ragged", "empty"])
def test_dispatch_edge_cases(case):
    rng = np.random.default_rng(0)
    if case == "all_experts":
        E, ids = 8, np.tile(np.arange(8), (5, 1))
    elif case == "one_expert":
        E, ids = 16, np.full((700, 1), 11)
    elif case == "sparse":     # most experts empty
        E, ids = 256, np.stack([rng.choice([3, 200, 255], 2, replace=False) for _ in range(513)])
    elif case == "ragged":
        E, ids = 37, np.stack([rng.permutation(37)[:3] for _ in range(333)])
    elif case == "single":
        E, ids = 128, rng.permutation(128)[:8][None, :]
    elif case == "E1":
        E, ids = 1, np.zeros((77, 1), int)
    elif case == "empty":      # T = 0: counts and offsets are all zero
        E, ids = 12, np.zeros((0, 3), int)
    else:
        E, ids = 64, np.stack([rng.permutation(64)[:6] for _ in range(10007)])
    x = synth.normal((ids.shape[0], 40), torch.bfloat16, 1, "xd", 1.0, device=DEV)
    _check_dispatch(ids, E, x)
    _check_dispatch(ids, E, None)


def test_dispatch_invalid_ids_set_status_and_are_skipped():
    rng = np.random.default_rng(1)
    E, k, T = 8, 2, 600
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    bad = rng.random(ids.shape) < 0.05
    ids[bad] = np.where(rng.random(bad.sum()) < 0.5, -1, E + 3)
    r = moe.moe_dispatch(torch.from_numpy(ids).to(DEV), E)
    assert moe.moe_read_device_status(r["workspace"]) == 5
    flat = ids.reshape(-1)
    valid = (flat >= 0) & (flat < E)
    # reference: the stable counting sort over the valid slots only
    order = [s for e in range(E) for s in range(flat.size) if flat[s] == e]
    assert r["sorted_to_slot"][:len(order)].cpu().numpy().tolist() == order
    p2s = r["slot_to_sorted"].cpu().numpy()
    assert np.all(p2s[~valid] == -1)
    assert r["offsets"][-1].item() == valid.sum()


# ------------------------------------------------------------------------------------------------
# combine
# ------------------------------------------------------------------------------------------------
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("k,weighted,shared", [(2, True, False), (8, True, True), (1, False, True),
                                               (4, False, False)])
def test_combine_matches_oracle(dtype, k, weighted, shared):
    rng = np.random.default_rng(k)
    T, E, d = 1000, 16, 264
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)])
    _, _, s2p, p2s = o.dispatch(ids, E)
    y = synth.make_y_sorted(T * k, d, device=DEV)
    w = torch.rand(T, k, device=DEV) if weighted else None
    ys = synth.normal((T, d), torch.float32, 2, "ys", 1.0, device=DEV) if shared else None
    p2s_t = torch.from_numpy(p2s.astype(np.int32)).to(DEV)
    out = moe.moe_combine(y, p2s_t, k, dtype, topk_weights=w, y_shared=ys)
    ref = o.combine(f64(y), p2s, None if w is None else f64(w), k,
                    None if ys is None else f64(ys))
    if dtype == torch.float32:
        assert err_rms(f64(out), ref) <= 1e-6
    else:
        # one rounding to bf16: within half a bf16 ulp (2^-9 relative) plus fp32 summation error
        assert np.all(np.abs(f64(out) - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-5)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_identity_experts_roundtrip(dtype):
    """Dispatch then combine with identity experts (y = x_sorted): k = 1, weight 1 returns x
    exactly; k = 2 with weight 1 returns 2x exactly (a power-of-two scale)."""
    rng = np.random.default_rng(7)
    T, E, d = 513, 8, 136
    x = synth.normal((T, d), dtype, 3, "xi", 1.0, device=DEV)
    for k, scale in [(1, 1.0), (2, 2.0)]:
        ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
        r = moe.moe_dispatch(torch.from_numpy(ids).to(DEV), E, x=x)
        out = moe.moe_combine(r["x_sorted"].float(), r["slot_to_sorted"], k, dtype)
        assert torch.equal(out, (x.float() * scale).to(dtype))


# ------------------------------------------------------------------------------------------------
# grouped GEMMs (gate_up + SwiGLU, down)
# ------------------------------------------------------------------------------------------------
def _gemm_case(counts, d, I, dtype, seed=0):
    E = len(counts)
    R = int(sum(counts))
    offsets = np.zeros(E + 1, np.int64)
    offsets[1:] = np.cumsum(counts)
    xs = synth.normal((R, d), dtype, seed, "gx", 1.0, device=DEV)
    wgu = synth.normal((E, d, 2 * I), dtype, seed, "gwgu", 0.05, device=DEV)
    wd = synth.normal((E, I, d), dtype, seed, "gwd", 0.05, device=DEV)
    return offsets, xs, wgu, wd


GEMM_SHAPES = [
    # counts per expert, d, I
    ([130, 0, 257], 256, 384),          # ragged M tails, an empty expert
    ([1, 2, 3, 128, 129], 128, 128),    # tiny groups, exact tile, one over
    ([300], 200, 200),                  # K and N not multiples of 64 (TMA zero fill, masks)
    ([64] * 16 + [0] * 4, 512, 768),    # many groups
    ([1000, 24], 1024, 1024),           # several M tiles and N tiles per expert
    ([700, 600], 384, 200),             # >= 512 rows per expert: down on CTA pairs, ragged K/N
    # more than 512 rows: routed down with the weights as the M side of CTA pairs; the experts'
    # last token tiles (5, 44, 17, 100, 250 rows) take the 8-, 32-, 16-, 64- and 128-row boxes
    ([5, 300, 0, 17, 100, 250], 320, 256),
    # experts averaging >= 512 rows: gate_up on 256-row CTA pairs, with empty experts and tails
    # that leave the second CTA of a pair without rows (90, 1700 = 6 x 256 + 164)
    ([0, 1700, 0, 90, 900], 256, 320),
    # more than 512 rows, experts ending on swapped gate_up tails: 600 = 2 x 256 + 88, exactly
    # 128 (the largest swapped tail, through the 64-row box), 129 (one over: a half-empty pair
    # tile), 300 = 256 + 44 and 17
    ([600, 128, 129, 300, 17], 256, 320),
]


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("shape", range(len(GEMM_SHAPES)))
def test_grouped_gemm_matches_oracle(dtype, shape):
    counts, d, I = GEMM_SHAPES[shape]
    offsets, xs, wgu, wd = _gemm_case(counts, d, I, dtype, seed=shape)
    off_t = torch.from_numpy(offsets.astype(np.int32)).to(DEV)
    ws = torch.empty(256, dtype=torch.uint8, device=DEV)
    h = moe.moe_gate_up(xs, off_t, wgu, workspace=ws)
    y = moe.moe_down(h, off_t, wd, workspace=ws)
    torch.cuda.synchronize()
    assert moe.moe_read_device_status(ws) == 0
    round_h = dtype == torch.bfloat16
    # reference h from the oracle's FFN pieces, expert by expert
    wgu_e, wd_e = Expertwise(wgu), Expertwise(wd)
    x64 = f64(xs)
    h_ref = np.zeros((xs.shape[0], I))
    for e in range(len(counts)):
        a, b = offsets[e], offsets[e + 1]
        if b > a:
            g = x64[a:b] @ wgu_e[e][:, :I]
            u = x64[a:b] @ wgu_e[e][:, I:]
            h_ref[a:b] = g / (1 + np.exp(-g)) * u
    if round_h:
        h_ref = o.round_bf16(h_ref)
    tol = TOL[dtype]
    if round_h:
        assert within_one_bf16_ulp(f64(h), h_ref)
    else:
        assert err_rms(f64(h), h_ref) <= tol
    y_ref = o.experts(x64, offsets, wgu_e, wd_e, round_h)
    assert err_rms(f64(y), y_ref) <= tol


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("counts", [[100, 200, 1], [900, 700], [1100], [600, 128, 129, 300, 17]])
def test_grouped_gemm_row_scale_and_weight(dtype, counts):
    d, I = 256, 256
    offsets, xs, wgu, wd = _gemm_case(counts, d, I, dtype, seed=9)
    R = xs.shape[0]
    off_t = torch.from_numpy(offsets.astype(np.int32)).to(DEV)
    perm = torch.randperm(R, generator=torch.Generator().manual_seed(0)).to(DEV).int()
    w = (torch.rand(R, generator=torch.Generator().manual_seed(1)) + 0.1).to(DEV)
    h, y = moe.moe_experts(xs, off_t, wgu, wd, sorted_to_slot=perm, topk_weights=w,
                           flags=moe.SCALE_INPUT)
    s = f64(w)[perm.cpu().numpy()]
    round_h = dtype == torch.bfloat16
    y_ref = o.experts(f64(xs), offsets, Expertwise(wgu), Expertwise(wd), round_h, row_scale=s)
    assert err_rms(f64(y), y_ref) <= TOL[dtype]
    h2, y2 = moe.moe_experts(xs, off_t, wgu, wd, sorted_to_slot=perm, topk_weights=w,
                             flags=moe.FUSE_COMBINE_WEIGHT)
    y_ref2 = o.experts(f64(xs), offsets, Expertwise(wgu), Expertwise(wd), round_h) * s[:, None]
    assert err_rms(f64(y2), y_ref2) <= TOL[dtype]


@pytest.mark.parametrize("R,d,I", [(333, 384, 512), (1100, 384, 200), (2049, 512, 640)])
def test_single_group_without_offsets(R, d, I):
    """offsets NULL: one expert owning every row (the always-on shared expert's form). Above 512
    rows both GEMMs run on CTA pairs; the 200-column case leaves a ragged h tile."""
    xs = synth.normal((R, d), torch.bfloat16, 4, "sx", 1.0, device=DEV)
    wgu = synth.normal((1, d, 2 * I), torch.bfloat16, 4, "swgu", 0.05, device=DEV)
    wd = synth.normal((1, I, d), torch.bfloat16, 4, "swd", 0.05, device=DEV)
    h = moe.moe_gate_up(xs, None, wgu)
    y = moe.moe_down(h, None, wd)
    ref = o.swiglu_ffn(f64(xs), f64(wgu[0]), f64(wd[0]), True)
    assert err_rms(f64(y), ref) <= TOL[torch.bfloat16]
    # the same single group through explicit offsets and through packed weights
    off_t = torch.tensor([0, R], dtype=torch.int32, device=DEV)
    h2 = moe.moe_gate_up(xs, off_t, moe.pack_weights(wgu, moe.W_GATE_UP))
    y2 = moe.moe_down(h2, off_t, moe.pack_weights(wd, moe.W_DOWN))
    assert torch.equal(h2, h)
    assert torch.equal(y2, y)


# ------------------------------------------------------------------------------------------------
# whole layer
# ------------------------------------------------------------------------------------------------
def _run_forward(cfg, inp, flags=None):
    flags = (moe.RENORMALIZE if cfg.renormalize else 0) | (moe.SCALE_INPUT if cfg.scale_input
                                                           else 0) if flags is None else flags
    return moe.moe_forward(inp["x"], inp["logits"], inp["w_gate_up"], inp["w_down"], cfg.k,
                           cfg.score_fn, flags, inp["w_shared_gate_up"], inp["w_shared_down"])


def _oracle_forward(cfg, inp):
    sh = inp["w_shared_gate_up"]
    return o.forward(f64(inp["x"]), inp["logits"].cpu().numpy(), Expertwise(inp["w_gate_up"]),
                     Expertwise(inp["w_down"]), cfg.k, cfg.score_fn, cfg.renormalize,
                     cfg.scale_input, cfg.dtype == torch.bfloat16,
                     None if sh is None else f64(sh),
                     None if sh is None else f64(inp["w_shared_down"]))


# T*k <= 1024 runs the fused small-batch router/dispatch; decode at T=128 (1024 slots) and
# T=129 (1032 slots) sit on either side of that boundary.
FORWARD_CASES = [("tiny_fp32", None), ("mixtral_8x7b", 600), ("gpt_oss_120b", 700),
                 ("decode", 1), ("decode", 8), ("decode", 64), ("decode", 128), ("decode", 129),
                 ("llama4_scout", 700)]


@pytest.mark.parametrize("name,T", FORWARD_CASES)
def test_forward_matches_oracle(name, T):
    cfg = _cfg(name, T)
    inp = synth.make_inputs(cfg, DEV)
    out, ids, w, ws = _run_forward(cfg, inp)
    ref = _oracle_forward(cfg, inp)
    assert moe.moe_read_device_status(ws) == 0
    assert np.array_equal(ids.cpu().numpy(), ref["topk_ids"])
    assert (np.abs(w.cpu().numpy() - ref["topk_weights"]) / ref["topk_weights"]).max() <= W_REL_TOL
    v = moe.forward_workspace_views(ws, cfg.T, cfg.d, cfg.E, cfg.k, cfg.I, cfg.I_shared, cfg.dtype)
    assert np.array_equal(v["counts"].cpu().numpy(), ref["counts"])
    assert np.array_equal(v["offsets"].cpu().numpy(), ref["offsets"])
    assert np.array_equal(v["sorted_to_slot"].cpu().numpy(), ref["sorted_to_slot"])
    assert np.array_equal(v["slot_to_sorted"].cpu().numpy(), ref["slot_to_sorted"])
    tol = TOL[cfg.dtype]
    if moe.moe_forward_kernel_count(cfg.T, cfg.k, cfg.I_shared, cfg.dtype) != 1:
        # (the fused decode path folds the combine into the down step: no y_sorted)
        assert err_rms(f64(v["y_sorted"]), ref["y_sorted"]) <= tol
    e = err_rms(f64(out), ref["out"])
    assert e <= tol, e


def test_forward_256_experts_matches_oracle():
    """The largest expert count the ABI takes (256), top-8 over 96 tokens: 768 routed rows, so
    the chain (not the one-kernel decode layer) runs, most experts get 1-6 rows and the down
    projection runs on CTA pairs with one 16-token tile per expert."""
    cfg = dataclasses.replace(synth.CONFIGS["decode"], name="e256", T=96, d=256, E=256, k=8,
                              I=192)
    inp = synth.make_inputs(cfg, DEV)
    out, ids, w, ws = _run_forward(cfg, inp)
    ref = _oracle_forward(cfg, inp)
    assert moe.moe_read_device_status(ws) == 0
    assert np.array_equal(ids.cpu().numpy(), ref["topk_ids"])
    v = moe.forward_workspace_views(ws, cfg.T, cfg.d, cfg.E, cfg.k, cfg.I, cfg.I_shared, cfg.dtype)
    assert np.array_equal(v["offsets"].cpu().numpy(), ref["offsets"])
    assert err_rms(f64(v["y_sorted"]), ref["y_sorted"]) <= TOL[cfg.dtype]
    assert err_rms(f64(out), ref["out"]) <= TOL[cfg.dtype]


@pytest.mark.parametrize("name,T,mem", [("mixtral_8x7b", 600, "pinned"), ("decode", 8, "pinned"),
                                        ("llama4_scout", 300, "pinned"),
                                        ("mixtral_8x7b", 600, "pageable"),
                                        ("decode", 8, "pageable"), ("mixtral_8x7b", 600, "mixed")])
def test_forward_host_equals_forward(name, T, mem):
    """moe_forward_host (host activations) returns exactly what moe_forward returns on the same
    inputs: the chain, the one-kernel decode layer and a shared expert. Page-locked buffers are
    read and written in place by the kernels; pageable ones go through the library's staging
    copies; "mixed" has x page-locked and the logits and out pageable."""
    cfg = _cfg(name, T)
    inp = synth.make_inputs(cfg, DEV)
    flags = (moe.RENORMALIZE if cfg.renormalize else 0) | (moe.SCALE_INPUT if cfg.scale_input
                                                           else 0)
    out, _, _, ws = moe.moe_forward(inp["x"], inp["logits"], inp["w_gate_up"], inp["w_down"],
                                    cfg.k, cfg.score_fn, flags, inp["w_shared_gate_up"],
                                    inp["w_shared_down"])
    xh, lh = inp["x"].cpu(), inp["logits"].cpu()
    outh = torch.empty(cfg.T, cfg.d, dtype=cfg.dtype)
    if mem in ("pinned", "mixed"):
        xh = xh.pin_memory()
    if mem == "pinned":
        lh, outh = lh.pin_memory(), outh.pin_memory()
    outh, hws = moe.moe_forward_host(xh, lh, inp["w_gate_up"], inp["w_down"], cfg.k,
                                     cfg.score_fn, flags, inp["w_shared_gate_up"],
                                     inp["w_shared_down"], out=outh)
    torch.cuda.synchronize()
    assert moe.moe_read_device_status(hws) == 0
    assert torch.equal(outh, out.cpu())


def test_forward_fused_combine_weight_matches():
    cfg = _cfg("gpt_oss_120b", 300)
    inp = synth.make_inputs(cfg, DEV)
    out, _, _, _ = _run_forward(cfg, inp, flags=moe.RENORMALIZE | moe.FUSE_COMBINE_WEIGHT)
    ref = _oracle_forward(cfg, inp)
    assert err_rms(f64(out), ref["out"]) <= TOL[cfg.dtype]


def test_forward_empty_batch_is_noop():
    cfg = _cfg("decode", 1)
    inp = synth.make_inputs(cfg, DEV)
    x = inp["x"][:0]
    out = torch.empty(0, cfg.d, dtype=cfg.dtype, device=DEV)
    moe.moe_forward(x, inp["logits"][:0], inp["w_gate_up"], inp["w_down"], cfg.k, out=out)


def test_forward_all_experts_equal_is_dense_mlp():
    """With one weight set copied to every expert and renormalised weights the layer is a dense
    SwiGLU MLP, whatever the routing."""
    cfg = _cfg("gpt_oss_120b", 256)
    x = synth.make_x(cfg, DEV)
    logits = synth.make_logits(cfg, x, synth.make_router_weight(cfg, DEV))
    w1 = synth.normal((1, cfg.d, 2 * cfg.I), cfg.dtype, 0, "eq_gu", 0.02, device=DEV)
    w2 = synth.normal((1, cfg.I, cfg.d), cfg.dtype, 0, "eq_d", 0.02, device=DEV)
    wgu = w1.expand(cfg.E, -1, -1).contiguous()
    wd = w2.expand(cfg.E, -1, -1).contiguous()
    out, _, _, _ = moe.moe_forward(x, logits, wgu, wd, cfg.k)
    dense = o.swiglu_ffn(f64(x), f64(w1[0]), f64(w2[0]), True)
    assert err_rms(f64(out), dense) <= TOL[cfg.dtype]


def test_forward_in_cuda_graph():
    """The call chain has no host synchronisation, so it can be captured and replayed."""
    cfg = _cfg("decode", 8)
    inp = synth.make_inputs(cfg, DEV)
    out, ids, w, ws = _run_forward(cfg, inp)
    ref = out.clone()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            moe.moe_forward(inp["x"], inp["logits"], inp["w_gate_up"], inp["w_down"], cfg.k,
                            out=out, topk_ids=ids, topk_weights=w, workspace=ws, stream=s)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, ref)


# ------------------------------------------------------------------------------------------------
# packed weights (moe_pack_weights): same results as the pages' layout
# ------------------------------------------------------------------------------------------------
def _ref_pack(w, kind):
    """The packed layout by plain tensor indexing: 64 x 64 blocks (e, nb, k rows, 64 columns),
    gate and up halves blocked separately for gate_up, zero padding."""
    E, K, C = w.shape
    N = C // 2 if kind == moe.W_GATE_UP else C
    kpad = (K + 63) // 64 * 64
    nbh = (N + 63) // 64
    halves = [w[..., :N], w[..., N:]] if kind == moe.W_GATE_UP else [w]
    blocks = []
    for hw in halves:
        padded = torch.zeros(E, kpad, nbh * 64, dtype=w.dtype, device=w.device)
        padded[:, :K, :N] = hw
        blocks.append(padded.view(E, kpad, nbh, 64).permute(0, 2, 1, 3))
    return torch.cat(blocks, dim=1).contiguous()


@pytest.mark.parametrize("E,K,N", [(3, 256, 384), (1, 200, 200), (5, 64, 8), (2, 130, 1000)])
def test_pack_layout(E, K, N):
    for kind in (moe.W_GATE_UP, moe.W_DOWN):
        C = 2 * N if kind == moe.W_GATE_UP else N
        w = synth.normal((E, K, C), torch.bfloat16, E + K, "pk", 1.0, device=DEV)
        pw = moe.pack_weights(w, kind)
        ref = _ref_pack(w, kind)
        assert pw.data.numel() == ref.numel() * 2
        assert torch.equal(pw.data.view(torch.bfloat16), ref.view(-1))


@pytest.mark.parametrize("shape", range(len(GEMM_SHAPES)))
def test_grouped_gemm_packed_weights(shape):
    counts, d, I = GEMM_SHAPES[shape]
    offsets, xs, wgu, wd = _gemm_case(counts, d, I, torch.bfloat16, seed=shape)
    off_t = torch.from_numpy(offsets.astype(np.int32)).to(DEV)
    h_ref = moe.moe_gate_up(xs, off_t, wgu)
    y_ref = moe.moe_down(h_ref, off_t, wd)
    h = moe.moe_gate_up(xs, off_t, moe.pack_weights(wgu, moe.W_GATE_UP))
    y = moe.moe_down(h, off_t, moe.pack_weights(wd, moe.W_DOWN))
    # the packed layout changes only where weights are read from, not the arithmetic
    assert torch.equal(h, h_ref)
    assert torch.equal(y, y_ref)


@pytest.mark.parametrize("name,T", [("gpt_oss_120b", 700), ("decode", 8), ("llama4_scout", 300),
                                    ("mixtral_8x7b", 600)])
def test_forward_packed_weights_matches_oracle(name, T):
    cfg = _cfg(name, T)
    inp = synth.make_inputs(cfg, DEV)
    pk = dict(inp)
    pk["w_gate_up"] = moe.pack_weights(inp["w_gate_up"], moe.W_GATE_UP)
    pk["w_down"] = moe.pack_weights(inp["w_down"], moe.W_DOWN)
    if inp["w_shared_gate_up"] is not None:
        pk["w_shared_gate_up"] = moe.pack_weights(inp["w_shared_gate_up"], moe.W_GATE_UP)
        pk["w_shared_down"] = moe.pack_weights(inp["w_shared_down"], moe.W_DOWN)
    out, ids, _, ws = _run_forward(cfg, pk)
    assert moe.moe_read_device_status(ws) == 0
    ref = _oracle_forward(cfg, inp)
    assert np.array_equal(ids.cpu().numpy(), ref["topk_ids"])
    e = err_rms(f64(out), ref["out"])
    assert e <= TOL[cfg.dtype], e
    out_u, _, _, _ = _run_forward(cfg, inp)
    assert torch.equal(out, out_u)
