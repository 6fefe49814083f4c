"""Parity of the backward pass (moe_forward_train + moe_backward and the single steps, called
through the C ABI) with the CPU backward oracle.

The oracle runs with the same storage points as the layer dtype (bf16 layers: h, the saved
gate/up accumulators, dy and d_ab rounded to bf16; fp32 layers: none), so the remaining
differences are fp32 accumulation and the odd value that lands on the other side of a bf16
rounding midpoint. Bar, as for the forward: max |gpu - ref| <= TOL * rms(ref) per tensor
(2e-2 bf16, 1e-4 fp32). Shapes span several tiles with ragged tails (d, I not multiples of the
64-column K block or the 256-column N tile, experts with a few rows, experts with none), every
router form, the score scaling the input with a shared expert, and packed weights.
"""
import numpy as np
import pytest
import torch

from oracle import moe_backward as B
from oracle import moe_oracle as o
from routing_dispatch_grouped_gb300 import moe, synth
from tests.helpers import TOL, Expertwise, err_rms, f64, within_one_bf16_ulp

pytestmark = pytest.mark.gpu
DEV = "cuda"
bf16, f32 = torch.bfloat16, torch.float32


@pytest.fixture(scope="module", autouse=True)
def _loaded():
    assert torch.cuda.is_available(), "GPU tests need a GPU"
    moe.lib()


def _cfg(name, T, d, E, k, I, dtype, fn=o.SOFTMAX, renorm=True, scale=False, Is=0,
         bias="none"):
    return synth.MoEConfig(name, T, d, E, k, I, dtype, score_fn=fn, renormalize=renorm,
                           scale_input=scale, I_shared=Is, bias=bias)


# (config, packed weights)
CASES = [
    (_cfg("mixtral_like", 200, 512, 8, 2, 640, bf16), False),
    (_cfg("mixtral_like_packed", 200, 512, 8, 2, 640, bf16), True),
    (_cfg("gptoss_like", 150, 264, 16, 4, 200, bf16, bias="normal0.5"), False),
    (_cfg("gptoss_like_packed", 150, 264, 16, 4, 200, bf16, bias="normal0.5"), True),
    (_cfg("scout_like", 160, 256, 4, 1, 384, bf16, o.SIGMOID, False, True, 192, "zipf1.2"),
     False),
    (_cfg("scout_like_packed", 160, 256, 4, 1, 384, bf16, o.SIGMOID, False, True, 192,
          "zipf1.2"), True),
    (_cfg("sigmoid_renorm", 100, 128, 12, 3, 128, bf16, o.SIGMOID, True), False),
    (_cfg("softmax_full", 90, 192, 10, 2, 96, bf16, o.SOFTMAX, False), False),
    (_cfg("empty_experts", 5, 128, 32, 2, 136, bf16), False),
    (_cfg("one_token", 1, 1024, 32, 8, 384, bf16), True),
    (_cfg("tiny_fp32", 64, 128, 8, 2, 256, f32), False),
    (_cfg("fp32_scale_shared", 48, 96, 4, 1, 64, f32, o.SIGMOID, False, True, 40), False),
]


def _flags(cfg):
    return (moe.RENORMALIZE if cfg.renormalize else 0) | (moe.SCALE_INPUT if cfg.scale_input
                                                            else 0)


def _run(cfg, packed):
    inp = synth.make_inputs(cfg, DEV)
    dout = synth.normal((cfg.T, cfg.d), cfg.dtype, 0, "dout_" + cfg.name, 1.0, device=DEV)
    wgu, wd = inp["w_gate_up"], inp["w_down"]
    sgu, sdn = inp["w_shared_gate_up"], inp["w_shared_down"]
    if packed:
        pgu, pd = moe.pack_weights(wgu, moe.W_GATE_UP), moe.pack_weights(wd, moe.W_DOWN)
        psgu = moe.pack_weights(sgu, moe.W_GATE_UP) if sgu is not None else None
        psd = moe.pack_weights(sdn, moe.W_DOWN) if sdn is not None else None
    else:
        pgu, pd, psgu, psd = wgu, wd, sgu, sdn
    out, ids, w, ws = moe.moe_forward_train(inp["x"], inp["logits"], pgu, pd, cfg.k,
                                            cfg.score_fn, _flags(cfg), psgu, psd)
    g = moe.moe_backward(dout, inp["x"], inp["logits"], pgu, pd, cfg.k, ids, w, ws, cfg.score_fn,
                         _flags(cfg), psgu, psd, want_logits=True)
    torch.cuda.synchronize()
    assert moe.moe_read_device_status(ws) == 0
    return inp, dout, out, ids, w, ws, g


def _oracle(cfg, inp, dout):
    lowp = cfg.dtype == bf16
    sh = {}
    if cfg.I_shared:
        sh = dict(w_shared_gate_up=f64(inp["w_shared_gate_up"]),
                  w_shared_down=f64(inp["w_shared_down"]))
    x64, lg = f64(inp["x"]), inp["logits"].cpu().numpy()
    wgu, wd = Expertwise(inp["w_gate_up"]), Expertwise(inp["w_down"])
    f = B.forward_train(x64, lg, wgu, wd, cfg.k, cfg.score_fn, cfg.renormalize, cfg.scale_input,
                        round_h=lowp, bf16_points=lowp, **sh)
    ref = B.backward(f, f64(dout), x64, lg, wgu, wd, cfg.k, cfg.score_fn, cfg.renormalize,
                     cfg.scale_input, bf16_points=lowp, **sh)
    return f, ref


def _fp32_sum_ok(got, a, b, slack=2):
    """got vs a @ b (float64 of the same inputs): an fp32 sum of n products in any order is
    within (n + 1) 2^-24 sum |a b| (slack 2 for the tensor core's internal alignment)."""
    ref = a @ b
    bound = slack * (a.shape[-1] + 1) * 2.0 ** -24 * (np.abs(a) @ np.abs(b))
    return bool(np.all(np.abs(got - ref) <= bound + 1e-30))


@pytest.mark.parametrize("cfg,packed", CASES, ids=[c[0].name for c in CASES])
def test_backward_matches_oracle(cfg, packed):
    inp, dout, out, ids, w, ws, g = _run(cfg, packed)
    f, ref = _oracle(cfg, inp, dout)
    assert np.array_equal(ids.cpu().numpy(), f["topk_ids"])
    tol = TOL[cfg.dtype]
    lowp = cfg.dtype == bf16
    # each step on the GPU's own inputs: the bf16 stores within one ulp of the oracle's, each
    # GEMM within the fp32 summation bound of its own operands
    fv = moe.forward_train_workspace_views(ws, cfg.T, cfg.d, cfg.E, cfg.k, cfg.I, cfg.I_shared,
                                           cfg.dtype)
    bv = moe.backward_workspace_views(g["workspace"], cfg.T, cfg.d, cfg.k, cfg.I, cfg.dtype)
    dy, d_ab, dxs = f64(bv["dy_sorted"]), f64(bv["d_ab"]), f64(bv["dx_sorted"])
    ab = f64(fv["ab"])
    if lowp:  # the GPU's fp32 weight and the oracle's fp64 one may round dy apart by an ulp
        assert within_one_bf16_ulp(dy, ref["dy_sorted"], rms_frac=0.0)
    else:
        assert err_rms(dy, ref["dy_sorted"]) <= 1e-6
    off = f["offsets"]
    xs, h = f64(fv["x_sorted"]), f64(fv["h"])
    wgu, wd = inp["w_gate_up"], inp["w_down"]
    dwgu, dwd = f64(g["d_w_gate_up"]), f64(g["d_w_down"])
    s_rows = f64(w).reshape(-1)[f["sorted_to_slot"]] if cfg.scale_input else np.ones(len(dy))
    for e in range(cfg.E):
        lo, hi = int(off[e]), int(off[e + 1])
        if hi == lo:
            assert not dwgu[e].any() and not dwd[e].any()
            continue
        # SwiGLU backward of the GPU's own dh and saved accumulators
        dh = dy[lo:hi] @ f64(wd[e]).T
        stage, _ = B.swiglu_backward(dh, ab[lo:hi], s_rows[lo:hi], bf16_points=lowp)
        if lowp:
            assert within_one_bf16_ulp(d_ab[lo:hi], stage, rms_frac=1e-4), e
        else:
            assert err_rms(d_ab[lo:hi], stage) <= 1e-5, e
        assert _fp32_sum_ok(dwd[e], h[lo:hi].T, dy[lo:hi]), e
        assert _fp32_sum_ok(dwgu[e], xs[lo:hi].T, d_ab[lo:hi]), e
        assert _fp32_sum_ok(dxs[lo:hi], d_ab[lo:hi], f64(wgu[e]).T), e
    # end to end against the oracle: the bar of the forward, for the tensors that sum over
    # many rows (a weight gradient of an expert with a handful of rows is an outer product of
    # bf16-rounded values, checked step by step above)
    names = ["dx", "d_topk_weights", "d_logits"]
    if np.min(np.diff(off)[np.diff(off) > 0]) >= 16:
        names += ["d_w_gate_up", "d_w_down"]
    if cfg.I_shared:
        names += ["d_w_shared_gate_up", "d_w_shared_down"]
    for name in names:
        e = err_rms(f64(g[name]), ref[name])
        assert e <= tol, (name, e)
    # the saved accumulators are the forward's, unscaled: within a bf16 ulp of the oracle's
    v = moe.forward_train_workspace_views(ws, cfg.T, cfg.d, cfg.E, cfg.k, cfg.I, cfg.I_shared,
                                          cfg.dtype)
    if cfg.dtype == bf16:
        assert within_one_bf16_ulp(f64(v["ab"]), f["ab"])
    else:
        assert err_rms(f64(v["ab"]), f["ab"]) <= 1e-5


def test_backward_is_deterministic():
    cfg = CASES[2][0]
    a = _run(cfg, False)[-1]
    b = _run(cfg, False)[-1]
    for name in ("dx", "d_w_gate_up", "d_w_down", "d_topk_weights", "d_logits"):
        assert torch.equal(a[name], b[name]), name


@pytest.mark.parametrize("dtype", [bf16, f32])
def test_weight_grad_ragged_and_empty_experts(dtype):
    # rows per expert: empty, 1, 63, 64, 65, 130, empty, 200
    counts = [0, 1, 63, 64, 65, 130, 0, 200]
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    R, M, N = int(off[-1]), 136, 264
    a = synth.normal((R, M), dtype, 0, "wg_a", 1.0, device=DEV)
    b = synth.normal((R, N), dtype, 0, "wg_b", 1.0, device=DEV)
    dw = moe.moe_weight_grad(a, b, torch.from_numpy(off).to(DEV), len(counts))
    torch.cuda.synchronize()
    A, Bm = f64(a), f64(b)
    got = f64(dw)
    for e in range(len(counts)):
        lo, hi = off[e], off[e + 1]
        ref = A[lo:hi].T @ Bm[lo:hi]
        if hi == lo:
            assert np.all(got[e] == 0.0)
            continue
        # an fp32 sum of n products in any order: error <= (n + 1) 2^-24 sum |a b| (fp32
        # products round too); twice that for the tensor core's internal alignment
        bound = 2 * (hi - lo + 1) * 2.0 ** -24 * (np.abs(A[lo:hi]).T @ np.abs(Bm[lo:hi]))
        assert np.all(np.abs(got[e] - ref) <= bound + 1e-30), e


@pytest.mark.parametrize("M,N", [(136, 264), (64, 200), (256, 512)])
def test_weight_grad_bf16_is_the_fp32_gradient_rounded_once(M, N):
    """moe_weight_grad_bf16 rounds the same fp32 accumulators moe_weight_grad stores: bit for bit
    the fp32 result rounded to nearest even, with ragged and empty experts and column tails that
    end inside a 64-column store tile (N = 200, 264)."""
    counts = [0, 1, 63, 64, 65, 130, 0, 200]
    off = torch.from_numpy(np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)).to(DEV)
    R = int(off[-1])
    a = synth.normal((R, M), bf16, 0, "wgb_a", 1.0, device=DEV)
    b = synth.normal((R, N), bf16, 0, "wgb_b", 1.0, device=DEV)
    dw32 = moe.moe_weight_grad(a, b, off, len(counts))
    dw16 = torch.full((len(counts), M, N), 3.0, dtype=bf16, device=DEV)  # every element written
    moe.moe_weight_grad(a, b, off, len(counts), dw=dw16)
    torch.cuda.synchronize()
    assert torch.equal(dw16, dw32.to(bf16))
    assert torch.count_nonzero(dw16[0]).item() == 0 and torch.count_nonzero(dw16[6]).item() == 0


@pytest.mark.parametrize("idx", [0, 2, 4])
def test_backward_bf16_weight_gradients(idx):
    """moe_backward with WGRAD_BF16: the weight gradients are the fp32 run's rounded once, and
    every other output is unchanged."""
    cfg, _ = CASES[idx]
    if cfg.dtype != bf16:
        pytest.skip("bf16 layers only")
    inp, dout, out, ids, w, ws, g = _run(cfg, False)
    sgu, sdn = inp["w_shared_gate_up"], inp["w_shared_down"]
    g16 = moe.moe_backward(dout, inp["x"], inp["logits"], inp["w_gate_up"], inp["w_down"], cfg.k,
                           ids, w, ws, cfg.score_fn, _flags(cfg) | moe.WGRAD_BF16, sgu, sdn,
                           want_logits=True)
    torch.cuda.synchronize()
    names = ["d_w_gate_up", "d_w_down"] + (["d_w_shared_gate_up", "d_w_shared_down"]
                                           if cfg.I_shared else [])
    for n in names:
        assert g16[n].dtype == bf16 and torch.equal(g16[n], g[n].to(bf16)), n
    for n in ("dx", "d_topk_weights", "d_logits"):
        assert torch.equal(g16[n], g[n]), n


def test_weight_grad_without_rows_writes_zeros():
    off = torch.zeros(5, dtype=torch.int32, device=DEV)
    a = torch.empty(0, 64, dtype=bf16, device=DEV)
    dw = torch.full((4, 64, 64), 7.0, device=DEV)
    moe.moe_weight_grad(a, a, off, 4, dw=dw)
    torch.cuda.synchronize()
    assert torch.count_nonzero(dw).item() == 0


@pytest.mark.parametrize("fn,renorm", [(o.SOFTMAX, True), (o.SOFTMAX, False),
                                       (o.SIGMOID, True), (o.SIGMOID, False)])
def test_route_backward_matches_oracle(fn, renorm):
    rng = np.random.default_rng(7)
    T, E, k = 300, 64, 6
    z = (rng.standard_normal((T, E)) * 1.5).astype(np.float32)
    lg = torch.from_numpy(z).to(DEV)
    ids, w = moe.moe_route(lg, k, fn, renorm)
    dw = torch.from_numpy(rng.standard_normal((T, k)).astype(np.float32)).to(DEV)
    dl = moe.moe_route_backward(lg, ids, w, dw, fn, renorm)
    torch.cuda.synchronize()
    ref = B.route_backward(z, ids.cpu().numpy(), f64(dw), fn, renorm)
    # fp32 weights, exp and sums: a few ulp of the largest term
    assert np.max(np.abs(f64(dl) - ref)) <= 1e-5 * (1 + np.max(np.abs(ref)))


@pytest.mark.parametrize("dtype", [bf16, f32])
def test_combine_backward_matches_oracle(dtype):
    T, d, E, k = 77, 264, 8, 3
    rng = np.random.default_rng(9)
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    _, _, s2p, p2s = o.dispatch(ids, E)
    R = T * k
    y = synth.normal((R, d), f32, 0, "cb_y", 1.0, device=DEV)
    w = torch.from_numpy(rng.uniform(0.1, 1.0, (T, k)).astype(np.float32)).to(DEV)
    dout = synth.normal((T, d), dtype, 0, "cb_dout", 1.0, device=DEV)
    p2s_t = torch.from_numpy(p2s.astype(np.int32)).to(DEV)
    dy, dw = moe.moe_combine_backward(dout, p2s_t, k, topk_weights=w, y_sorted=y)
    torch.cuda.synchronize()
    D, Y, W = f64(dout), f64(y), f64(w)
    ref_dy = np.zeros((R, d))
    ref_dw = np.zeros((T, k))
    for t in range(T):
        for j in range(k):
            p = p2s[t * k + j]
            ref_dy[p] = W[t, j] * D[t]
            ref_dw[t, j] = D[t] @ Y[p]
    got = f64(dy)
    if dtype == bf16:  # the fp32 product rounded again to bf16: half a bf16 ulp plus fp32's
        assert np.all(np.abs(got - ref_dy) <= (2.0 ** -8 + 2.0 ** -23) * np.abs(ref_dy))
    else:
        assert np.all(np.abs(got - ref_dy) <= 2.0 ** -23 * np.abs(ref_dy))
    yk = Y[p2s.reshape(T, k)]  # [T, k, d]: the row each slot reads
    bound = (d + 2) * 2.0 ** -24 * (np.abs(D)[:, None, :] * np.abs(yk)).sum(-1)
    assert np.all(np.abs(f64(dw) - ref_dw) <= bound + 1e-30)


def test_backward_chain_replays_in_a_graph():
    cfg = CASES[0][0]
    inp = synth.make_inputs(cfg, DEV)
    dout = synth.normal((cfg.T, cfg.d), cfg.dtype, 0, "dout_graph", 1.0, device=DEV)
    args = (inp["x"], inp["logits"], inp["w_gate_up"], inp["w_down"], cfg.k, cfg.score_fn,
            _flags(cfg))
    out, ids, w, ws = moe.moe_forward_train(*args)
    g0 = moe.moe_backward(dout, inp["x"], inp["logits"], inp["w_gate_up"], inp["w_down"], cfg.k,
                          ids, w, ws, cfg.score_fn, _flags(cfg))
    torch.cuda.synchronize()
    ref = {k_: v.clone() for k_, v in g0.items() if v is not None and k_ != "workspace"}
    bws = torch.empty(moe.moe_backward_workspace_size(cfg.T, cfg.d, cfg.E, cfg.k, cfg.I, 0,
                                                      cfg.dtype), dtype=torch.uint8, device=DEV)
    graph = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        moe.moe_forward_train(*args, out=out, topk_ids=ids, topk_weights=w, workspace=ws)
        moe.moe_backward(dout, inp["x"], inp["logits"], inp["w_gate_up"], inp["w_down"], cfg.k,
                         ids, w, ws, cfg.score_fn, _flags(cfg), out=g0, workspace=bws)
        torch.cuda.current_stream().synchronize()
        with torch.cuda.graph(graph, stream=s):
            moe.moe_forward_train(*args, out=out, topk_ids=ids, topk_weights=w, workspace=ws)
            moe.moe_backward(dout, inp["x"], inp["logits"], inp["w_gate_up"], inp["w_down"],
                             cfg.k, ids, w, ws, cfg.score_fn, _flags(cfg), out=g0, workspace=bws)
    torch.cuda.current_stream().wait_stream(s)
    for name in ref:
        g0[name].zero_()
    graph.replay()
    torch.cuda.synchronize()
    for name, v in ref.items():
        assert torch.equal(g0[name], v), name
