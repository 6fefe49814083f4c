"""Full-size parity of the backward pass in the configuration the benchmark times (packed
weights, moe_forward_train then moe_backward), on samples the oracle computes one by one.

Every step is checked on the GPU's own inputs to it:
- for a sample of routed rows (heaviest and lightest experts included): the saved
  accumulators a, b against x_sorted W_gate_up (one bf16 ulp); dy = w dout (one ulp); d_ab
  against the oracle's SwiGLU backward of dy W_down^T and the saved a, b (one ulp); dx_sorted
  against d_ab W_gate_up^T (fp32 summation bound); the routing-weight gradient against
  dout . y_sorted (fp32 bound);
- for sampled entries of three experts' weight gradients: the sums over the expert's rows of
  x_sorted^T d_ab and h^T dy (fp32 bound);
- for sampled tokens: dx against the sum of their slots' dx_sorted rows (+ the shared
  expert's, itself checked the same way), rounded once;
- over every token: the logit gradient against the oracle's router backward of the GPU's
  routing-weight gradient.
"""
import numpy as np
import pytest
import torch

from oracle import moe_backward as B
from routing_dispatch_grouped_gb300 import moe, synth
from tests.helpers import f64, within_one_bf16_ulp

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _flags(cfg):
    return (moe.RENORMALIZE if cfg.renormalize else 0) | (moe.SCALE_INPUT if cfg.scale_input
                                                            else 0)


def _fp32_ok(got, terms_abs_sum, ref, n, slack=2):
    return bool(np.all(np.abs(got - ref) <= slack * (n + 1) * 2.0 ** -24 * terms_abs_sum + 1e-30))


@pytest.mark.parametrize("name", ["mixtral_8x7b", "gpt_oss_120b", "llama4_scout"])
def test_backward_full_size(name):
    cfg = synth.CONFIGS[name]
    T, d, E, k, I, Is = cfg.T, cfg.d, cfg.E, cfg.k, cfg.I, cfg.I_shared
    inp = synth.make_inputs(cfg, DEV)
    pk = {n: moe.pack_weights(inp[n], moe.W_GATE_UP if "gate_up" in n else moe.W_DOWN)
          if inp[n] is not None else None
          for n in ("w_gate_up", "w_down", "w_shared_gate_up", "w_shared_down")}
    dout = synth.normal((T, d), cfg.dtype, 0, "dout_full", 1.0, device=DEV)
    out, ids, w, ws = moe.moe_forward_train(inp["x"], inp["logits"], pk["w_gate_up"],
                                            pk["w_down"], k, cfg.score_fn, _flags(cfg),
                                            pk["w_shared_gate_up"], pk["w_shared_down"])
    g = moe.moe_backward(dout, inp["x"], inp["logits"], pk["w_gate_up"], pk["w_down"], k, ids, w,
                         ws, cfg.score_fn, _flags(cfg), pk["w_shared_gate_up"],
                         pk["w_shared_down"])
    torch.cuda.synchronize()
    del pk
    assert moe.moe_read_device_status(ws) == 0
    assert moe.moe_read_device_status(g["workspace"]) == 0
    fv = moe.forward_train_workspace_views(ws, T, d, E, k, I, Is, cfg.dtype)
    bv = moe.backward_workspace_views(g["workspace"], T, d, k, I, cfg.dtype)
    ids_np = ids.cpu().numpy()
    off = fv["offsets"].cpu().numpy()
    s2p = fv["sorted_to_slot"].cpu().numpy()
    p2s = fv["slot_to_sorted"].cpu().numpy()
    w64 = f64(w)
    counts = np.diff(off)

    # --- routed rows of a token sample, heaviest and lightest experts included ---
    rng = np.random.default_rng(0)
    toks = set(rng.choice(T, size=12, replace=False).tolist()) | {0, T - 1}
    for e in (int(np.argmax(counts)), int(np.argmin(np.where(counts > 0, counts, 1 << 30)))):
        toks |= set(np.nonzero((ids_np == e).any(axis=1))[0][:2].tolist())
    toks = sorted(toks)
    rows = sorted(int(p2s[t * k + j]) for t in toks for j in range(k))
    row_t = torch.tensor(rows, device=DEV)
    xs = f64(fv["x_sorted"][row_t])
    ab = f64(fv["ab"][row_t])
    h = f64(fv["h"][row_t])
    y = f64(fv["y_sorted"][row_t])
    dy = f64(bv["dy_sorted"][row_t])
    dab = f64(bv["d_ab"][row_t])
    dxs = f64(bv["dx_sorted"][row_t])
    dout64 = f64(dout)
    dtw = f64(g["d_topk_weights"])
    by_e = {}
    for i, p in enumerate(rows):
        e = int(np.searchsorted(off, p, side="right") - 1)
        by_e.setdefault(e, []).append(i)
    for e, idx in by_e.items():
        wgu = f64(inp["w_gate_up"][e])
        wd = f64(inp["w_down"][e])
        slots = s2p[[rows[i] for i in idx]]
        tt, jj = slots // k, slots % k
        s = w64[tt, jj] if cfg.scale_input else np.ones(len(idx))
        # saved accumulators: x_sorted W_gate_up, rounded once
        assert within_one_bf16_ulp(ab[idx], xs[idx] @ wgu, rms_frac=1e-4), e
        # dy = w dout (dout itself when the score scaled the input)
        ref_dy = dout64[tt] * (1.0 if cfg.scale_input else w64[tt, jj][:, None])
        assert within_one_bf16_ulp(dy[idx], ref_dy, rms_frac=0.0), e
        # d_ab: the oracle's SwiGLU backward of the GPU's dh inputs
        ref_dab, ref_ds = B.swiglu_backward(dy[idx] @ wd.T, ab[idx], s, bf16_points=True)
        assert within_one_bf16_ulp(dab[idx], ref_dab, rms_frac=1e-4), e
        # dx_sorted = d_ab W_gate_up^T (fp32 sum over 2I)
        assert _fp32_ok(dxs[idx], np.abs(dab[idx]) @ np.abs(wgu).T, dab[idx] @ wgu.T, 2 * I), e
        if cfg.scale_input:  # the score's gradient: sum_c dg a + du b, fp32 over I
            dg_a = np.abs(ref_dab[:, :I] / s[:, None] * ab[idx][:, :I])
            du_b = np.abs(ref_dab[:, I:] / s[:, None] * ab[idx][:, I:])
            absum = (dg_a + du_b).sum(axis=1)
            # fp32 sum over 2I terms, and dg, du formed in fp32 (a few ulp each)
            assert _fp32_ok(dtw[tt, jj], absum, ref_ds, 2 * I, slack=4), e
        else:  # d w = dout . y_sorted (fp32 over d)
            ref = np.einsum("ic,ic->i", dout64[tt], y[idx])
            assert _fp32_ok(dtw[tt, jj], np.einsum("ic,ic->i", np.abs(dout64[tt]), np.abs(y[idx])),
                            ref, d), e

    # --- weight gradients: sampled entries of three experts, summed over all their rows ---
    for e in sorted({int(np.argmax(counts)), int(np.argmin(np.where(counts > 0, counts, 1 << 30))),
                     int(rng.integers(0, E))}):
        lo, hi = int(off[e]), int(off[e + 1])
        if hi == lo:
            assert not g["d_w_gate_up"][e].any().item() and not g["d_w_down"][e].any().item()
            continue
        for dw, A, Bt, M, N in ((g["d_w_gate_up"], fv["x_sorted"], bv["d_ab"], d, 2 * I),
                                (g["d_w_down"], fv["h"], bv["dy_sorted"], I, d)):
            m = torch.tensor(rng.integers(0, M, 64), device=DEV)
            n = torch.tensor(rng.integers(0, N, 64), device=DEV)
            a_s, b_s = f64(A[lo:hi][:, m]), f64(Bt[lo:hi][:, n])  # [rows, 64] each
            ref = np.einsum("rs,rs->s", a_s, b_s)
            absum = np.einsum("rs,rs->s", np.abs(a_s), np.abs(b_s))
            assert _fp32_ok(f64(dw[e][m, n]), absum, ref, hi - lo), e

    # --- dx of the sampled tokens: the sum of their slots' dx_sorted (+ the shared expert) ---
    tok_t = torch.tensor(toks, device=DEV)
    at = {p: i for i, p in enumerate(rows)}  # sampled rows' dx_sorted, from the GPU
    ref_dx = np.zeros((len(toks), d))
    for i, t in enumerate(toks):
        for j in range(k):
            ref_dx[i] += dxs[at[int(p2s[t * k + j])]]
    if Is:
        # shared expert: d_ab_s from the oracle's SwiGLU backward of dout W_sd^T and the saved
        # accumulators, then dx_s = d_ab_s W_sgu^T (compared after the sum, within its bound)
        wsgu, wsd = f64(inp["w_shared_gate_up"]), f64(inp["w_shared_down"])
        abs_ = f64(fv["ab_shared"][tok_t])
        assert within_one_bf16_ulp(abs_, f64(inp["x"][tok_t]) @ wsgu, rms_frac=1e-4)
        dabs, _ = B.swiglu_backward(dout64[toks] @ wsd.T, abs_, np.ones(len(toks)),
                                    bf16_points=True)
        ref_dx = ref_dx + dabs @ wsgu.T
    got = f64(g["dx"][tok_t])
    rms = np.sqrt(np.mean(ref_dx ** 2))
    # one bf16 rounding of the fp32 sum, plus (shared expert) d_ab_s values that land on the
    # other side of a rounding midpoint
    assert np.all(np.abs(got - ref_dx) <= 2.0 ** -8 * np.abs(ref_dx) + 2e-3 * rms)

    # --- logits: the oracle's router backward of the GPU's routing-weight gradient ---
    ref_dl = B.route_backward(inp["logits"].cpu().numpy(), ids_np, dtw, cfg.score_fn,
                              cfg.renormalize)
    got_dl = f64(g["d_logits"])
    assert np.max(np.abs(got_dl - ref_dl)) <= 1e-5 * (1 + np.max(np.abs(ref_dl)))
