"""Pins for the CPU oracle: each check compares it with something other than itself (hand-derived
values, brute force in plain Python, closed forms, invariants, or a library routine)."""
import json
import math
import os
import random
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import moe_oracle as o

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_cases.json")


def _val(v):
    if isinstance(v, str):
        return {"nan": math.nan, "inf": math.inf, "-inf": -math.inf, "-0": -0.0,
                "ln3": float(np.float32(math.log(3.0)))}[v]
    return float(v)


def _golden():
    with open(GOLDEN) as f:
        return json.load(f)


# ----------------------------------------------------------------------------------------------
# bf16 rounding
# ----------------------------------------------------------------------------------------------
def test_round_bf16_matches_torch_on_fp32_values():
    """fp32 -> bf16 through torch (a library conversion, round to nearest even) agrees with the
    oracle's definition on every fp32 input, including exact ties and subnormals."""
    rng = np.random.default_rng(0)
    a = rng.standard_normal(200_000) * np.exp2(rng.integers(-140, 120, 200_000))
    a = a.astype(np.float32)
    bits = rng.integers(0, 1 << 16, 50_000, dtype=np.uint32)
    ties = ((rng.integers(0, 1 << 15, 50_000, dtype=np.uint32) << 16) | 0x8000).view(np.float32)
    mixed = ((rng.integers(0x0080, 0x7F00, 50_000, dtype=np.uint32) << 16) | bits).view(np.float32)
    a = np.concatenate([a, ties, mixed, np.float32([0.0, -0.0, 1e-45, -1e-45, 3.4e38])])
    a = a[np.isfinite(a)]
    ref = torch.from_numpy(a).to(torch.bfloat16).double().numpy()
    got = o.round_bf16(a.astype(np.float64))
    assert np.array_equal(got, ref)


def _bf16_nearest_exact(v: float) -> float:
    """Brute force in exact rationals: the two bf16 neighbours of v and the nearer one (ties to
    the even significand)."""
    if v == 0:
        return v
    f = Fraction(v)
    m, e = math.frexp(abs(v))
    q = Fraction(2) ** max(e - 8, -133)
    lo = (abs(f) // q) * q
    hi = lo + q
    dlo, dhi = abs(f) - lo, hi - abs(f)
    if dlo < dhi:
        r = lo
    elif dhi < dlo:
        r = hi
    else:
        r = lo if (lo / q) % 2 == 0 else hi
    return math.copysign(float(r), v)


def test_round_bf16_exact_on_fp64_values():
    rng = random.Random(1)
    vals = [rng.gauss(0, 1) * 2.0 ** rng.randint(-130, 100) for _ in range(5000)]
    # values exactly half-way between bf16 neighbours in fp64, and just off them
    for s in range(200):
        base = float(np.float32(rng.uniform(1, 2)))
        q = 2.0 ** -7
        mid = (math.floor(base / q) + 0.5) * q
        vals += [mid, mid + 2 ** -40, mid - 2 ** -40]
    got = o.round_bf16(np.array(vals))
    ref = np.array([_bf16_nearest_exact(v) for v in vals])
    assert np.array_equal(got, ref)


# ----------------------------------------------------------------------------------------------
# Route
# ----------------------------------------------------------------------------------------------
@pytest.mark.parametrize("case", range(len(_golden()["route"])))
def test_route_hand_cases(case):
    c = _golden()["route"][case]
    logits = np.array([[_val(v) for v in c["logits"]]], dtype=np.float32)
    fn = o.SOFTMAX if c["score"] == "softmax" else o.SIGMOID
    ids, w = o.route(logits, c["k"], fn, c["renormalize"])
    assert ids[0].tolist() == c["ids"]
    if c["weights"] is not None:
        assert np.max(np.abs(w[0] - np.array(c["weights"]))) <= c["tol"]


def _brute_topk(row, k):
    """Plain-Python ranking: NaN last, larger value first, lower index first."""
    keyed = [((1 if math.isnan(v) else 0), (0.0 if math.isnan(v) else -v), i)
             for i, v in enumerate(row)]
    return [i for _, _, i in sorted(keyed)[:k]]


@pytest.mark.parametrize("E,k", [(8, 2), (16, 1), (128, 4), (128, 8), (5, 5), (256, 8)])
def test_route_ids_match_brute_force_with_ties(E, k):
    rng = np.random.default_rng(E * 31 + k)
    # few distinct values -> many ties; sprinkle -inf, -0.0 and NaN
    z = rng.integers(-3, 4, size=(64, E)).astype(np.float32) * np.float32(0.5)
    z[rng.random(z.shape) < 0.05] = -np.inf
    z[rng.random(z.shape) < 0.05] = -0.0
    z[rng.random(z.shape) < 0.02] = np.nan
    ids, _ = o.route(z, k)
    for t in range(z.shape[0]):
        assert ids[t].tolist() == _brute_topk([float(v) for v in z[t]], k)


@pytest.mark.parametrize("E,k", [(8, 2), (128, 4), (128, 8), (16, 1)])
def test_route_softmax_renorm_identity(E, k):
    """Softmax over all E then renormalised over the top k equals a softmax over the k selected
    logits alone (the closed-form identity behind the two wordings of the router)."""
    rng = np.random.default_rng(7)
    z = (rng.standard_normal((200, E)) * 1.5).astype(np.float32)
    ids, w = o.route(z, k, o.SOFTMAX, True)
    for t in range(z.shape[0]):
        sel = [float(z[t, i]) for i in ids[t]]
        ex = [math.exp(v - sel[0]) for v in sel]
        ref = [v / sum(ex) for v in ex]
        assert np.max(np.abs(w[t] - ref)) <= 1e-12
    assert np.max(np.abs(w.sum(1) - 1.0)) <= 1e-15 * 4
    assert all(len(set(r.tolist())) == k for r in ids)
    # weights follow slot order (slot 0 = best)
    assert np.all(np.diff(w, axis=1) <= 0)


def test_route_softmax_without_renorm_is_full_softmax():
    rng = np.random.default_rng(3)
    z = rng.standard_normal((50, 16)).astype(np.float32)
    ids, w = o.route(z, 4, o.SOFTMAX, False)
    for t in range(50):
        ex = [math.exp(float(v)) for v in z[t]]
        for j in range(4):
            assert abs(w[t, j] - ex[ids[t, j]] / sum(ex)) <= 1e-13


def test_route_sigmoid_closed_form():
    rng = np.random.default_rng(4)
    z = rng.standard_normal((50, 16)).astype(np.float32) * 3
    ids, w = o.route(z, 2, o.SIGMOID, False)
    for t in range(50):
        for j in range(2):
            v = float(z[t, ids[t, j]])
            assert abs(w[t, j] - 1.0 / (1.0 + math.exp(-v))) <= 1e-15
    _, wr = o.route(z, 2, o.SIGMOID, True)
    assert np.allclose(wr.sum(1), 1.0, atol=1e-15, rtol=0)


# ----------------------------------------------------------------------------------------------
# Dispatch
# ----------------------------------------------------------------------------------------------
@pytest.mark.parametrize("case", range(len(_golden()["dispatch"])))
def test_dispatch_hand_cases(case):
    c = _golden()["dispatch"][case]
    counts, offsets, s2p, p2s = o.dispatch(np.array(c["ids"]), c["E"])
    assert counts.tolist() == c["counts"]
    assert offsets.tolist() == c["offsets"]
    assert s2p.tolist() == c["sorted_to_slot"]
    assert p2s.tolist() == c["slot_to_sorted"]


@pytest.mark.parametrize("T,E,k", [(37, 8, 2), (64, 128, 8), (1, 128, 8), (100, 5, 1), (0, 4, 2)])
def test_dispatch_invariants_and_brute_force(T, E, k):
    rng = np.random.default_rng(T + E + k)
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]) if T else np.zeros((0, k), int)
    counts, offsets, s2p, p2s = o.dispatch(ids, E)
    R = T * k
    assert counts.sum() == R
    assert offsets[0] == 0 and offsets[-1] == R and np.all(np.diff(offsets) >= 0)
    assert np.array_equal(p2s[s2p], np.arange(R)) and np.array_equal(s2p[p2s], np.arange(R))
    # O(R * E) stable scan in plain Python
    flat = ids.reshape(-1).tolist()
    ref = [s for e in range(E) for s in range(R) if flat[s] == e]
    assert s2p.tolist() == ref
    for e in range(E):
        assert all(flat[s] == e for s in s2p[offsets[e]:offsets[e + 1]])


def test_permute_rows():
    x = np.arange(12.0).reshape(4, 3)
    ids = np.array([[1, 0], [0, 1], [1, 0], [0, 1]])
    _, _, s2p, _ = o.dispatch(ids, 2)
    xs = o.permute_rows(x, s2p, 2)
    assert xs.tolist() == [x[0].tolist(), x[1].tolist(), x[2].tolist(), x[3].tolist(),
                           x[0].tolist(), x[1].tolist(), x[2].tolist(), x[3].tolist()]


# ----------------------------------------------------------------------------------------------
# Experts
# ----------------------------------------------------------------------------------------------
def test_ffn_hand_case():
    c = _golden()["ffn"]
    for round_h in (False, True):
        y = o.swiglu_ffn(np.array([c["x"]], float), np.array(c["w_gate_up"], float),
                         np.array(c["w_down"], float), round_h)
        assert np.max(np.abs(y[0] - np.array(c["y"]))) <= c["tol"]


def test_activation_hand_case():
    """The activation alone on the same hand case: gate = [40, -50, 50], up = [5, 13, 1], so
    h = [200, SiLU(-50) * 13 (about -2.5e-20), 50] (the fixture's derivation)."""
    c = _golden()["ffn"]
    x, wgu = np.array([c["x"]], float), np.array(c["w_gate_up"], float)
    for round_h in (False, True):
        h = o.swiglu_activation(x, wgu, round_h)
        assert h.shape == (1, 3)
        assert h[0, 0] == 200.0 and h[0, 2] == 50.0
        assert -1e-18 < h[0, 1] < 0
    # experts() hands back the same activation, row by row, for rows split over two experts
    offsets = np.array([0, 1, 2])
    xs = np.array([c["x"], [0.5, -1.0]], float)
    y, h = o.experts(xs, offsets, [wgu, wgu * 0.5], [np.array(c["w_down"], float)] * 2, False,
                     return_h=True)
    assert np.array_equal(h[0], o.swiglu_activation(xs[:1], wgu, False)[0])
    assert np.array_equal(h[1], o.swiglu_activation(xs[1:], wgu * 0.5, False)[0])
    assert np.max(np.abs(y[0] - np.array(c["y"]))) <= c["tol"]


def _dense_swiglu_loops(x, wgu, wd):
    """Textbook dense SwiGLU MLP as plain triple loops."""
    n, d = len(x), len(x[0])
    I = len(wgu[0]) // 2
    out = []
    for r in range(n):
        h = []
        for c in range(I):
            g = sum(x[r][i] * wgu[i][c] for i in range(d))
            u = sum(x[r][i] * wgu[i][I + c] for i in range(d))
            h.append(g / (1.0 + math.exp(-g)) * u)
        out.append([sum(h[c] * wd[c][j] for c in range(I)) for j in range(len(wd[0]))])
    return np.array(out)


def test_ffn_matches_dense_loops_nonsquare():
    rng = np.random.default_rng(11)
    x = rng.standard_normal((5, 3))
    wgu = rng.standard_normal((3, 14))
    wd = rng.standard_normal((7, 3))
    ref = _dense_swiglu_loops(x.tolist(), wgu.tolist(), wd.tolist())
    got = o.swiglu_ffn(x, wgu, wd, round_h=False)
    assert np.max(np.abs(got - ref)) <= 1e-12


def test_ffn_round_h_within_half_ulp_bound():
    """Rounding h to bf16 moves each h element by at most 2^-9 relative, so the output moves
    by at most 2^-9 * sum_c |h_c| |Wd[c, j]|."""
    rng = np.random.default_rng(12)
    x = rng.standard_normal((6, 16))
    wgu = rng.standard_normal((16, 64)) * 0.2
    wd = rng.standard_normal((32, 16)) * 0.2
    g, u = x @ wgu[:, :32], x @ wgu[:, 32:]
    h = g / (1 + np.exp(-g)) * u
    bound = 2.0 ** -9 * (np.abs(h) @ np.abs(wd)) + 1e-15
    diff = np.abs(o.swiglu_ffn(x, wgu, wd, True) - o.swiglu_ffn(x, wgu, wd, False))
    assert np.all(diff <= bound)
    assert np.any(diff > 0)


def _layer_weights():
    c = _golden()["ffn"]
    wgu = np.array(c["w_gate_up"], float)
    wd = np.array(c["w_down"], float)
    return np.stack([wgu, wgu]), np.stack([wd, -wd])


@pytest.mark.parametrize("kc", [0, 1])
def test_layer_hand_case(kc):
    lay = _golden()["layer"]
    case = lay["k_cases"][kc]
    x = np.array(lay["x"], float)
    logits = np.array([[_val(v) for v in r] for r in lay["logits"]], dtype=np.float32)
    wgu, wd = _layer_weights()
    r = o.forward(x, logits, wgu, wd, case["k"], round_h=True)
    assert np.max(np.abs(r["out"] - np.array(case["out"]))) <= case["tol"]


def _brute_layer(x, logits, wgu, wd, k, score_fn, renorm, scale_input, round_h, wsgu=None, wsd=None):
    """Per-token loop with no permutation: ranking by a plain-Python sort, weights by math.exp,
    FFN by the textbook loops (with the bf16 rounding of h when asked)."""
    T = x.shape[0]
    out = np.zeros((T, wd.shape[-1]))
    for t in range(T):
        row = [float(v) for v in logits[t]]
        ids = _brute_topk(row, k)
        if score_fn == o.SOFTMAX:
            m = max(row)
            tot = sum(math.exp(v - m) for v in row)
            w = [math.exp(row[i] - m) / tot for i in ids]
        else:
            w = [1.0 / (1.0 + math.exp(-row[i])) for i in ids]
        if renorm:
            s = sum(w)
            w = [v / s for v in w]
        for j, e in enumerate(ids):
            xin = x[t] * (w[j] if scale_input else 1.0)
            g = xin @ wgu[e][:, :wgu.shape[-1] // 2]
            u = xin @ wgu[e][:, wgu.shape[-1] // 2:]
            h = np.array([gc / (1 + math.exp(-gc)) * uc for gc, uc in zip(g, u)])
            if round_h:
                h = np.array([_bf16_nearest_exact(v) for v in h])
            y = h @ wd[e]
            out[t] += y if scale_input else w[j] * y
        if wsgu is not None:
            I = wsgu.shape[1] // 2
            g, u = x[t] @ wsgu[:, :I], x[t] @ wsgu[:, I:]
            h = np.array([gc / (1 + math.exp(-gc)) * uc for gc, uc in zip(g, u)])
            if round_h:
                h = np.array([_bf16_nearest_exact(v) for v in h])
            out[t] += h @ wsd
    return out


@pytest.mark.parametrize("T,d,E,k,I,fn,renorm,scale,shared,round_h", [
    (24, 8, 4, 2, 6, o.SOFTMAX, True, False, False, False),
    (40, 16, 8, 3, 12, o.SOFTMAX, False, False, False, True),
    (33, 12, 6, 1, 10, o.SIGMOID, False, True, True, True),
    (64, 32, 8, 8, 16, o.SOFTMAX, True, False, False, True),
    (1, 8, 8, 2, 4, o.SOFTMAX, True, False, False, True),
])
def test_layer_matches_brute_force(T, d, E, k, I, fn, renorm, scale, shared, round_h):
    rng = np.random.default_rng(T * 7 + d)
    x = rng.standard_normal((T, d))
    logits = (rng.standard_normal((T, E)) * 1.3).astype(np.float32)
    wgu = rng.standard_normal((E, d, 2 * I)) * 0.3
    wd = rng.standard_normal((E, I, d)) * 0.3
    wsgu = rng.standard_normal((d, 2 * I)) * 0.3 if shared else None
    wsd = rng.standard_normal((I, d)) * 0.3 if shared else None
    r = o.forward(x, logits, wgu, wd, k, fn, renorm, scale, round_h, wsgu, wsd)
    ref = _brute_layer(x, logits, wgu, wd, k, fn, renorm, scale, round_h, wsgu, wsd)
    assert np.max(np.abs(r["out"] - ref)) <= 1e-12 * max(1.0, np.abs(ref).max())
    # the sampled per-token form agrees with the permuted form
    toks = list(range(0, T, 3))
    got = o.token_outputs(toks, x, r["topk_ids"], r["topk_weights"], wgu, wd, scale, round_h,
                          wsgu, wsd)
    assert np.max(np.abs(got - r["out"][toks])) <= 1e-12 * max(1.0, np.abs(ref).max())


def test_all_experts_equal_is_dense_mlp_times_weight_sum():
    """With every expert holding the same weights the layer is one dense MLP scaled by the sum
    of the selected gate weights (1 when renormalised)."""
    rng = np.random.default_rng(5)
    T, d, E, k, I = 30, 10, 6, 3, 7
    x = rng.standard_normal((T, d))
    logits = rng.standard_normal((T, E)).astype(np.float32)
    wgu1, wd1 = rng.standard_normal((d, 2 * I)), rng.standard_normal((I, d))
    wgu, wd = np.stack([wgu1] * E), np.stack([wd1] * E)
    dense = _dense_swiglu_loops(x.tolist(), wgu1.tolist(), wd1.tolist())
    for renorm in (True, False):
        r = o.forward(x, logits, wgu, wd, k, o.SOFTMAX, renorm, round_h=False)
        wsum = r["topk_weights"].sum(1, keepdims=True)
        assert np.max(np.abs(r["out"] - dense * wsum)) <= 1e-12 * np.abs(dense).max()
        if renorm:
            assert np.max(np.abs(r["out"] - dense)) <= 1e-12 * np.abs(dense).max()


def test_identity_experts_dispatch_combine_returns_input():
    """Dispatch then combine with identity experts (y = x_sorted): weight 1 and k = 1 gives x
    exactly; k = 2 with weight 1 gives 2x exactly; renormalised weights give x (sum w = 1)."""
    rng = np.random.default_rng(9)
    T, E, d = 50, 8, 12
    x = rng.standard_normal((T, d))
    for k, weights, scale in [(1, None, 1.0), (2, None, 2.0), (4, None, 4.0)]:
        ids = np.stack([rng.permutation(E)[:k] for _ in range(T)])
        _, _, s2p, p2s = o.dispatch(ids, E)
        xs = o.permute_rows(x, s2p, k)
        assert np.array_equal(o.combine(xs, p2s, weights, k), scale * x)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    ids, w = o.route(logits, 3)
    _, _, s2p, p2s = o.dispatch(ids, E)
    out = o.combine(o.permute_rows(x, s2p, 3), p2s, w, 3)
    assert np.max(np.abs(out - x)) <= 4e-16 * np.abs(x).max() * 4


def test_scale_input_form_equals_mlp_of_scaled_x_plus_shared():
    """Llama-4 form: out = FFN_e(s * x) + FFN_shared(x) with s the sigmoid score."""
    rng = np.random.default_rng(10)
    T, d, E, I = 20, 8, 4, 6
    x = rng.standard_normal((T, d))
    logits = rng.standard_normal((T, E)).astype(np.float32)
    wgu, wd = rng.standard_normal((E, d, 2 * I)), rng.standard_normal((E, I, d))
    wsgu, wsd = rng.standard_normal((d, 2 * I)), rng.standard_normal((I, d))
    r = o.forward(x, logits, wgu, wd, 1, o.SIGMOID, False, True, False, wsgu, wsd)
    for t in range(T):
        e = int(np.argmax(logits[t]))
        s = 1.0 / (1.0 + math.exp(-float(logits[t, e])))
        ref = _dense_swiglu_loops([list(s * x[t])], wgu[e].tolist(), wd[e].tolist())[0]
        ref = ref + _dense_swiglu_loops([list(x[t])], wsgu.tolist(), wsd.tolist())[0]
        assert np.max(np.abs(r["out"][t] - ref)) <= 1e-12 * np.abs(ref).max()


def test_empty_inputs():
    r = o.forward(np.zeros((0, 4)), np.zeros((0, 3), np.float32), np.zeros((3, 4, 4)),
                  np.zeros((3, 2, 4)), 2)
    assert r["out"].shape == (0, 4) and r["counts"].tolist() == [0, 0, 0]


def test_planted_mistakes_are_caught():
    """Each plausible mistake, planted in a copy of the oracle's FFN, fails the hand case."""
    c = _golden()["ffn"]
    x = np.array([c["x"]], float)
    wgu = np.array(c["w_gate_up"], float)
    wd = np.array(c["w_down"], float)
    I = wgu.shape[1] // 2

    def swapped(x):   # gate and up exchanged
        g, u = x @ wgu[:, I:], x @ wgu[:, :I]
        return (g / (1 + np.exp(-g)) * u) @ wd

    def no_gate(x):   # activation dropped
        g, u = x @ wgu[:, :I], x @ wgu[:, I:]
        return (g * u) @ wd

    def wrong_sign(x):
        g, u = x @ wgu[:, :I], x @ wgu[:, I:]
        return (g / (1 + np.exp(g)) * u) @ wd

    for bad in (swapped, no_gate, wrong_sign):
        assert np.max(np.abs(bad(x)[0] - np.array(c["y"]))) > 1.0


# ----------------------------------------------------------------------------------------------
# router logits from hidden states
# ----------------------------------------------------------------------------------------------
def test_router_logits_one_hot_rows_pick_weight_rows():
    """x = one-hot rows: each logit row is a row of the router weight (+ bias), exactly."""
    rng = np.random.default_rng(3)
    d, E = 7, 5
    w = rng.standard_normal((d, E)).astype(np.float32)
    b = rng.standard_normal(E).astype(np.float32)
    x = np.eye(d)[[3, 0, 6, 3]]
    z = o.router_logits(x, w, b)
    assert np.array_equal(z, w[[3, 0, 6, 3]].astype(np.float64) + b.astype(np.float64))
    assert np.array_equal(o.router_logits(x, w), w[[3, 0, 6, 3]].astype(np.float64))


def test_router_logits_match_plain_loops():
    """Brute force in plain Python with exact rational arithmetic on small shapes."""
    rng = np.random.default_rng(4)
    T, d, E = 3, 6, 4
    x = rng.standard_normal((T, d)).astype(np.float32)
    w = rng.standard_normal((d, E)).astype(np.float32)
    b = rng.standard_normal(E).astype(np.float32)
    z = o.router_logits(x, w, b)
    for t in range(T):
        for e in range(E):
            exact = sum(Fraction(float(x[t, i])) * Fraction(float(w[i, e])) for i in range(d))
            exact += Fraction(float(b[e]))
            assert abs(z[t, e] - float(exact)) <= 1e-15 * (1 + abs(float(exact)))
    # a transposed weight (a plausible mistake) gives different logits
    assert not np.allclose(o.router_logits(x[:, :4], w[:4, :].T), z[:, :4])
