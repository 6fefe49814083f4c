"""Pins of the backward oracle against something other than itself:
- central finite differences of the forward oracle (exact fp64 layer: no rounding points) for
  every gradient it returns: hidden states, expert weights, shared-expert weights, routing
  weights and router logits, in the four router forms (softmax / sigmoid, renormalised or not)
  and with the score scaling the input;
- closed forms of the router Jacobian: the softmax gradients sum to zero over the experts
  (a softmax does not change when every logit moves by the same amount), and renormalised
  weights, which always sum to one, give a zero gradient for a cotangent of all ones;
- the bf16 storage points change the gradients by no more than bf16 rounding can.
"""
import numpy as np
import pytest

from oracle import moe_backward as B
from oracle import moe_oracle as o


def _layer(seed, T=6, d=8, E=4, k=2, I=6, Is=0, gap=0.15):
    rng = np.random.default_rng(seed)
    x = rng.normal(0, 1, (T, d))
    wgu = rng.normal(0, 0.4, (E, d, 2 * I))
    wd = rng.normal(0, 0.4, (E, I, d))
    # logits whose sorted values are at least `gap` apart, so a small move keeps the top-k
    base = np.arange(E, dtype=np.float64) * gap
    logits = np.stack([rng.permutation(base) for _ in range(T)]) + rng.normal(0, 1, (T, 1))
    logits = logits.astype(np.float32)
    sh = {}
    if Is:
        sh = dict(w_shared_gate_up=rng.normal(0, 0.4, (d, 2 * Is)),
                  w_shared_down=rng.normal(0, 0.4, (Is, d)))
    G = rng.normal(0, 1, (T, d))
    return x, logits, wgu, wd, sh, G


def _loss(x, logits, wgu, wd, k, fn, renorm, scale, sh, G):
    f = o.forward(x, logits, wgu, wd, k, fn, renorm, scale, round_h=False, **sh)
    return float(np.sum(f["out"] * G))


def _grads(x, logits, wgu, wd, k, fn, renorm, scale, sh, G):
    f = B.forward_train(x, logits, wgu, wd, k, fn, renorm, scale, round_h=False,
                        bf16_points=False, **sh)
    return B.backward(f, G, x, logits, wgu, wd, k, fn, renorm, scale, bf16_points=False, **sh)


MODES = [  # (score fn, renormalise, score scales the input, k, shared expert size)
    (o.SOFTMAX, True, False, 2, 0),
    (o.SOFTMAX, False, False, 2, 0),
    (o.SIGMOID, False, False, 2, 0),
    (o.SIGMOID, True, False, 3, 0),
    (o.SIGMOID, False, True, 1, 5),
    (o.SOFTMAX, True, True, 2, 0),
]


def _fd(fun, arr, idx, eps):
    a0 = arr[idx]
    arr[idx] = a0 + eps
    lp = fun()
    arr[idx] = a0 - eps
    lm = fun()
    arr[idx] = a0
    return (lp - lm) / (2 * eps)


@pytest.mark.parametrize("mode", MODES, ids=[f"fn{m[0]}_r{int(m[1])}_s{int(m[2])}_k{m[3]}_is{m[4]}"
                                            for m in MODES])
def test_gradients_match_finite_differences(mode):
    fn, renorm, scale, k, Is = mode
    x, logits, wgu, wd, sh, G = _layer(11 + k + 3 * Is + 5 * fn, k=k, Is=Is)
    g = _grads(x, logits, wgu, wd, k, fn, renorm, scale, sh, G)

    def L():
        return _loss(x, logits, wgu, wd, k, fn, renorm, scale, sh, G)

    rng = np.random.default_rng(0)
    checks = [("dx", x), ("d_w_gate_up", wgu), ("d_w_down", wd)]
    if Is:
        checks += [("d_w_shared_gate_up", sh["w_shared_gate_up"]),
                   ("d_w_shared_down", sh["w_shared_down"])]
    for name, arr in checks:
        for _ in range(12):
            idx = tuple(int(rng.integers(0, n)) for n in arr.shape)
            num = _fd(L, arr, idx, 1e-5)
            ana = g[name][idx]
            assert abs(num - ana) <= 1e-7 * (1 + abs(num)), (name, idx, num, ana)
    # logits: the forward reads them as fp32, so move them by exact fp32 steps and cancel the
    # O(h^2) term with Richardson extrapolation
    lg = logits.astype(np.float32)

    def Lg():
        return _loss(x, lg, wgu, wd, k, fn, renorm, scale, sh, G)

    for t in range(lg.shape[0]):
        for e in range(lg.shape[1]):
            d1 = _fd(Lg, lg, (t, e), np.float32(2.0 ** -8))
            d2 = _fd(Lg, lg, (t, e), np.float32(2.0 ** -9))
            num = (4 * d2 - d1) / 3
            assert abs(num - g["d_logits"][t, e]) <= 2e-6 * (1 + abs(num)), (t, e)


@pytest.mark.parametrize("fn,renorm", [(o.SOFTMAX, True), (o.SOFTMAX, False),
                                       (o.SIGMOID, True), (o.SIGMOID, False)])
def test_route_backward_matches_finite_differences(fn, renorm):
    rng = np.random.default_rng(3)
    T, E, k = 5, 9, 3
    base = np.arange(E) * 0.2
    logits = (np.stack([rng.permutation(base) for _ in range(T)])
              + rng.normal(0, 1, (T, 1))).astype(np.float32)
    c = rng.normal(0, 1, (T, k))
    ids, _ = o.route(logits, k, fn, renorm)
    dl = B.route_backward(logits, ids, c, fn, renorm)

    def L():
        ids2, w2 = o.route(logits, k, fn, renorm)
        assert np.array_equal(ids2, ids)
        return float(np.sum(w2 * c))

    for t in range(T):
        for e in range(E):
            d1 = _fd(L, logits, (t, e), np.float32(2.0 ** -8))
            d2 = _fd(L, logits, (t, e), np.float32(2.0 ** -9))
            assert abs((4 * d2 - d1) / 3 - dl[t, e]) <= 2e-6 * (1 + abs(dl[t, e]))


def test_route_backward_closed_forms():
    rng = np.random.default_rng(4)
    T, E, k = 7, 16, 4
    logits = rng.normal(0, 1.3, (T, E)).astype(np.float32)
    c = rng.normal(0, 1, (T, k))
    for renorm in (True, False):
        ids, _ = o.route(logits, k, o.SOFTMAX, renorm)
        dl = B.route_backward(logits, ids, c, o.SOFTMAX, renorm)
        np.testing.assert_allclose(dl.sum(axis=1), 0.0, atol=1e-14)
        # only the selected experts move when renormalised
        if renorm:
            mask = np.zeros((T, E), bool)
            np.put_along_axis(mask, ids.astype(np.int64), True, axis=1)
            assert np.all(dl[~mask] == 0.0)
    for fn in (o.SOFTMAX, o.SIGMOID):
        ids, _ = o.route(logits, k, fn, True)
        dl = B.route_backward(logits, ids, np.ones((T, k)), fn, True)
        np.testing.assert_allclose(dl, 0.0, atol=1e-15)


def test_swiglu_backward_matches_finite_differences():
    rng = np.random.default_rng(5)
    n, I = 4, 7
    ab = rng.normal(0, 1.5, (n, 2 * I))
    s = rng.uniform(0.2, 1.0, n)
    dh = rng.normal(0, 1, (n, I))

    def L():
        g, u = s[:, None] * ab[:, :I], s[:, None] * ab[:, I:]
        return float(np.sum(g / (1 + np.exp(-g)) * u * dh))

    d_ab, d_s = B.swiglu_backward(dh, ab, s, bf16_points=False)
    for i in range(n):
        for c in range(2 * I):
            assert abs(_fd(L, ab, (i, c), 1e-6) - d_ab[i, c]) <= 1e-8 * (1 + abs(d_ab[i, c]))
        assert abs(_fd(L, s, (i,), 1e-6) - d_s[i]) <= 1e-8 * (1 + abs(d_s[i]))


def test_bf16_points_stay_within_rounding():
    x, logits, wgu, wd, sh, G = _layer(21, T=10, d=16, E=4, k=2, I=8)
    G = o.round_bf16(G)
    exact = _grads(x, logits, wgu, wd, 2, o.SOFTMAX, True, False, sh, G)
    f = B.forward_train(x, logits, wgu, wd, 2, o.SOFTMAX, True, False, round_h=True,
                        bf16_points=True)
    mixed = B.backward(f, G, x, logits, wgu, wd, 2, o.SOFTMAX, True, False, bf16_points=True)
    for name in ("dx", "d_w_gate_up", "d_w_down", "d_topk_weights", "d_logits"):
        a, b = exact[name], mixed[name]
        # rms error over rms value: two bf16 roundings (2^-9 relative each) on the way
        err = np.sqrt(np.mean((a - b) ** 2) / np.mean(a ** 2))
        assert 0 < err < 1e-2, (name, err)


def test_all_experts_equal_gives_the_dense_gradient():
    # every expert the same FFN and renormalised weights: the layer is that FFN, so dx and the
    # summed weight gradients equal a dense SwiGLU MLP's (written out here by the chain rule)
    rng = np.random.default_rng(6)
    T, d, E, k, I = 5, 6, 3, 2, 4
    x = rng.normal(0, 1, (T, d))
    w1 = rng.normal(0, 0.5, (d, 2 * I))
    w2 = rng.normal(0, 0.5, (I, d))
    wgu = np.stack([w1] * E)
    wd = np.stack([w2] * E)
    logits = rng.normal(0, 1, (T, E)).astype(np.float32)
    G = rng.normal(0, 1, (T, d))
    f = B.forward_train(x, logits, wgu, wd, k, o.SOFTMAX, True, False, round_h=False,
                        bf16_points=False)
    g = B.backward(f, G, x, logits, wgu, wd, k, o.SOFTMAX, True, False, bf16_points=False)
    a, b = x @ w1[:, :I], x @ w1[:, I:]
    sig = 1 / (1 + np.exp(-a))
    h = a * sig * b
    dh = G @ w2.T
    da = dh * b * sig * (1 + a * (1 - sig))
    db = dh * a * sig
    dx = np.concatenate([da, db], 1) @ w1.T
    np.testing.assert_allclose(g["dx"], dx, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(g["d_w_down"].sum(0), h.T @ G, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(g["d_w_gate_up"].sum(0), x.T @ np.concatenate([da, db], 1),
                               rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(g["d_logits"], 0.0, atol=1e-12)
