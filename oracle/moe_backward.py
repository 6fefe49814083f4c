"""CPU oracle for the backward pass of the MoE expert layer.

TEST INFRASTRUCTURE ONLY, like ``moe_oracle``: only the tests, the smoke check and the
benchmark's CPU-baseline leg may import it; the CUDA package never does, and this module
imports nothing from the CUDA package.

The pages train these layers ("Expert parallelism", intro: the router's weights multiply the
expert outputs, so the loss reaches the router through them; the pages' only measured numbers
are training runs). The forward is ``moe_oracle.forward``; this module states its gradient with
respect to the hidden states x, the expert weights W_gate_up / W_down (and the shared expert's),
the routing weights and the router logits, for a cotangent ``dout`` of the layer output.

Arithmetic is float64 (numpy; a matrix product is the only library primitive used as a step).
With ``bf16_points=True`` the oracle mirrors the values a bf16 layer stores between kernels,
each rounded to nearest even, the reading adopted where the pages are silent:
  - the gate/up accumulators a = x W_gate, b = x W_up are saved as bf16 for the backward pass
    (unscaled: the router score of a scaled-input layer is applied when they are used);
  - dy = w * dout (the down projection's incoming gradient, one row per routed slot) is bf16;
  - [d_a | d_b], the gradient of the gate/up accumulators, is bf16;
  - h (the forward activation) is the forward's bf16 h.
Everything else (the weight gradients, the gradient of x before its final rounding, the
routing-weight and logit gradients) is exact. With ``bf16_points=False`` and a forward run
with ``round_h=False`` the result is the exact gradient of the exact fp64 layer, which the
tests pin with central finite differences.

Notation per routed row p (token t, slot j, expert e) with router score s (s = 1 unless the
score scales the input):
  a = x_t W_gate[e], b = x_t W_up[e], g = s a, u = s b, h = SiLU(g) u, y = h W_down[e],
  out_t = sum_j w_tj y_p (combine weight w = 1 when the score scales the input) + shared(x_t).
"""
from __future__ import annotations

import numpy as np

from oracle import moe_oracle as fwd

SOFTMAX, SIGMOID = fwd.SOFTMAX, fwd.SIGMOID


def _rb(a, on: bool):
    return fwd.round_bf16(a) if on else np.asarray(a, dtype=np.float64)


def forward_train(x, logits, w_gate_up, w_down, k: int, score_fn: int = SOFTMAX,
                  renormalize: bool = True, scale_input: bool = False, round_h: bool = True,
                  bf16_points: bool = True, w_shared_gate_up=None, w_shared_down=None):
    """The forward pass with what the backward pass needs: the routing, the saved gate/up
    accumulators (``ab`` [R, 2I], unscaled) and the activations ``h`` [R, I] of the routed rows
    (and ``ab_shared``, ``h_shared`` of the shared expert), besides ``moe_oracle.forward``'s
    outputs. round_h rounds h to bf16 as the forward does; bf16_points rounds the saved ``ab``.
    """
    f = fwd.forward(x, logits, w_gate_up, w_down, k, score_fn, renormalize, scale_input,
                    round_h, w_shared_gate_up, w_shared_down)
    xs = f["x_sorted"]
    offsets = f["offsets"]
    R, d = xs.shape
    I = np.asarray(w_down[0]).shape[0] if len(w_down) else 0
    ab = np.zeros((R, 2 * I), dtype=np.float64)
    h = np.zeros((R, I), dtype=np.float64)
    s = (f["topk_weights"].reshape(-1)[f["sorted_to_slot"]] if scale_input
         else np.ones(R, dtype=np.float64))
    for e in range(len(offsets) - 1):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi > lo:
            acc = xs[lo:hi] @ np.asarray(w_gate_up[e], dtype=np.float64)
            g = s[lo:hi, None] * acc[:, :I]
            u = s[lo:hi, None] * acc[:, I:]
            h[lo:hi] = _rb(g / (1.0 + np.exp(-g)) * u, round_h)
            ab[lo:hi] = acc
    f["ab"] = _rb(ab, bf16_points)
    f["h"] = h
    f["row_scale"] = s
    if w_shared_gate_up is not None:
        xx = np.asarray(x, dtype=np.float64)
        acc = xx @ np.asarray(w_shared_gate_up, dtype=np.float64)
        Is = acc.shape[1] // 2
        g, u = acc[:, :Is], acc[:, Is:]
        f["h_shared"] = _rb(g / (1.0 + np.exp(-g)) * u, round_h)
        f["ab_shared"] = _rb(acc, bf16_points)
    return f


def swiglu_backward(dh, ab, s, bf16_points: bool):
    """Gradient of h = SiLU(s a) (s b) with respect to the accumulators a, b (and to s).

    dh [n, I], ab [n, 2I] (a = first half), s [n]. With g = s a, u = s b and
    sigma = 1 / (1 + exp(-g)): dh/dg = u sigma (1 + g (1 - sigma)), dh/du = g sigma, so
    d_a = s dg, d_b = s du and d_s = sum_c (dg_c a_c + du_c b_c).
    Returns d_ab [n, 2I] (bf16 when bf16_points) and d_s [n] (exact).
    """
    dh = np.asarray(dh, dtype=np.float64)
    ab = np.asarray(ab, dtype=np.float64)
    I = dh.shape[1]
    a, b = ab[:, :I], ab[:, I:]
    s = np.asarray(s, dtype=np.float64)[:, None]
    g, u = s * a, s * b
    sig = 1.0 / (1.0 + np.exp(-g))
    dg = dh * u * sig * (1.0 + g * (1.0 - sig))
    du = dh * g * sig
    d_s = np.sum(dg * a + du * b, axis=1)
    d_ab = np.concatenate([s * dg, s * du], axis=1)
    return _rb(d_ab, bf16_points), d_s


def route_backward(logits, ids, d_weights, score_fn: int = SOFTMAX, renormalize: bool = True):
    """Gradient of the routing weights ``route`` returns with respect to the fp32 logits, for
    the selected experts held fixed (the top-k choice is piecewise constant in the logits).

    Softmax over all E (then the k selected taken): w_j = p_{i_j}, so
    dl_m = p_m (D_m - sum_j w_j d_j) with D_m = d_j when m = i_j, else 0.
    Softmax renormalised over the k selected (= a softmax over the k selected logits):
    dl_{i_j} = w_j (d_j - sum_l w_l d_l), zero for the other experts.
    Sigmoid: sigma_j = 1 / (1 + exp(-l_{i_j})), dl_{i_j} = d sigma_j * sigma_j (1 - sigma_j) with
    d sigma_j = d_j, or, renormalised (w_j = sigma_j / S, S = sum over the selected),
    d sigma_j = (d_j - sum_l w_l d_l) / S.
    Returns d_logits float64 [T, E].
    """
    z = np.asarray(logits, dtype=np.float32).astype(np.float64)
    ids = np.asarray(ids, dtype=np.int64)
    dw = np.asarray(d_weights, dtype=np.float64)
    T, E = z.shape
    _, w = fwd.route(logits, ids.shape[1], score_fn, renormalize)
    dl = np.zeros((T, E), dtype=np.float64)
    for t in range(T):
        sel = ids[t]
        inner = float(np.dot(w[t], dw[t]))
        if score_fn == SOFTMAX:
            if renormalize:
                dl[t, sel] = w[t] * (dw[t] - inner)
            else:
                m = np.max(z[t])
                p = np.exp(z[t] - m)
                p = p / np.sum(p)
                D = np.zeros(E)
                D[sel] = dw[t]
                dl[t] = p * (D - inner)
        elif score_fn == SIGMOID:
            sig = 1.0 / (1.0 + np.exp(-z[t, sel]))
            if renormalize:
                dsig = (dw[t] - inner) / np.sum(sig)
            else:
                dsig = dw[t]
            dl[t, sel] = dsig * sig * (1.0 - sig)
        else:
            raise ValueError(score_fn)
    return dl


def backward(f, dout, x, logits, w_gate_up, w_down, k: int, score_fn: int = SOFTMAX,
             renormalize: bool = True, scale_input: bool = False, bf16_points: bool = True,
             w_shared_gate_up=None, w_shared_down=None):
    """Gradients of sum(out * dout) for the forward ``f`` (from ``forward_train`` with the same
    arguments). Returns a dict with:
      dx [T, d] (exact sum of the routed rows' and the shared expert's contributions),
      dy_sorted [R, d], d_ab [R, 2I], dx_sorted [R, d], d_scale [R] (scaled-input layers),
      d_w_gate_up [E, d, 2I], d_w_down [E, I, d], d_topk_weights [T, k], d_logits [T, E],
      and for a shared expert d_w_shared_gate_up [d, 2Is], d_w_shared_down [Is, d].
    Steps, per the chain rule through the forward's steps in reverse:
      combine:  dy_p = w_tj dout_t (dout_t for scaled-input layers); d w_tj = dout_t . y_p;
      down:     dh_p = dy_p W_down[e]^T; d W_down[e] = sum_p h_p^T dy_p;
      SwiGLU:   swiglu_backward;
      gate/up:  dx_p = d_ab_p W_gate_up[e]^T; d W_gate_up[e] = sum_p x_p^T d_ab_p;
      dispatch: dx_t = sum_j dx_{p(t, j)} (the permutation's transpose);
      route:    route_backward of d w (for scaled-input layers d w_tj = d_s of its row).
    """
    dout = np.asarray(dout, dtype=np.float64)
    x = np.asarray(x, dtype=np.float64)
    T, d = dout.shape
    ids, w = f["topk_ids"], f["topk_weights"]
    offsets, s2p, p2s = f["offsets"], f["sorted_to_slot"], f["slot_to_sorted"]
    R = s2p.size
    E = len(offsets) - 1
    tok = s2p // k
    slot_j = s2p % k
    # combine
    if scale_input:
        dy = dout[tok]
    else:
        dy = w[tok, slot_j][:, None] * dout[tok]
    dy = _rb(dy, bf16_points)
    d_w = np.zeros((T, k), dtype=np.float64)
    if not scale_input:
        y = f["y_sorted"]
        for t in range(T):
            for j in range(k):
                d_w[t, j] = float(np.dot(dout[t], y[p2s[t * k + j]]))
    I = np.asarray(w_down[0]).shape[0]
    d_ab = np.zeros((R, 2 * I), dtype=np.float64)
    d_s = np.zeros(R, dtype=np.float64)
    dx_sorted = np.zeros((R, d), dtype=np.float64)
    dwgu = np.zeros((E, d, 2 * I), dtype=np.float64)
    dwd = np.zeros((E, I, d), dtype=np.float64)
    xs = f["x_sorted"]
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi <= lo:
            continue  # an expert with no rows gets a zero weight gradient
        wgu = np.asarray(w_gate_up[e], dtype=np.float64)
        wd = np.asarray(w_down[e], dtype=np.float64)
        dh = dy[lo:hi] @ wd.T
        dwd[e] = f["h"][lo:hi].T @ dy[lo:hi]
        d_ab[lo:hi], d_s[lo:hi] = swiglu_backward(dh, f["ab"][lo:hi], f["row_scale"][lo:hi],
                                                  bf16_points)
        dx_sorted[lo:hi] = d_ab[lo:hi] @ wgu.T
        dwgu[e] = xs[lo:hi].T @ d_ab[lo:hi]
    dx = np.zeros((T, d), dtype=np.float64)
    for j in range(k):
        dx += dx_sorted[p2s[j::k]]
    if scale_input:
        d_w = d_s[p2s].reshape(T, k)
    out = dict(dy_sorted=dy, d_ab=d_ab, d_scale=d_s, dx_sorted=dx_sorted,
               d_w_gate_up=dwgu, d_w_down=dwd, d_topk_weights=d_w,
               d_logits=route_backward(logits, ids, d_w, score_fn, renormalize))
    if w_shared_gate_up is not None:
        wsgu = np.asarray(w_shared_gate_up, dtype=np.float64)
        wsd = np.asarray(w_shared_down, dtype=np.float64)
        dys = _rb(dout, bf16_points)
        dhs = dys @ wsd.T
        out["d_w_shared_down"] = f["h_shared"].T @ dys
        dabs, _ = swiglu_backward(dhs, f["ab_shared"], np.ones(T), bf16_points)
        out["d_ab_shared"] = dabs
        out["dx_shared"] = dabs @ wsgu.T
        out["d_w_shared_gate_up"] = x.T @ dabs
        dx = dx + out["dx_shared"]
    out["dx"] = dx
    return out
