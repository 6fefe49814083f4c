"""CPU oracle for the MoE expert layer: route -> dispatch -> per-expert SwiGLU FFN -> combine.

TEST INFRASTRUCTURE ONLY. This module is the plain, slow, obviously correct statement of what the
CUDA path computes. Only the tests, the smoke check and the benchmark's CPU-baseline leg may
import it; the product path never does. It imports nothing from the CUDA package and the CUDA
package imports nothing from it.

Arithmetic is float64 throughout (numpy; a matrix product is the only library primitive used as
a step). Inputs are the exact values the GPU receives (bf16 or fp32 widened to fp64; fp32
logits). The one rounding the oracle mirrors is the bf16 storage of the SwiGLU activation ``h``
in bf16 layers; the final output is left unrounded.

Sources (Transformers documentation pages):
- "Expert parallelism", intro and "DistributedConfig": a router sends each token to a few
  experts and gathers the results; Llama-4 experts receive tokens already scaled by the router
  score.
- "Expert parallelism", "Adding an implementation": ``__call__(hidden_states, top_k_index,
  top_k_weights)`` returns the weighted expert output for each token; ``experts_forward`` runs on
  the rows routed to each expert.
- "Expert parallelism", "Token dispatch": every (token, expert) pair goes to that expert, the
  expert runs on what it received, and the outputs are combined with the routing weights.
- "Expert parallelism", "With tensor parallelism": token slices may be uneven or empty.
- "Tensor parallelism for inference", "Packed strategies": ``gate_up_proj`` is
  ``[num_experts, hidden, 2 * expert_dim]``, multiplied with ``bmm`` and split with
  ``chunk(2, dim=-1)`` into gate (first half) and up (second half).

Readings where the pages are silent (router score function, tie order, row order, activation,
rounding points) are stated at each function. Every function here is pinned by the
``-m "not gpu"`` tests against brute force, closed forms or invariants.
"""
from __future__ import annotations

import numpy as np

SOFTMAX, SIGMOID = 0, 1


# ----------------------------------------------------------------------------------------------
# bf16 rounding (round to nearest, ties to even), written from the format's definition:
# 8 significant bits, exponent range of fp32 (min normal 2**-126, subnormal quantum 2**-133).
# ----------------------------------------------------------------------------------------------
_BF16_MAX = (2.0 - 2.0 ** -7) * 2.0 ** 127


def round_bf16(a) -> np.ndarray:
    """Round float64 values to the nearest bf16 value (ties to even); returns float64."""
    a = np.asarray(a, dtype=np.float64)
    _, e = np.frexp(a)                        # a = m * 2**e with 0.5 <= |m| < 1
    q = np.maximum(e - 8, -133)               # quantum of the bf16 binade holding a
    r = np.ldexp(np.rint(np.ldexp(a, -q)), q)  # np.rint rounds half to even; ldexp is exact
    r = np.where(np.abs(r) > _BF16_MAX, np.copysign(np.inf, a), r)
    return np.where(np.isfinite(a), r, a)


# ----------------------------------------------------------------------------------------------
# Step 1: router top-k gating
# ----------------------------------------------------------------------------------------------
def router_logits(x, w_router, bias=None):
    """The router's logits from hidden states: x [T, d] @ w_router [d, E] (+ bias [E]), in
    float64 ("Expert parallelism", intro: a router sends each token to its experts; the
    workloads define the logits as the hidden states times a router weight, plus an optional
    per-expert bias). No rounding: the GPU rounds once to fp32 at the end of a sequential fp32
    sum, and the tests compare against this exact value within that sum's error bound."""
    z = np.asarray(x, dtype=np.float64) @ np.asarray(w_router, dtype=np.float64)
    if bias is not None:
        z = z + np.asarray(bias, dtype=np.float64)[None, :]
    return z


def route(logits, k: int, score_fn: int = SOFTMAX, renormalize: bool = True):
    """Top-k experts per token and their weights ("top_k_index", "top_k_weights").

    Reading (the pages fix only the outputs' names and shapes):
    - selection is on the fp32 logits, in descending value, ties to the lower expert index;
      -0.0 equals +0.0; NaN ranks below -inf (then lower index);
    - slot j = 0 holds the best expert;
    - softmax: weight_j = exp(l_j - max) / sum over all E of exp(l_i - max); with renormalize the
      k selected weights are divided by their sum (equal to a softmax over the k selected logits);
    - sigmoid: weight_j = 1 / (1 + exp(-l_j)); divided by the sum over the k selected only when
      renormalize is set.
    Returns ids int32 [T, k] and weights float64 [T, k].
    """
    z = np.asarray(logits, dtype=np.float32).astype(np.float64)
    T, E = z.shape
    assert 1 <= k <= E
    # Primary key: NaN last; secondary: descending value. lexsort is stable, so equal keys keep
    # ascending expert index.
    nan = np.isnan(z)
    order = np.lexsort((np.where(nan, 0.0, -z), nan), axis=-1)
    ids = order[:, :k].astype(np.int32)
    sel = np.take_along_axis(z, ids.astype(np.int64), axis=1)
    if score_fn == SOFTMAX:
        m = np.max(np.where(np.isnan(z), -np.inf, z), axis=1, keepdims=True)
        p_all = np.exp(z - m)
        w = np.exp(sel - m) / np.sum(p_all, axis=1, keepdims=True)
    elif score_fn == SIGMOID:
        w = 1.0 / (1.0 + np.exp(-sel))
    else:
        raise ValueError(score_fn)
    if renormalize:
        w = w / np.sum(w, axis=1, keepdims=True)
    return ids, w


# ----------------------------------------------------------------------------------------------
# Step 2: dispatch (the one-GPU form of sending each (token, expert) pair to its expert)
# ----------------------------------------------------------------------------------------------
def dispatch(ids, E: int):
    """Group the T*k routed slots by expert.

    Slot s = t*k + j holds (token t, expert ids[t, j]). Reading: inside an expert, rows keep
    ascending slot order (a stable counting sort), which fixes the permutation exactly.
    Returns counts [E], offsets [E+1] (exclusive prefix), sorted_to_slot [R] (sorted position ->
    slot) and slot_to_sorted [R] (its inverse), all int64.
    """
    flat = np.asarray(ids, dtype=np.int64).reshape(-1)
    R = flat.size
    counts = np.zeros(E, dtype=np.int64)
    for e in flat:
        counts[e] += 1
    offsets = np.zeros(E + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts)
    cursor = offsets[:-1].copy()
    sorted_to_slot = np.empty(R, dtype=np.int64)
    for s in range(R):
        e = flat[s]
        sorted_to_slot[cursor[e]] = s
        cursor[e] += 1
    slot_to_sorted = np.empty(R, dtype=np.int64)
    slot_to_sorted[sorted_to_slot] = np.arange(R)
    return counts, offsets, sorted_to_slot, slot_to_sorted


def permute_rows(x, sorted_to_slot, k: int):
    """x_sorted[p] = x[token of slot sorted_to_slot[p]]."""
    return np.asarray(x)[np.asarray(sorted_to_slot) // k]


# ----------------------------------------------------------------------------------------------
# Step 3: per-expert gated feed-forward (gate/up projection, SwiGLU, down projection)
# ----------------------------------------------------------------------------------------------
def swiglu_activation(xrows, w_gate_up, round_h: bool):
    """h = SiLU(x @ W_gate) * (x @ W_up) for a block of rows of one expert: the first half of
    the gated feed-forward, the value the down projection reads.

    w_gate_up is [d, 2I] with gate = columns [0, I) and up = columns [I, 2I) (the packed
    layout and chunk order of "Packed strategies"). SiLU(z) = z * sigmoid(z).
    round_h: store the activation as bf16 (round to nearest even), the one intermediate
    rounding a bf16 layer fixes.
    """
    x = np.asarray(xrows, dtype=np.float64)
    wgu = np.asarray(w_gate_up, dtype=np.float64)
    I = wgu.shape[1] // 2
    gate = x @ wgu[:, :I]
    up = x @ wgu[:, I:]
    h = gate / (1.0 + np.exp(-gate)) * up
    if round_h:
        h = round_bf16(h)
    return h


def swiglu_ffn(xrows, w_gate_up, w_down, round_h: bool, return_h: bool = False):
    """y = (SiLU(x @ W_gate) * (x @ W_up)) @ W_down for a block of rows of one expert
    (``swiglu_activation`` then the down projection; w_down is [I, d]).
    return_h: also return the activation h, as (y, h).
    """
    h = swiglu_activation(xrows, w_gate_up, round_h)
    y = h @ np.asarray(w_down, dtype=np.float64)
    return (y, h) if return_h else y


def experts(x_sorted, offsets, w_gate_up, w_down, round_h: bool, row_scale=None,
            return_h: bool = False):
    """Run expert e on its rows [offsets[e], offsets[e+1]); returns y_sorted float64 [R, d]
    (with return_h, the pair (y_sorted, h) with h [R, I] the activation of every row).

    w_gate_up[e] / w_down[e] are read one expert at a time, so any indexable of per-expert
    arrays works (e.g. one that widens bf16 blocks to float64 on access).

    row_scale (optional, [R]): the router score that multiplies each row's expert input (the
    Llama-4 form, "experts receive each token already scaled by the router score").
    """
    xs = np.asarray(x_sorted, dtype=np.float64)
    if row_scale is not None:
        xs = xs * np.asarray(row_scale, dtype=np.float64)[:, None]
    R, d = xs.shape   # the layer maps hidden size d back to d
    y = np.zeros((R, d), dtype=np.float64)
    h = None
    E = len(offsets) - 1
    for e in range(E):
        a, b = int(offsets[e]), int(offsets[e + 1])
        if b > a:  # an expert with no rows does no work (uneven or empty slices)
            y[a:b], he = swiglu_ffn(xs[a:b], w_gate_up[e], w_down[e], round_h, return_h=True)
            if return_h:
                if h is None:
                    h = np.zeros((R, he.shape[1]), dtype=np.float64)
                h[a:b] = he
    if return_h:
        if h is None:   # no rows at all: the width comes from the down projection
            h = np.zeros((R, np.asarray(w_down[0]).shape[0]), dtype=np.float64)
        return y, h
    return y


# ----------------------------------------------------------------------------------------------
# Step 4: weighted combine back to token order
# ----------------------------------------------------------------------------------------------
def combine(y_sorted, slot_to_sorted, weights, k: int, y_shared=None):
    """out[t] = sum_j weights[t, j] * y_sorted[slot_to_sorted[t*k + j]]  (+ y_shared[t]).

    weights None means weight 1 for every slot (the score was already applied to the input).
    Summed in float64 in slot order, then the shared-expert row is added; never rounded.
    """
    y = np.asarray(y_sorted, dtype=np.float64)
    pos = np.asarray(slot_to_sorted, dtype=np.int64)
    T = pos.size // k
    out = np.zeros((T, y.shape[1]), dtype=np.float64)
    for j in range(k):
        rows = y[pos[j::k]]
        if weights is not None:
            rows = rows * np.asarray(weights, dtype=np.float64)[:, j:j + 1]
        out += rows
    if y_shared is not None:
        out += np.asarray(y_shared, dtype=np.float64)
    return out


# ----------------------------------------------------------------------------------------------
# The whole layer
# ----------------------------------------------------------------------------------------------
def forward(x, logits, w_gate_up, w_down, k: int, score_fn: int = SOFTMAX,
            renormalize: bool = True, scale_input: bool = False, round_h: bool = True,
            w_shared_gate_up=None, w_shared_down=None):
    """Route, dispatch, experts and combine, returning every intermediate in a dict.

    scale_input: the router weight multiplies the expert input and the combine weight is 1.
    Shared expert (optional): an always-on SwiGLU expert on the unscaled input, added after the
    routed sum.
    """
    x = np.asarray(x, dtype=np.float64)
    E = len(w_gate_up)   # per-expert blocks are only ever indexed one expert at a time
    ids, w = route(logits, k, score_fn, renormalize)
    counts, offsets, s2p, p2s = dispatch(ids, E)
    xs = permute_rows(x, s2p, k)
    scale = w.reshape(-1)[s2p] if scale_input else None
    y, h = experts(xs, offsets, w_gate_up, w_down, round_h, row_scale=scale, return_h=True)
    ys = hs = None
    if w_shared_gate_up is not None:
        ys, hs = swiglu_ffn(x, w_shared_gate_up, w_shared_down, round_h, return_h=True)
    out = combine(y, p2s, None if scale_input else w, k, ys)
    return dict(topk_ids=ids, topk_weights=w, counts=counts, offsets=offsets,
                sorted_to_slot=s2p, slot_to_sorted=p2s, x_sorted=xs, h=h, y_sorted=y,
                h_shared=hs, y_shared=ys, out=out)


def token_outputs(tokens, x, ids, weights, w_gate_up, w_down, scale_input: bool = False,
                  round_h: bool = True, w_shared_gate_up=None, w_shared_down=None):
    """The layer output for a few tokens, one token at a time, with no permutation at all:
    out[t] = sum_j w[t, j] * FFN_{ids[t, j]}(x[t]) (+ shared FFN(x[t])).

    Used for sampled checks at sizes where the whole oracle would be slow; ids/weights come from
    ``route``. Weight blocks are converted to float64 one expert at a time.
    """
    x = np.asarray(x)
    ids = np.asarray(ids)
    weights = np.asarray(weights, dtype=np.float64)
    tokens = [int(t) for t in tokens]
    d = x.shape[1]
    out = np.zeros((len(tokens), d), dtype=np.float64)
    k = ids.shape[1]
    by_expert: dict[int, list] = {}
    for r, t in enumerate(tokens):
        for j in range(k):
            by_expert.setdefault(int(ids[t, j]), []).append((r, t, j))
    for e, items in by_expert.items():
        wgu, wd = _as64(w_gate_up[e]), _as64(w_down[e])
        for r, t, j in items:
            xt = x[t:t + 1].astype(np.float64)
            if scale_input:
                out[r] += swiglu_ffn(xt * weights[t, j], wgu, wd, round_h)[0]
            else:
                out[r] += weights[t, j] * swiglu_ffn(xt, wgu, wd, round_h)[0]
    if w_shared_gate_up is not None:
        xt = x[tokens].astype(np.float64)
        out += swiglu_ffn(xt, _as64(w_shared_gate_up), _as64(w_shared_down), round_h)
    return out


def _as64(a):
    """Widen a numpy array or a CPU torch tensor (including bf16) to a float64 numpy array."""
    if hasattr(a, "detach"):
        return a.detach().to("cpu").double().numpy()
    return np.asarray(a, dtype=np.float64)
