"""CPU oracle for the block-scaled low-precision form of the expert layer (MX formats).

TEST INFRASTRUCTURE ONLY, like ``moe_oracle``: only the tests, the smoke check and the
benchmark's CPU-baseline leg may import it; the CUDA package never does.

The pages name 8-bit activations times 4-bit weights with block scales as the low-precision
expert variant for the newest GPUs ("Expert parallelism", the Mega MoE fused kernel paragraph);
they give no format details, so this module follows the public OCP Microscaling (MX)
specification v1.0 (reading stated in each function):
  - a block is 32 consecutive elements along the reduction axis K; the block shares one E8M0
    scale X = 2^s (s in [-127, 127]; code s + 127);
  - elements are FP8 E4M3 (activations: x and the SwiGLU activation h) or FP4 E2M1 (expert
    weights);
  - quantisation: s = floor(log2(max |v|)) - emax_elem (emax 8 for E4M3, 2 for E2M1), clamped to
    [-127, 127] (s = -127 for an all-zero block); each element is v / X rounded to nearest even
    in the element format and saturated at its largest finite value (448 for E4M3, 6 for E2M1);
  - a block shorter than 32 (the end of a K that is not a multiple of 32) uses its own elements.
The quantisation decisions are taken on the value as stored: bf16 x and weights (exact in
float64), and the fp32 SwiGLU activation h, the layer's one computed quantised value.

Layer (``mx_forward``): route and dispatch as ``moe_oracle``; x_sorted quantised to MXFP8 along d;
gate/up with MXFP4 W_gate_up (blocks along d); h = SiLU(g) u quantised to MXFP8 along I (instead
of the bf16 rounding of the bf16 layer); down with MXFP4 W_down (blocks along I); y and the
combine exact (float64), as in ``moe_oracle``.
"""
from __future__ import annotations

import numpy as np

from oracle import moe_oracle as fwd

BLOCK = 32
E4M3, E2M1 = "e4m3", "e2m1"
EMAX = {E4M3: 8, E2M1: 2}
MAXV = {E4M3: 448.0, E2M1: 6.0}


# ----------------------------------------------------------------------------------------------
# element formats, from their definitions
# ----------------------------------------------------------------------------------------------
def e2m1_value(code) -> np.ndarray:
    """FP4 E2M1: bit 3 sign, bits 1-2 exponent (bias 1), bit 0 mantissa; exponent 0 is
    subnormal (0 or 0.5). Magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6; no inf or NaN."""
    c = np.asarray(code, dtype=np.int64)
    e, m = (c >> 1) & 3, c & 1
    mag = np.where(e == 0, 0.5 * m, (1.0 + 0.5 * m) * np.exp2(e - 1.0))
    return np.where(c & 8, -mag, mag)


def e4m3_value(code) -> np.ndarray:
    """FP8 E4M3 (OCP): bit 7 sign, bits 3-6 exponent (bias 7), bits 0-2 mantissa; exponent 0 is
    subnormal (m/8 * 2^-6); S.1111.111 is NaN (never produced here), no infinities, largest
    finite 448."""
    c = np.asarray(code, dtype=np.int64)
    e, m = (c >> 3) & 15, c & 7
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return np.where(c & 128, -mag, mag)


def _grid(fmt):
    """All non-negative finite values of the element format with their codes, ascending."""
    codes = np.arange(8 if fmt == E2M1 else 127)  # E4M3: 0..126 (127 is NaN)
    vals = e2m1_value(codes) if fmt == E2M1 else e4m3_value(codes)
    return vals, codes


def encode_rne(v, fmt) -> np.ndarray:
    """Round |v| to the nearest element value, ties to the even code (the even mantissa),
    saturating at the largest finite value; the sign bit is kept (-0 encodes as 0x8 / 0x80)."""
    v = np.asarray(v, dtype=np.float64)
    vals, codes = _grid(fmt)
    a = np.minimum(np.abs(v), vals[-1])
    i = np.clip(np.searchsorted(vals, a), 1, len(vals) - 1)   # vals[i-1] < a <= vals[i]
    lo, hi = vals[i - 1], vals[i]
    pick_hi = (a - lo > hi - a) | ((a - lo == hi - a) & (codes[i] % 2 == 0))
    pick_hi |= a == hi
    c = np.where(pick_hi, codes[i], codes[i - 1])
    c = np.where(a == 0, 0, c)
    sign = 8 if fmt == E2M1 else 128
    return np.where(np.signbit(v), c | sign, c).astype(np.uint8)


def floor_log2(a) -> np.ndarray:
    """floor(log2(a)) for a > 0, exactly (from the binary exponent, no logarithm)."""
    _, e = np.frexp(np.asarray(a, dtype=np.float64))   # a = m 2^e, 0.5 <= m < 1
    return e - 1


# ----------------------------------------------------------------------------------------------
# block quantisation along an axis
# ----------------------------------------------------------------------------------------------
def quantize_mx(a, fmt, axis=-1):
    """MX quantisation of `a` in blocks of 32 along `axis`. Returns (codes uint8 with the shape
    of a, scale codes uint8 with ceil(K/32) along axis): scale code = s + 127."""
    a = np.moveaxis(np.asarray(a, dtype=np.float64), axis, -1)
    K = a.shape[-1]
    nb = (K + BLOCK - 1) // BLOCK
    codes = np.zeros(a.shape, dtype=np.uint8)
    scales = np.zeros(a.shape[:-1] + (nb,), dtype=np.uint8)
    for b in range(nb):
        blk = a[..., b * BLOCK:(b + 1) * BLOCK]
        amax = np.max(np.abs(blk), axis=-1)
        s = np.where(amax > 0, floor_log2(np.where(amax > 0, amax, 1.0)) - EMAX[fmt], -127)
        s = np.clip(s, -127, 127)
        scales[..., b] = (s + 127).astype(np.uint8)
        codes[..., b * BLOCK:(b + 1) * BLOCK] = encode_rne(blk / np.exp2(s)[..., None], fmt)
    return np.moveaxis(codes, -1, axis), np.moveaxis(scales, -1, axis)


def dequantize_mx(codes, scales, fmt, axis=-1):
    """Values of MX codes: element value times 2^(scale code - 127)."""
    c = np.moveaxis(np.asarray(codes), axis, -1)
    sc = np.moveaxis(np.asarray(scales, dtype=np.int64), axis, -1)
    v = e2m1_value(c) if fmt == E2M1 else e4m3_value(c)
    s = np.repeat(sc, BLOCK, axis=-1)[..., :c.shape[-1]] - 127
    return np.moveaxis(v * np.exp2(s), -1, axis)


def fake_quant(a, fmt, axis=-1):
    """dequantize_mx(quantize_mx(a))."""
    c, s = quantize_mx(a, fmt, axis)
    return dequantize_mx(c, s, fmt, axis)


# ----------------------------------------------------------------------------------------------
# the layer
# ----------------------------------------------------------------------------------------------
def mx_weights(w, axis):
    """Expert weights (one expert, [K, N]) as MXFP4 along K (axis 0): (codes, scales)."""
    return quantize_mx(np.asarray(w, dtype=np.float64), E2M1, axis=axis)


def mx_swiglu_ffn(xq, wgu, wd, row_scale=None):
    """One expert on MXFP8 rows xq (already dequantized values) with dequantized MXFP4 weights
    wgu [d, 2I], wd [I, d]: h = SiLU(s g) (s u) quantised to MXFP8 along I, y = h_q . wd."""
    I = wgu.shape[1] // 2
    acc = xq @ wgu
    s = np.ones(len(xq)) if row_scale is None else np.asarray(row_scale, dtype=np.float64)
    g, u = s[:, None] * acc[:, :I], s[:, None] * acc[:, I:]
    h = g / (1.0 + np.exp(-g)) * u
    hq = fake_quant(h, E4M3, axis=-1)
    return hq @ wd, h, hq


def mx_forward(x, logits, wgu_deq, wd_deq, k: int, score_fn: int = fwd.SOFTMAX,
               renormalize: bool = True, scale_input: bool = False, wsgu_deq=None,
               wsd_deq=None):
    """The layer with MX numerics. wgu_deq / wd_deq: per-expert dequantized MXFP4 weights
    (indexable by expert, [d, 2I] and [I, d]); wsgu_deq / wsd_deq: the shared expert's, or None.
    Returns the intermediates of moe_oracle.forward plus xq (quantised x rows), h (before its
    quantisation) and hq."""
    x = np.asarray(x, dtype=np.float64)
    E = len(wgu_deq)
    ids, w = fwd.route(logits, k, score_fn, renormalize)
    counts, offsets, s2p, p2s = fwd.dispatch(ids, E)
    xq_tok = fake_quant(x, E4M3, axis=-1)            # quantised once per token
    xs = fwd.permute_rows(xq_tok, s2p, k)
    R, d = xs.shape
    I = np.asarray(wd_deq[0]).shape[0]
    scale = w.reshape(-1)[s2p] if scale_input else None
    y = np.zeros((R, d))
    h = np.zeros((R, I))
    hq = np.zeros((R, I))
    for e in range(E):
        a, b = int(offsets[e]), int(offsets[e + 1])
        if b > a:
            y[a:b], h[a:b], hq[a:b] = mx_swiglu_ffn(
                xs[a:b], np.asarray(wgu_deq[e]), np.asarray(wd_deq[e]),
                None if scale is None else scale[a:b])
    ys = None
    if wsgu_deq is not None:
        ys, _, _ = mx_swiglu_ffn(xq_tok, np.asarray(wsgu_deq), np.asarray(wsd_deq))
    out = fwd.combine(y, p2s, None if scale_input else w, k, ys)
    return dict(topk_ids=ids, topk_weights=w, counts=counts, offsets=offsets, sorted_to_slot=s2p,
                slot_to_sorted=p2s, x_sorted=xs, h=h, hq=hq, y_sorted=y, y_shared=ys, out=out)
