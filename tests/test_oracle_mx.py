"""Pins of the MX oracle against something other than itself:
- the element formats' value tables against values worked out by hand from the format
  definitions (E2M1 magnitudes, E4M3's largest finite value, smallest normal and subnormal,
  NaN code), and every code round-tripping;
- E4M3 rounding against PyTorch's float8_e4m3fn conversion (a library routine, round to
  nearest even) on random values and on every midpoint between adjacent codes;
- E2M1 rounding against a plain-Python nearest search with ties to the even code;
- block quantisation on hand-worked blocks (scale choice, saturation, all-zero and short
  blocks) and its error bound (half the element spacing at the block's scale);
- the layer: with x and weights already representable, the gate/up accumulators equal the
  exact layer's, and h is quantised as PyTorch's float8 conversion of h / 2^s quantises it.
"""
import numpy as np
import pytest
import torch

from oracle import moe_mx as M
from oracle import moe_oracle as o


def test_e2m1_table():
    assert list(M.e2m1_value(np.arange(8))) == [0, 0.5, 1, 1.5, 2, 3, 4, 6]
    assert list(M.e2m1_value(np.arange(8, 16))) == [-0.0, -0.5, -1, -1.5, -2, -3, -4, -6]


def test_e4m3_table():
    v = M.e4m3_value(np.arange(256))
    assert v[0x7E] == 448.0 and v[0x08] == 2.0 ** -6 and v[0x01] == 2.0 ** -9
    assert v[0x38] == 1.0 and v[0x3C] == 1.5 and np.isnan(v[0x7F]) and np.isnan(v[0xFF])
    assert v[0xFE] == -448.0
    assert np.all(np.diff(v[:127]) > 0)  # positive codes ascend
    # every value of torch's float8_e4m3fn bit patterns
    t = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    same = np.isnan(t) == np.isnan(v)
    assert np.all(same) and np.array_equal(t[~np.isnan(t)], v[~np.isnan(v)])


@pytest.mark.parametrize("fmt", [M.E4M3, M.E2M1])
def test_codes_round_trip(fmt):
    n = 127 if fmt == M.E4M3 else 8
    codes = np.arange(n)
    vals = M.e4m3_value(codes) if fmt == M.E4M3 else M.e2m1_value(codes)
    assert np.array_equal(M.encode_rne(vals, fmt), codes)
    sign = 128 if fmt == M.E4M3 else 8
    assert np.array_equal(M.encode_rne(-vals[1:], fmt), codes[1:] | sign)


def test_e4m3_rounding_matches_torch():
    rng = np.random.default_rng(0)
    v = np.concatenate([rng.normal(0, 30, 20000), rng.normal(0, 0.01, 5000),
                        rng.uniform(-448, 448, 5000)]).astype(np.float32)
    vals = M.e4m3_value(np.arange(127))
    mids = ((vals[1:] + vals[:-1]) / 2).astype(np.float32)  # exact in fp32
    v = np.concatenate([v, mids, -mids])
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(M.encode_rne(v.astype(np.float64), M.E4M3), ref)


def test_e2m1_rounding_brute_force():
    grid = [0, 0.5, 1, 1.5, 2, 3, 4, 6]

    def nearest(a):
        a = min(abs(a), 6.0)
        best = None
        for c, g in enumerate(grid):
            dist = abs(a - g)
            if best is None or dist < best[0] or (dist == best[0] and c % 2 == 0):
                best = (dist, c)
        return best[1]

    rng = np.random.default_rng(1)
    v = np.concatenate([rng.uniform(-8, 8, 3000), [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 7.0]])
    got = M.encode_rne(v, M.E2M1)
    ref = np.array([nearest(a) | (8 if a < 0 else 0) for a in v], dtype=np.uint8)
    assert np.array_equal(got, ref)
    # ties to even: 0.25 -> 0, 0.75 -> 1 (code 2), 1.25 -> 1, 1.75 -> 2, 2.5 -> 2, 3.5 -> 4, 5 -> 4
    assert list(M.e2m1_value(M.encode_rne([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], M.E2M1))) == \
        [0, 1, 1, 2, 2, 4, 4]


def test_block_quantisation_hand_cases():
    # E2M1, amax 1.0: s = 0 - 2 = -2 (X = 1/4): 1.0 -> 4, 0.5 -> 2, -0.25 -> 1, 0.3 -> 1 (1.2)
    blk = np.zeros(32)
    blk[:4] = [1.0, 0.5, -0.25, 0.3]
    c, s = M.quantize_mx(blk, M.E2M1)
    assert s[0] == 125 and list(M.e2m1_value(c[:4])) == [4.0, 2.0, -1.0, 1.0]
    # amax 7: s = 2 - 2 = 0, 7 saturates to 6
    c, s = M.quantize_mx(np.array([7.0] + [0.0] * 31), M.E2M1)
    assert s[0] == 127 and M.e2m1_value(c[0]) == 6.0
    # E4M3, amax 1.0: s = -8, 1.0 -> 256, 2^-17 -> 2^-9 (smallest subnormal)
    c, s = M.quantize_mx(np.array([1.0, 2.0 ** -17] + [0.0] * 30), M.E4M3)
    assert s[0] == 119 and list(M.e4m3_value(c[:2])) == [256.0, 2.0 ** -9]
    # all-zero block: smallest scale, zero codes; a 5-element tail block scales on its own
    a = np.concatenate([np.full(32, 0.01), [0.0] * 3 + [100.0, -1.0]])
    c, s = M.quantize_mx(a, M.E4M3)
    assert s.shape == (2,) and s[1] == 6 - 8 + 127
    c, s = M.quantize_mx(np.zeros(40), M.E4M3)
    assert list(s) == [0, 0] and not c.any()


@pytest.mark.parametrize("fmt", [M.E4M3, M.E2M1])
def test_quantisation_error_bound(fmt):
    rng = np.random.default_rng(2)
    a = rng.normal(0, 1, (64, 96)) * np.exp2(rng.integers(-20, 20, (64, 1)))
    c, s = M.quantize_mx(a, fmt, axis=1)
    back = M.dequantize_mx(c, s, fmt, axis=1)
    mbits = 3 if fmt == M.E4M3 else 1
    X = np.exp2(np.repeat(s.astype(np.int64), 32, axis=1)[:, :96] - 127)
    q = a / X
    # within half a spacing at the element's own binade (subnormal spacing below it), unless it
    # saturated at the largest value
    e = np.maximum(np.floor(np.log2(np.maximum(np.abs(q), 1e-300))), 1 - (7 if fmt == M.E4M3
                                                                           else 1))
    half = 0.5 * np.exp2(e - mbits) * X
    sat = np.abs(q) > M.MAXV[fmt]
    assert np.all((np.abs(back - a) <= half) | sat)
    # representable values come back exactly
    assert np.array_equal(M.dequantize_mx(*M.quantize_mx(back, fmt, axis=1), fmt, axis=1), back)


def test_layer_on_representable_inputs():
    rng = np.random.default_rng(3)
    T, d, E, k, I = 12, 64, 4, 2, 64
    x = M.fake_quant(rng.normal(0, 1, (T, d)), M.E4M3)
    wgu = [M.fake_quant(rng.normal(0, 0.2, (d, 2 * I)), M.E2M1, axis=0) for _ in range(E)]
    wd = [M.fake_quant(rng.normal(0, 0.2, (I, d)), M.E2M1, axis=0) for _ in range(E)]
    logits = rng.normal(0, 1, (T, E)).astype(np.float32)
    f = M.mx_forward(x, logits, wgu, wd, k)
    ref = o.forward(x, logits, wgu, wd, k, round_h=False)
    # x and the weights are fixed points of their quantisers: the accumulators, hence h, are
    # the exact layer's
    assert np.array_equal(f["x_sorted"], ref["x_sorted"])
    for e in range(E):
        a, b = int(f["offsets"][e]), int(f["offsets"][e + 1])
        acc = ref["x_sorted"][a:b] @ wgu[e]
        h = acc[:, :I] / (1 + np.exp(-acc[:, :I])) * acc[:, I:]
        np.testing.assert_allclose(f["h"][a:b], h, rtol=1e-15, atol=0)
    # h is quantised along I as torch's float8 conversion does it, block scale from its amax.
    # torch rounds an fp32 input once: where rounding h / 2^s to fp32 first moved it across an
    # E4M3 midpoint the two may differ, and only there.
    vals = M.e4m3_value(np.arange(127))
    mids = (vals[1:] + vals[:-1]) / 2
    h = f["h"]
    for r in range(h.shape[0]):
        for b in range(I // 32):
            blk = h[r, 32 * b:32 * b + 32]
            s = np.floor(np.log2(np.abs(blk).max())) - 8
            v = blk / 2.0 ** s
            v32 = v.astype(np.float32)
            q = torch.from_numpy(v32).to(torch.float8_e4m3fn).to(torch.float64).numpy()
            ours = f["hq"][r, 32 * b:32 * b + 32] / 2.0 ** s
            # |v| in (448, 512): the MX conversion saturates at 448 (torch's conversion does not)
            big = np.abs(v) > 448
            assert np.all(ours[big] == np.sign(v[big]) * 448.0)
            for i in np.nonzero((ours != q) & ~big)[0]:
                gap = np.min(np.abs(np.abs(v[i]) - mids))
                assert gap <= abs(float(v32[i]) - v[i]), (r, b, i)
