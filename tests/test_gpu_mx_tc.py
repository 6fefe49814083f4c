"""Parity of the MX layer on the block-scaled tensor cores (moe_forward_mx_tc) with the MX
oracle.

The weights' and activations' codes and scales are decoded on the host from the layouts
include/moe.h documents and compared bit for bit with the oracle's quantisation (the decisions
are taken on the same bf16 values on both sides). h is rounded to MXFP8 by the GPU from its fp32
value and by the oracle from its float64 value, so a value on either side of a rounding midpoint
may land one E4M3 step apart (rare; checked elementwise as in the other MX tests); y_sorted and
the layer output are held to the bar of a bf16 layer (2e-2 rms).
"""
import numpy as np
import pytest
import torch

from oracle import moe_mx as M
from oracle import moe_oracle as o
from routing_dispatch_grouped_gb300 import moe, synth
from tests.helpers import HostMX, err_rms, f64

pytestmark = pytest.mark.gpu
DEV = "cuda"
bf16 = torch.bfloat16


@pytest.fixture(scope="module", autouse=True)
def _loaded():
    assert torch.cuda.is_available(), "GPU tests need a GPU"
    moe.lib()


def atom_index(m, j):
    """Byte of (row or column m of a 128 block, K block j of a 128-element chunk) in an atom."""
    return 16 * (m % 32) + 4 * (m // 32) + j


def decode_tc_weights(mx: moe.MxWeights):
    """Codes uint8 [E, K, C] and scales uint8 [E, ceil(K/32), C] from the MX tensor-core
    buffer, read back by the layout rule (not by any library routine)."""
    raw = mx.data.cpu().numpy()
    gu = mx.kind == moe.W_GATE_UP
    E, K, N = mx.E, mx.K, mx.N
    C = 2 * N if gu else N
    Kp = (K + 127) // 128 * 128
    KC = Kp // 128
    cbh = (N + 127) // 128
    CB = 2 * cbh if gu else cbh
    packed = raw[:E * C * Kp // 2].reshape(E, C, Kp // 2)
    lo, hi = packed & 15, packed >> 4
    codes = np.stack([lo, hi], axis=-1).reshape(E, C, Kp)[:, :, :K].transpose(0, 2, 1)
    sf_off = (E * C * Kp // 2 + 1023) // 1024 * 1024
    atoms = raw[sf_off:sf_off + E * CB * KC * 512].reshape(E, CB, KC, 512)
    KB = K // 32
    scales = np.zeros((E, KB, C), dtype=np.uint8)
    for c in range(C):
        half, cc = (1, c - N) if gu and c >= N else (0, c)
        cb, n = half * cbh + cc // 128, cc % 128
        for kb in range(KB):
            scales[:, kb, c] = atoms[:, cb, kb // 4, atom_index(n, kb % 4)]
    return codes, scales, atoms, (CB, KC, cbh)


@pytest.mark.parametrize("kind,E,K,N", [(moe.W_GATE_UP, 3, 256, 160), (moe.W_DOWN, 2, 288, 96),
                                        (moe.W_GATE_UP, 1, 128, 128)])
def test_tc_weight_layout_bit_exact(kind, E, K, N):
    cols = 2 * N if kind == moe.W_GATE_UP else N
    w = synth.normal((E, K, cols), bf16, 0, f"mxtc{kind}{K}", 0.02, device=DEV)
    w[0, 0:32, 0] = 0                      # an all-zero block
    w[0, 32:64, 1] = 7.0 * 2 ** -6         # a block whose values saturate
    mx = moe.quantize_weights_mx_tc(w, kind)
    deq = moe.dequantize_weights_mx_tc(mx)
    torch.cuda.synchronize()
    codes, scales, atoms, (CB, KC, cbh) = decode_tc_weights(mx)
    rc, rs = M.quantize_mx(f64(w), M.E2M1, axis=1)
    assert np.array_equal(scales, rs)
    assert np.array_equal(codes, rc)
    host = HostMX(w)
    for e in range(E):
        assert np.array_equal(f64(deq[e]), host[e])
    # padding: codes past K are zero, scales of padding columns and K blocks are 127
    Kp = KC * 128
    raw = mx.data.cpu().numpy()
    packed = raw[:E * cols * Kp // 2].reshape(E, cols, Kp // 2)
    assert not packed[:, :, K // 2:].any()
    gu = kind == moe.W_GATE_UP
    for cb in range(CB):
        for n in range(128):
            c = (cb % cbh) * 128 + n
            if c >= N:
                for kc in range(KC):
                    assert (atoms[:, cb, kc, atom_index(n, 0):atom_index(n, 0) + 4] == 127).all()
    for kb in range(K // 32, Kp // 32):
        assert (atoms[:, :, kb // 4, [atom_index(n, kb % 4) for n in range(128)]] == 127).all()
    assert gu or CB == cbh


def _padded_rows(counts):
    """Padded row of every sorted row: every expert's rows start at a multiple of 128."""
    poff = np.concatenate([[0], np.cumsum((np.asarray(counts) + 127) // 128 * 128)])
    off = np.concatenate([[0], np.cumsum(counts)])
    rows = np.zeros(int(off[-1]), dtype=np.int64)
    for e in range(len(counts)):
        rows[off[e]:off[e + 1]] = poff[e] + np.arange(counts[e])
    return rows


def decode_rows(codes, atoms, prow, K):
    """MXFP8 values [len(prow), K] of the padded rows prow from codes [Rp, K] and atoms."""
    c = codes.cpu().numpy()[prow, :K]
    a = atoms.cpu().numpy()
    KB = K // 32
    sc = np.zeros((len(prow), KB), dtype=np.int64)
    m = prow % 128
    for kb in range(KB):
        sc[:, kb] = a[prow // 128, kb // 4, atom_index(m, kb % 4)]
    return M.dequantize_mx(c, sc, M.E4M3, axis=1), c, sc


CASES = [  # (name, T, d, E, k, I, score fn, renorm, scaled input, shared I, bias)
    ("one_tile", 128, 256, 1, 1, 128, o.SOFTMAX, True, False, 0, "none"),
    ("mixtral_like", 200, 512, 8, 2, 640, o.SOFTMAX, True, False, 0, "none"),
    # K and N not multiples of 128: zero-filled K tails, half-empty h tiles
    ("ragged_K_N", 150, 288, 16, 4, 224, o.SOFTMAX, True, False, 0, "normal0.5"),
    ("scout_like", 96, 256, 4, 1, 384, o.SIGMOID, False, True, 192, "zipf1.2"),
    ("several_row_tiles", 700, 512, 4, 2, 256, o.SOFTMAX, True, False, 0, "none"),
    ("decode_T1", 1, 1024, 32, 8, 384, o.SOFTMAX, True, False, 0, "none"),
    ("down_ragged_d", 64, 416, 8, 2, 128, o.SOFTMAX, False, False, 0, "none"),
    # most experts receive no rows (no tiles, nothing written for them)
    ("empty_experts", 20, 256, 16, 1, 128, o.SOFTMAX, False, False, 0, "none"),
    # decode batches on the one-kernel layer: d and I not multiples of 128 (a zero-filled last
    # K chunk, a half h block, an odd number of output blocks)
    ("decode_T4_ragged", 4, 416, 16, 4, 224, o.SOFTMAX, True, False, 0, "normal0.5"),
    # more h blocks (64 experts x 5) than SMs: runs of several h blocks of one expert per SM
    ("decode_T16_runs", 16, 512, 64, 8, 640, o.SOFTMAX, True, False, 0, "none"),
    # the routing weight scaling the expert input (SiLU(s g) (s u), combine weight 1)
    ("decode_T8_scaled", 8, 256, 8, 2, 384, o.SIGMOID, False, True, 0, "zipf1.2"),
    # every token on one expert
    ("decode_T3_one_expert", 3, 384, 1, 1, 256, o.SOFTMAX, False, False, 0, "none"),
    # one expert owning every row: several row tiles of one group
    ("one_expert", 300, 256, 1, 1, 256, o.SOFTMAX, True, False, 0, "none"),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_mx_tc_layer_matches_oracle(case):
    name, T, d, E, k, I, fn, renorm, scale, Is, bias = case
    cfg = synth.MoEConfig(name, T, d, E, k, I, bf16, score_fn=fn, renormalize=renorm,
                          scale_input=scale, I_shared=Is, bias=bias)
    inp = synth.make_inputs(cfg, DEV)
    q = lambda w, kind: moe.quantize_weights_mx_tc(w, kind) if w is not None else None
    mgu, mdn = q(inp["w_gate_up"], moe.W_GATE_UP), q(inp["w_down"], moe.W_DOWN)
    msgu, msdn = q(inp["w_shared_gate_up"], moe.W_GATE_UP), q(inp["w_shared_down"], moe.W_DOWN)
    flags = (moe.RENORMALIZE if renorm else 0) | (moe.SCALE_INPUT if scale else 0)
    out, ids, w, ws = moe.moe_forward_mx_tc(inp["x"], inp["logits"], mgu, mdn, k, fn, flags,
                                            msgu, msdn)
    torch.cuda.synchronize()
    assert moe.moe_read_device_status(ws) == 0
    hgu, hdn = HostMX(inp["w_gate_up"]), HostMX(inp["w_down"])
    sh = {}
    if Is:
        sh = dict(wsgu_deq=HostMX(inp["w_shared_gate_up"][None])[0],
                  wsd_deq=HostMX(inp["w_shared_down"][None])[0])
    ref = M.mx_forward(f64(inp["x"]), inp["logits"].cpu().numpy(), hgu, hdn, k, fn, renorm,
                       scale, **sh)
    assert np.array_equal(ids.cpu().numpy(), ref["topk_ids"])
    v = moe.mx_tc_workspace_views(ws, T, d, E, k, I, Is)
    for n_ in ("counts", "offsets", "sorted_to_slot", "slot_to_sorted"):
        assert np.array_equal(v[n_].cpu().numpy(), ref[n_]), n_
    prow = _padded_rows(ref["counts"])
    # x: the MXFP8 codes and scales of each routed row, bit for bit
    xq, xc, xs = decode_rows(v["x_codes"], v["x_sf"], prow, d)
    rc, rs = M.quantize_mx(f64(inp["x"])[ref["sorted_to_slot"] // k], M.E4M3, axis=1)
    assert np.array_equal(xc, rc)
    assert np.array_equal(xs, rs)
    assert np.array_equal(xq, ref["x_sorted"])
    # h: MXFP8 values decoded from codes and atoms; one E4M3 step apart where the GPU's fp32 h
    # and the oracle's float64 h straddle a rounding midpoint
    hg, _, _ = decode_rows(v["h_codes"], v["h_sf"], prow, I)
    hr = ref["hq"]
    off = np.abs(hg - hr) > 0
    assert off.mean() <= 2e-3, off.mean()
    assert np.all(np.abs(hg - hr)[off] <= 2.0 ** -3 * np.maximum(np.abs(hg), np.abs(hr))[off]
                  + 2.0 ** -9 * np.abs(hr).max())
    if moe.moe_forward_mx_tc_kernel_count(T, d, k, I, Is) > 1:  # the one-kernel layer keeps no y
        assert err_rms(f64(v["y_sorted"]), ref["y_sorted"]) <= 2e-2
    if Is:
        hsg, _, _ = decode_rows(v["sh_codes"], v["sh_sf"], np.arange(T), Is)
        xs_tok = f64(inp["x"])
        _, _, hsq_ref = M.mx_swiglu_ffn(M.fake_quant(xs_tok, M.E4M3, axis=-1), sh["wsgu_deq"],
                                        sh["wsd_deq"])
        offs = np.abs(hsg - hsq_ref) > 0
        assert offs.mean() <= 2e-3
        assert err_rms(f64(v["y_shared"]), ref["y_shared"]) <= 2e-2
    e = err_rms(f64(out), ref["out"])
    assert e <= 2e-2, e


@pytest.mark.parametrize("name", ["mixtral_8x7b"])
def test_mx_tc_full_size(name):
    """The Mixtral-shaped workload the benchmark times the MX layer on, at full size, every
    token, against the MX oracle's whole layer (x codes and scales bit for bit, h within one
    E4M3 step where rounding midpoints straddle, y_sorted and the output within the bar). The
    oracle quantises every expert's weights block by block in plain numpy (about a minute
    here; the 128-expert and Scout shapes would take several), so the other shapes are
    covered at reduced sizes above."""
    cfg = synth.CONFIGS[name]
    T, d, E, k, I, Is = cfg.T, cfg.d, cfg.E, cfg.k, cfg.I, cfg.I_shared
    inp = synth.make_inputs(cfg, DEV)
    q = lambda w, kind: moe.quantize_weights_mx_tc(w, kind) if w is not None else None
    mgu, mdn = q(inp["w_gate_up"], moe.W_GATE_UP), q(inp["w_down"], moe.W_DOWN)
    msgu, msdn = q(inp["w_shared_gate_up"], moe.W_GATE_UP), q(inp["w_shared_down"], moe.W_DOWN)
    flags = (moe.RENORMALIZE if cfg.renormalize else 0) | (moe.SCALE_INPUT if cfg.scale_input
                                                           else 0)
    out, ids, w, ws = moe.moe_forward_mx_tc(inp["x"], inp["logits"], mgu, mdn, k, cfg.score_fn,
                                            flags, msgu, msdn)
    torch.cuda.synchronize()
    assert moe.moe_read_device_status(ws) == 0
    del mgu, mdn, msgu, msdn
    sh = {}
    if Is:
        sh = dict(wsgu_deq=HostMX(inp["w_shared_gate_up"][None])[0],
                  wsd_deq=HostMX(inp["w_shared_down"][None])[0])
    ref = M.mx_forward(f64(inp["x"]), inp["logits"].cpu().numpy(), HostMX(inp["w_gate_up"]),
                       HostMX(inp["w_down"]), k, cfg.score_fn, cfg.renormalize,
                       cfg.scale_input, **sh)
    assert np.array_equal(ids.cpu().numpy(), ref["topk_ids"])
    v = moe.mx_tc_workspace_views(ws, T, d, E, k, I, Is)
    prow = _padded_rows(ref["counts"])
    xq, _, _ = decode_rows(v["x_codes"], v["x_sf"], prow, d)
    assert np.array_equal(xq, ref["x_sorted"])
    hg, _, _ = decode_rows(v["h_codes"], v["h_sf"], prow, I)
    hr = ref["hq"]
    off = np.abs(hg - hr) > 0
    assert off.mean() <= 2e-3, off.mean()
    assert np.all(np.abs(hg - hr)[off] <= 2.0 ** -3 * np.maximum(np.abs(hg), np.abs(hr))[off]
                  + 2.0 ** -9 * np.abs(hr).max())
    assert err_rms(f64(v["y_sorted"]), ref["y_sorted"]) <= 2e-2
    if Is:
        assert err_rms(f64(v["y_shared"]), ref["y_shared"]) <= 2e-2
    e = err_rms(f64(out), ref["out"])
    assert e <= 2e-2, e


def test_mx_tc_steps_equal_the_layer():
    """The step entry points (rows, gate_up, down) give the layer's own intermediates, bit for
    bit, when called one by one on its dispatch."""
    cfg = synth.MoEConfig("steps", 300, 512, 8, 2, 384, bf16, bias="normal0.5")
    T, d, E, k, I = cfg.T, cfg.d, cfg.E, cfg.k, cfg.I
    inp = synth.make_inputs(cfg, DEV)
    mgu = moe.quantize_weights_mx_tc(inp["w_gate_up"], moe.W_GATE_UP)
    mdn = moe.quantize_weights_mx_tc(inp["w_down"], moe.W_DOWN)
    out, ids, w, ws = moe.moe_forward_mx_tc(inp["x"], inp["logits"], mgu, mdn, k)
    torch.cuda.synchronize()
    v = moe.mx_tc_workspace_views(ws, T, d, E, k, I, 0)
    R, Rp = T * k, v["Rp"]
    xc = torch.zeros_like(v["x_codes"])
    xs = torch.zeros_like(v["x_sf"])
    hc = torch.zeros_like(v["h_codes"])
    hs = torch.zeros_like(v["h_sf"])
    y = torch.zeros_like(v["y_sorted"])
    moe.mx_tc_rows(inp["x"], ids, v["slot_to_sorted"], v["offsets"], E, xc, xs)
    g = moe.moe_gate_up_mx_tc(xc, xs, v["offsets"], mgu, R, hc, hs)
    moe.moe_down_mx_tc(hc, hs, v["offsets"], mdn, R, y, g)
    torch.cuda.synchronize()
    assert moe.moe_read_device_status(g) == 0
    counts = v["counts"].cpu().numpy()
    prow = _padded_rows(counts)
    assert torch.equal(xc[prow], v["x_codes"][prow])
    assert torch.equal(hc[prow], v["h_codes"][prow])
    assert torch.equal(y, v["y_sorted"])
    a_ref, a_got = decode_rows(v["h_codes"], v["h_sf"], prow, I)[0], decode_rows(hc, hs, prow, I)[0]
    assert np.array_equal(a_ref, a_got)


def test_mx_tc_empty_batch_is_a_noop():
    cfg = synth.MoEConfig("empty", 8, 256, 4, 2, 128, bf16)
    inp = synth.make_inputs(cfg, DEV)
    mgu = moe.quantize_weights_mx_tc(inp["w_gate_up"], moe.W_GATE_UP)
    mdn = moe.quantize_weights_mx_tc(inp["w_down"], moe.W_DOWN)
    x0, lg0 = inp["x"][:0], inp["logits"][:0]
    out, ids, w, ws = moe.moe_forward_mx_tc(x0, lg0, mgu, mdn, cfg.k)
    torch.cuda.synchronize()
    assert out.shape == (0, cfg.d) and ids.shape == (0, cfg.k)


def test_mx_tc_mixtral_cut_to_4_experts():
    """The Mixtral shape with 4 experts and 2048 tokens: inputs larger than the L2 (0.24 GB of
    MXFP4 weights), a few GB on the device; the case the kernel's profile summary is taken on.
    Routing, x codes and scales bit for bit, the output within the bar."""
    import dataclasses
    cfg = dataclasses.replace(synth.CONFIGS["mixtral_8x7b"].with_T(2048), E=4)
    T, d, E, k, I = cfg.T, cfg.d, cfg.E, cfg.k, cfg.I
    inp = synth.make_inputs(cfg, DEV)
    mgu = moe.quantize_weights_mx_tc(inp["w_gate_up"], moe.W_GATE_UP)
    mdn = moe.quantize_weights_mx_tc(inp["w_down"], moe.W_DOWN)
    out, ids, w, ws = moe.moe_forward_mx_tc(inp["x"], inp["logits"], mgu, mdn, k)
    torch.cuda.synchronize()
    assert moe.moe_read_device_status(ws) == 0
    ref = M.mx_forward(f64(inp["x"]), inp["logits"].cpu().numpy(), HostMX(inp["w_gate_up"]),
                       HostMX(inp["w_down"]), k)
    assert np.array_equal(ids.cpu().numpy(), ref["topk_ids"])
    v = moe.mx_tc_workspace_views(ws, T, d, E, k, I, 0)
    xq, _, _ = decode_rows(v["x_codes"], v["x_sf"], _padded_rows(ref["counts"]), d)
    assert np.array_equal(xq, ref["x_sorted"])
    assert err_rms(f64(v["y_sorted"]), ref["y_sorted"]) <= 2e-2
    assert err_rms(f64(out), ref["out"]) <= 2e-2


@pytest.mark.parametrize("T,E,k", [(600, 8, 2), (8, 128, 8), (1, 128, 8)],
                         ids=["chain_T600", "one_kernel_T8", "one_kernel_T1"])
def test_mx_tc_is_deterministic_and_replays_in_a_graph(T, E, k):
    """Every sum of the tensor-core MX layer has a fixed order: two calls give the same bits, and
    the call captured once in a CUDA graph (no host synchronisation inside) replays to them; on
    the multi-kernel chain and on the one-kernel decode layer."""
    cfg = synth.MoEConfig("graph", T, 512, E, k, 384, bf16, bias="normal0.5")
    assert (moe.moe_forward_mx_tc_kernel_count(T, 512, k, 384) == 1) == (T <= 16)
    inp = synth.make_inputs(cfg, DEV)
    mgu = moe.quantize_weights_mx_tc(inp["w_gate_up"], moe.W_GATE_UP)
    mdn = moe.quantize_weights_mx_tc(inp["w_down"], moe.W_DOWN)
    out1, ids, w, ws = moe.moe_forward_mx_tc(inp["x"], inp["logits"], mgu, mdn, cfg.k)
    out2 = torch.empty_like(out1)
    moe.moe_forward_mx_tc(inp["x"], inp["logits"], mgu, mdn, cfg.k, out=out2, topk_ids=ids,
                          topk_weights=w, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))
    out3 = torch.zeros_like(out1)
    graph = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            moe.moe_forward_mx_tc(inp["x"], inp["logits"], mgu, mdn, cfg.k, out=out3,
                                  topk_ids=ids, topk_weights=w, workspace=ws, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(2):
        out3.zero_()
        graph.replay()
    torch.cuda.synchronize()
    assert moe.moe_read_device_status(ws) == 0
    assert torch.equal(out1.view(torch.int16), out3.view(torch.int16))
