"""Shared helpers for the tests: expert-wise float64 views of device weights for the oracle, the
error measures the parity bar is written in, and the seeded inputs of each workload."""
import numpy as np
import torch

from routing_dispatch_grouped_gb300 import moe

# Parity bar. Outputs: max-abs error over the tensor <= TOL * rms(reference) (2e-2 for bf16
# layers, 1e-4 for fp32 layers). Router weights (fp32, from fp32 logits): relative error
# <= 2e-6, the fp32 rounding of l_j - max (<= 2^-24 |l_j - max|, |l_j - max| < 16 here) plus a few
# ulp from exp, the sum and the division.
TOL = {torch.bfloat16: 2e-2, torch.float32: 1e-4}
W_REL_TOL = 2e-6


def within_one_bf16_ulp(got, ref, rms_frac=1e-4) -> bool:
    """For a tensor both sides round to bf16 on their own (the SwiGLU activation h): the fp32
    value on the GPU and the fp64 value in the oracle may fall on either side of a rounding
    midpoint, so the stored values may differ by one bf16 ulp (at most 2^-7 of the value).
    The absolute slack covers the fp32 accumulation error of gate and up, which does not shrink
    with h where gate * up cancels (about K * 2^-24 * sum |x_i w_i|, below 1e-4 rms here)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    rms = np.sqrt(np.mean(ref * ref)) if ref.size else 0.0
    return bool(np.all(np.abs(got - ref) <= 2.0 ** -7 * np.abs(ref) + rms_frac * rms))


class Expertwise:
    """Indexable of float64 numpy blocks, widened from a [E, ...] tensor one expert at a time."""

    def __init__(self, t: torch.Tensor):
        self.t = t

    def __len__(self):
        return self.t.shape[0]

    def __getitem__(self, e):
        return self.t[e].detach().to("cpu", torch.float64).numpy()


class HostMX:
    """Expert weights [E, K, N] as the MX oracle's dequantized MXFP4 values (blocks of 32 along
    K), quantised on the host from the bf16 values one expert at a time (cached)."""

    def __init__(self, t: torch.Tensor):
        self.t = t
        self.cache = {}

    def __len__(self):
        return self.t.shape[0]

    def __getitem__(self, e):
        from oracle import moe_mx as M
        if e not in self.cache:
            self.cache[e] = M.fake_quant(f64(self.t[e]), M.E2M1, axis=0)
        return self.cache[e]


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def err_rms(got, ref) -> float:
    """max |got - ref| / rms(ref)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if ref.size == 0:
        return 0.0
    rms = np.sqrt(np.mean(ref * ref))
    return float(np.max(np.abs(got - ref)) / max(rms, 1e-300))


def bits16(t: torch.Tensor) -> np.ndarray:
    """Raw bit patterns of a 16-bit tensor (for byte-exact checks)."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy()


def bits(t: torch.Tensor) -> np.ndarray:
    if t.element_size() == 2:
        return bits16(t)
    return t.detach().contiguous().view(torch.int32).cpu().numpy()


def mx_weight_views(mx):
    """The stored codes unpacked to one E2M1 code per element, uint8 [E, K, cols], and the
    E8M0 scales, uint8 [E, ceil(K / 32), cols], in the logical column order (numpy, on the
    host; for tests)."""
    gu = mx.kind == moe.W_GATE_UP
    cols = 2 * mx.N if gu else mx.N
    nbh = (mx.N + 63) // 64
    NB = 2 * nbh if gu else nbh
    KB = (mx.K + 31) // 32
    raw = mx.data.cpu().numpy()
    ncode = mx.E * NB * KB * 1024
    cb = raw[:ncode].reshape(mx.E, NB, KB, 1024)
    sb = raw[ncode:ncode + mx.E * NB * KB * 64].reshape(mx.E, NB, KB, 64)
    m = np.arange(64)[:, None]
    kk = np.arange(32)[None, :]
    mt, r16 = m // 16, m % 16
    hi, lq = r16 // 8, r16 % 8
    ks, kx = kk // 16, kk % 16
    kh, bit = kx // 8, kx % 2
    lane = lq * 4 + (kx % 8) // 2
    byte = (((ks * 4 + mt) * 32 + lane) * 4 + hi + 2 * kh)      # [64, 32]
    nib = (cb[..., byte] >> (4 * bit)) & 15                      # [E, NB, KB, 64, 32]
    # logical column of (nb, m)
    nb = np.arange(NB)[:, None]
    if gu:
        up = nb >= nbh
        c = (nb - np.where(up, nbh, 0)) * 64 + np.arange(64)[None, :]
        col = np.where(c < mx.N, c + np.where(up, mx.N, 0), -1)
    else:
        c = nb * 64 + np.arange(64)[None, :]
        col = np.where(c < mx.N, c, -1)
    codes = np.zeros((mx.E, KB * 32, cols), dtype=np.uint8)
    scales = np.zeros((mx.E, KB, cols), dtype=np.uint8)
    for b in range(NB):
        ok = col[b] >= 0
        cs = col[b][ok]
        # nib[:, b] is [E, KB, 64, 32] -> rows kb*32 + kk
        blk = nib[:, b][:, :, ok, :]                               # [E, KB, n, 32]
        codes[:, :, cs] = blk.transpose(0, 1, 3, 2).reshape(mx.E, KB * 32, len(cs))
        scales[:, :, cs] = sb[:, b][:, :, ok]
    return codes[:, :mx.K], scales
