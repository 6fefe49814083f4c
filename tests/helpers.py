"""Shared helpers for the tests: expert-wise float64 views of device weights for the oracle, the
error measures the parity bar is written in, and the seeded inputs of each workload."""
import numpy as np
import torch

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
