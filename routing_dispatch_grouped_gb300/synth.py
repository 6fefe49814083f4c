"""Seeded synthetic inputs for the MoE expert layer, shared by the tests, the benchmark and the
oracle's callers.

This module holds no step of the method itself (no routing, dispatch, expert FFN or combine):
only the workload table and a counter-based value generator. Both sides of every parity check
receive tensors made here.

Generator
---------
Element ``i`` of tensor ``name`` under ``seed`` is a function of ``(seed, name, i)`` only, so any
slice can be regenerated on its own and a prefix of a longer tensor equals the shorter tensor.
The value is an Irwin-Hall(8) approximation of a normal draw: eight 16-bit uniform fields come
from four 32-bit integer hashes (the two-round xor-shift-multiply mixer with multiplier
0x45d9f3b), their integer sum is centred, and one multiply by ``sigma / sd`` turns it into a
float64. Every step before that multiply is exact integer arithmetic (products stay below 2**59,
so int64 never overflows) and the multiply and the later fp64->fp32->bf16 conversions are
correctly rounded, so CPU and CUDA produce the same bits.

Workloads
---------
The five configurations below are the expert-layer shapes of the models the Expert parallelism
pages name (gpt-oss-120b, Qwen3-30B-A3B in "Token dispatch", Llama-4 in the intro) plus a
Mixtral-8x7B shape and a decode shape; no trained weights or datasets exist here, so seeded
synthetic tensors with those shapes stand in for them.
"""
from __future__ import annotations

import dataclasses
import math
import zlib

import torch

_M32 = 0xFFFFFFFF
_MUL = 0x45D9F3B
# Irwin-Hall(8) of 16-bit fields: mean 8 * 65535 / 2, variance 8 * (65536**2 - 1) / 12.
_IH_MEAN = 262140
_IH_SD = math.sqrt(8.0 * (65536.0 ** 2 - 1.0) / 12.0)
_CHUNK = 1 << 24


def _mix32_int(x: int) -> int:
    x &= _M32
    x = (((x >> 16) ^ x) * _MUL) & _M32
    x = (((x >> 16) ^ x) * _MUL) & _M32
    return ((x >> 16) ^ x) & _M32


def _mix32(x: torch.Tensor) -> torch.Tensor:
    # x: int64 holding values in [0, 2**32); each product is < 2**32 * 2**27 and cannot overflow.
    x = (((x >> 16) ^ x) * _MUL) & _M32
    x = (((x >> 16) ^ x) * _MUL) & _M32
    return (x >> 16) ^ x


def _keys(seed: int, name: str):
    base = zlib.crc32(f"{seed}:{name}".encode())
    ks = []
    for j in range(4):
        a = _mix32_int(base ^ _mix32_int(0x9E3779B9 * (2 * j + 1)))
        b = _mix32_int(a ^ _mix32_int(0x85EBCA6B * (2 * j + 2)))
        ks.append((a, b))
    return ks


def normal_f64(seed: int, name: str, start: int, count: int, sigma: float,
               device="cpu") -> torch.Tensor:
    """float64 values of elements [start, start+count) of stream ``name``, ~N(0, sigma^2)."""
    assert start >= 0 and count >= 0 and start + count <= (1 << 32), "index space is 32-bit"
    ks = _keys(seed, name)
    scale = float(sigma) / _IH_SD
    i = torch.arange(start, start + count, dtype=torch.int64, device=device)
    s = torch.zeros_like(i)
    for a, b in ks:
        h = _mix32(_mix32(i ^ a) ^ b)
        s += (h & 0xFFFF) + (h >> 16)
    return (s - _IH_MEAN).to(torch.float64) * scale


def fill_normal(out: torch.Tensor, seed: int, name: str, sigma: float) -> torch.Tensor:
    """Fill a contiguous fp32/bf16/fp64 tensor in place, chunk by chunk, on its own device."""
    assert out.is_contiguous()
    flat = out.view(-1)
    n = flat.numel()
    for s in range(0, n, _CHUNK):
        c = min(_CHUNK, n - s)
        v = normal_f64(seed, name, s, c, sigma, device=out.device)
        if out.dtype == torch.float64:
            flat[s:s + c] = v
        else:
            # fixed two-step rounding: fp64 -> fp32 (RNE), then fp32 -> bf16 (RNE) when needed
            flat[s:s + c] = v.to(torch.float32).to(out.dtype)
    return out


def normal(shape, dtype, seed: int, name: str, sigma: float, device="cpu") -> torch.Tensor:
    out = torch.empty(tuple(shape), dtype=dtype, device=device)
    return fill_normal(out, seed, name, sigma)


# --------------------------------------------------------------------------------------------
# Workload table
# --------------------------------------------------------------------------------------------

SOFTMAX, SIGMOID = 0, 1


@dataclasses.dataclass(frozen=True)
class MoEConfig:
    name: str
    T: int
    d: int
    E: int
    k: int
    I: int
    dtype: torch.dtype
    score_fn: int = SOFTMAX
    renormalize: bool = True
    scale_input: bool = False       # router score multiplies the expert input (Llama-4 form)
    I_shared: int = 0               # 0 = no always-on shared expert
    bias: str = "none"              # "none" | "normal0.5" | "zipf1.2"
    seed: int = 0

    @property
    def R(self) -> int:
        return self.T * self.k

    def with_T(self, T: int) -> "MoEConfig":
        return dataclasses.replace(self, T=T, name=f"{self.name.split('@')[0]}@T{T}")

    def expert_flops(self) -> int:
        """6*d*I per routed row (gate, up, down), plus 6*d*I_shared per token."""
        return 6 * self.d * self.I * self.R + 6 * self.d * self.I_shared * self.T


CONFIGS = {
    "tiny_fp32": MoEConfig("tiny_fp32", 256, 128, 8, 2, 256, torch.float32),
    "mixtral_8x7b": MoEConfig("mixtral_8x7b", 4096, 4096, 8, 2, 14336, torch.bfloat16),
    "gpt_oss_120b": MoEConfig("gpt_oss_120b", 8192, 2880, 128, 4, 2880, torch.bfloat16,
                              bias="normal0.5"),
    "decode": MoEConfig("decode", 64, 2048, 128, 8, 768, torch.bfloat16),
    "llama4_scout": MoEConfig("llama4_scout", 16384, 5120, 16, 1, 8192, torch.bfloat16,
                              score_fn=SIGMOID, renormalize=False, scale_input=True,
                              I_shared=8192, bias="zipf1.2"),
}
DECODE_T = (1, 8, 64)


# Scale of the Zipf bias. With beta = 1 the seeded Scout-shaped workload sends 40.4% of tokens to
# expert 0; the workload asks for about 30%, and beta = 0.75 (found by bisection on the seeded
# logits, 0.7437 gives 30.0%) gives 30.3%.
ZIPF_BETA = 0.75


def zipf_bias(E: int, s: float = 1.2, beta: float = ZIPF_BETA) -> torch.Tensor:
    """b_e = beta * ln p_e with p_e proportional to (e+1)^-s, normalised over the E experts."""
    p = torch.tensor([(e + 1.0) ** (-s) for e in range(E)], dtype=torch.float64)
    return beta * torch.log(p / p.sum())


def router_bias(cfg: MoEConfig, device="cpu") -> torch.Tensor | None:
    if cfg.bias == "none":
        return None
    if cfg.bias == "normal0.5":
        return normal_f64(cfg.seed, "router_bias", 0, cfg.E, 0.5, device=device)
    if cfg.bias == "zipf1.2":
        return zipf_bias(cfg.E).to(device)
    raise ValueError(cfg.bias)


def make_x(cfg: MoEConfig, device="cpu") -> torch.Tensor:
    return normal((cfg.T, cfg.d), cfg.dtype, cfg.seed, "x", 1.0, device)


def make_router_weight(cfg: MoEConfig, device="cpu") -> torch.Tensor:
    return normal((cfg.d, cfg.E), torch.float32, cfg.seed, "w_router", 0.02, device)


def make_logits(cfg: MoEConfig, x: torch.Tensor, w_router: torch.Tensor) -> torch.Tensor:
    """fp32 router logits: fp32(fp64(x) @ fp64(W_r) + b). An input of the routing step."""
    z = x.to(torch.float64) @ w_router.to(torch.float64)
    b = router_bias(cfg, device=x.device)
    if b is not None:
        z = z + b
    return z.to(torch.float32).contiguous()


def make_weights(cfg: MoEConfig, device="cpu"):
    """Packed gate|up [E, d, 2I] (gate = columns [0, I)) and down [E, I, d]."""
    w_gu = normal((cfg.E, cfg.d, 2 * cfg.I), cfg.dtype, cfg.seed, "w_gate_up", 0.02, device)
    w_dn = normal((cfg.E, cfg.I, cfg.d), cfg.dtype, cfg.seed, "w_down", 0.02, device)
    return w_gu, w_dn


def make_shared_weights(cfg: MoEConfig, device="cpu"):
    if cfg.I_shared == 0:
        return None, None
    Is = cfg.I_shared
    w_gu = normal((cfg.d, 2 * Is), cfg.dtype, cfg.seed, "w_shared_gate_up", 0.02, device)
    w_dn = normal((Is, cfg.d), cfg.dtype, cfg.seed, "w_shared_down", 0.02, device)
    return w_gu, w_dn


def make_inputs(cfg: MoEConfig, device="cpu", weights=True) -> dict:
    x = make_x(cfg, device)
    wr = make_router_weight(cfg, device)
    out = {"x": x, "logits": make_logits(cfg, x, wr)}
    if weights:
        out["w_gate_up"], out["w_down"] = make_weights(cfg, device)
        out["w_shared_gate_up"], out["w_shared_down"] = make_shared_weights(cfg, device)
    return out


def make_y_sorted(R: int, d: int, seed: int = 0, device="cpu") -> torch.Tensor:
    """Synthetic fp32 expert outputs for checking the combine step on its own."""
    return normal((R, d), torch.float32, seed, "y_sorted", 1.0, device)
