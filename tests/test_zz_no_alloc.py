"""moe_dispatch_noalloc: the dispatch entry point for callers that cannot allocate device
memory at the call site (its scratch lives in a fixed array inside the library instead of a
caller workspace). Checked through the C ABI against moe_dispatch on the same inputs, on two
calls in a row (the shared array keeps the previous call's contents, which must not leak into
the next result)."""
import ctypes

import numpy as np
import pytest
import torch

from routing_dispatch_grouped_gb300 import moe, synth

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _noalloc(ids, E, x):
    T, k = ids.shape
    R = T * k
    out = {"counts": torch.full((E,), -7, dtype=torch.int32, device=DEV),
           "offsets": torch.full((E + 1,), -7, dtype=torch.int32, device=DEV),
           "sorted_to_slot": torch.full((R,), -7, dtype=torch.int32, device=DEV),
           "slot_to_sorted": torch.full((R,), -7, dtype=torch.int32, device=DEV),
           "x_sorted": torch.zeros(R, x.shape[1], dtype=x.dtype, device=DEV)}
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    st = moe.lib().moe_dispatch_noalloc(
        p(ids), p(x), moe.BF16 if x.dtype == torch.bfloat16 else moe.F32, T, x.shape[1], E, k,
        p(out["counts"]), p(out["offsets"]), p(out["sorted_to_slot"]), p(out["slot_to_sorted"]),
        p(out["x_sorted"]), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, moe.STATUS.get(st, st)
    return out


def _case(T, E, k, d, seed, dtype):
    rng = np.random.default_rng(seed)
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    x = synth.normal((T, d), dtype, seed, "noalloc_x", 1.0, device=DEV)
    return torch.from_numpy(ids).to(DEV), x


def test_noalloc_dispatch_matches_workspace_dispatch_twice():
    assert torch.cuda.is_available()
    # two different problems back to back: the second must not see the first's scratch
    for (T, E, k, d, seed, dtype) in [(4096, 128, 8, 256, 1, torch.bfloat16),
                                      (777, 16, 2, 136, 2, torch.float32)]:
        ids, x = _case(T, E, k, d, seed, dtype)
        ref = moe.moe_dispatch(ids, E, x=x)
        got = _noalloc(ids, E, x)
        torch.cuda.synchronize()
        for name in ("counts", "offsets", "sorted_to_slot", "slot_to_sorted"):
            assert torch.equal(got[name], ref[name]), name
        assert torch.equal(got["x_sorted"].view(torch.uint8), ref["x_sorted"].view(torch.uint8))


def test_noalloc_dispatch_rejects_sizes_beyond_its_scratch():
    cap = 262144
    E = 256
    T = (cap // E + 1) * 256   # one chunk more than the fixed array holds, with k = 1
    st = moe.lib().moe_dispatch_noalloc(ctypes.c_void_p(0x10000), None, moe.BF16, T, 0, E, 1,
                                        ctypes.c_void_p(0x10000), ctypes.c_void_p(0x10000),
                                        ctypes.c_void_p(0x10000), ctypes.c_void_p(0x10000), None,
                                        None)
    assert st == 2
