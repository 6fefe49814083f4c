"""The bounded-wait path of a tcgen05 kernel, made to run out on purpose (no GPU fault).

Every mbarrier wait of the tensor-core kernels gives up after a time limit, records
MOE_ERR_TIMEOUT in the call's status word, stops the kernel's other roles, lets its own copies
and MMAs finish, frees its tensor memory and returns. Here the test hook
moe_debug_set_gemm_stall_ns makes the MMA issuer of the 128-row gate_up kernel wait on a barrier
that nothing completes; the test checks that the status word reports the timeout, that the
stream completes, and that the next call on the same context gives the oracle's result."""
import numpy as np
import pytest
import torch

from oracle import moe_oracle as o
from routing_dispatch_grouped_gb300 import moe, synth
from tests.helpers import Expertwise, f64, within_one_bf16_ulp

pytestmark = pytest.mark.gpu
DEV = "cuda"
TIMEOUT = 6


def _case(R, d, I):
    xs = synth.normal((R, d), torch.bfloat16, 3, "tmo_x", 1.0, device=DEV)
    wgu = synth.normal((1, d, 2 * I), torch.bfloat16, 3, "tmo_wgu", 0.05, device=DEV)
    off = torch.tensor([0, R], dtype=torch.int32, device=DEV)
    return xs, wgu, off


@pytest.mark.parametrize("R,d,I", [(64, 128, 128), (700, 512, 384)])
def test_expired_wait_reports_timeout_and_the_context_stays_usable(R, d, I):
    assert torch.cuda.is_available()
    xs, wgu, off = _case(R, d, I)
    ws = torch.zeros(moe.moe_experts_workspace_size(), dtype=torch.uint8, device=DEV)
    moe.lib().moe_debug_set_gemm_stall_ns(2_000_000)   # 2 ms on a barrier nothing completes
    try:
        moe.moe_gate_up_train(xs, off, wgu, workspace=ws)
        torch.cuda.synchronize()   # the kernel ended: the stream completes
    finally:
        moe.lib().moe_debug_set_gemm_stall_ns(0)
    assert moe.moe_read_device_status(ws) == TIMEOUT
    # the same call on the same context, hook off: the oracle's activation, status clear
    ws2 = torch.zeros_like(ws)
    h, ab = moe.moe_gate_up_train(xs, off, wgu, workspace=ws2)
    torch.cuda.synchronize()
    assert moe.moe_read_device_status(ws2) == 0
    ref = o.swiglu_activation(f64(xs), Expertwise(wgu)[0], True)
    assert within_one_bf16_ulp(f64(h), ref)
