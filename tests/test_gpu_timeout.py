"""The give-up path of the tensor-core FFN kernels' bounded waits.

With the wait limit set to 1 ns, a kernel's roles give up at their first wait
that does not succeed at once: each kernel must then let what it already
issued finish, free its tensor memory, report MOE_STATUS_TIMEOUT in the call's
status word and return. The context must stay usable: with the default limit
restored, the next call matches the oracle and reports nothing.
No GPU fault is involved: the waits that run out are the kernels' own
mbarrier waits on their other roles, or (one token) the one-kernel decode
FFN's waits for the other CTAs' FC1 work (its per-expert counters).
"""
import numpy as np
import pytest
import torch

from gpu_util import DEV, assert_close_rel_max, layer_tolerance, need_gpu, to_dev, to_np64
from moe_inputs import make_layer_inputs
from oracle import ffn

pytestmark = pytest.mark.gpu


# prefill pair kernels; decode weight-streaming kernels; the one-kernel decode FFN's counter waits
@pytest.mark.parametrize("T", [600, 8, 1])
def test_expired_waits_report_timeout_and_leave_the_context_usable(T):
    moe = need_gpu()
    H, I, E, k = 256, 256, 8, 2
    d = make_layer_inputs(T=T, H=H, I=I, E=E, k=k, dtype="bf16", logits="distinct", seed=21)
    args = (to_dev(d["hidden"], "bf16"), torch.from_numpy(d["logits"]).to(DEV), to_dev(d["w13"], "bf16"),
            to_dev(d["w2"], "bf16"), k, True)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    prev = moe.set_wait_limit_ns(1)
    try:
        assert prev == 2_000_000_000
        moe.moe_layer_forward(*args, status=st)
        torch.cuda.synchronize()
    finally:
        assert moe.set_wait_limit_ns(0) == 1          # back to the default
    assert int(st.item()) & moe.MOE_STATUS_TIMEOUT
    st2 = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = moe.moe_layer_forward(*args, status=st2)
    torch.cuda.synchronize()
    assert int(st2.item()) == 0
    ref = ffn.layer_forward(d["logits"], d["hidden"], d["w13"], d["w2"], k, True, "bf16")["out"]
    assert_close_rel_max(to_np64(out), ref, layer_tolerance("bf16"), "after the timed-out call")
    assert moe.set_wait_limit_ns(0) == 2_000_000_000
