"""The kernels' failure path on a GB300, without a fault: every wait in the
persistent kernels is bounded, and a wait that runs out records a timeout bit
in a status word, raises its CTA's abort flag so that the CTA's other waits
give up too, and lets the kernel return.  The self-test entry point runs that
code on barriers nothing ever arrives at (about 2 s); the status must show
the timeout, every thread must have given up, and the device must still run
attention correctly afterwards.  A normal run leaves the plan's status word
clear."""
import numpy as np
import pytest

import oracle as O
import workloads as W
from ffa_testlib import check_out_lse, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ffa():
    import torch
    assert torch.cuda.is_available()
    import __graft_entry__
    __graft_entry__.build()
    import flexible_mask_flashattention_gb300 as m
    return m


def test_bounded_wait_times_out_and_the_device_stays_usable(ffa):
    import torch
    status, gave_up = ffa.selftest_bounded_wait()
    assert status == 1 << 4, f"status word {status:#x}"   # the "other wait" timeout bit, nothing else
    assert gave_up == 64
    # the context is intact: a forward right after matches the oracle, and its plan reports no failure
    S = 300
    sl = W.random_slices(7, S, S)
    t = W.make_tensors(S, 4, 2, 128, 8, with_dout=False)
    plan = ffa.Plan(sl, S, S)
    out, lse = ffa.fwd(t["q"].cuda(), t["k"].cuda(), t["v"].cuda(), plan, 0.1)
    plan.check_status()
    torch.cuda.synchronize()
    r_out, r_lse = O.attention_forward(t["q"], t["k"], t["v"], sl, 0.1)
    check_out_lse(to_np(out), to_np(lse), r_out, r_lse, "forward after the self-test")
