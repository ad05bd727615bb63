"""The allocation-free backward entry point, ffa_bwd_noalloc.

Some callers cannot allocate device memory: for example a plugin inside a
runtime that owns every device byte, or code that must not risk an
allocation's device-wide synchronization.  ffa_bwd_noalloc serves them by
keeping its scratch in a fixed array inside the library.  This test calls it
through the C ABI, twice in a row with different gradients, and checks each
result against ffa_bwd (which takes a caller-allocated workspace) and against
the fp64 oracle, within the gradient tolerance of the other tests; the second
call must leave the device's free memory unchanged.  It also checks that a problem whose
scratch would not fit is refused.  This file is collected last so that a run
stopping at the first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest

import oracle as O
import workloads as W
from ffa_testlib import check_grad, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ffa():
    import torch
    assert torch.cuda.is_available()
    import __graft_entry__
    __graft_entry__.build()
    import flexible_mask_flashattention_gb300 as m
    return m


def call_noalloc(lib, q, k, v, out, lse, dout, plan, scale, dq, dk, dv):
    import torch
    sq, hq, d = q.shape
    sk, hkv, _ = k.shape
    return lib.ffa_bwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                               dout.data_ptr(), sq, sk, hq, hkv, d, plan.handle, ctypes.c_float(scale),
                               dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                               torch.cuda.current_stream().cuda_stream)


def test_noalloc_backward_matches_ffa_bwd_twice(ffa):
    import torch
    lib = ffa.load_library()
    S, hq, hkv, d = 700, 4, 2, 128
    scale = 1.0 / np.sqrt(d)
    sl = W.random_slices(21, S, S, max_segments=4, max_pieces=4)
    t = W.make_tensors(S, hq, hkv, d, 31)
    q, k, v = (t[n].cuda() for n in ("q", "k", "v"))
    plan = ffa.Plan(sl, S, S)
    out, lse = ffa.fwd(q, k, v, plan, scale)
    for call, seed in enumerate((41, 42)):
        dout_h = W.make_tensors(S, hq, hkv, d, seed)["dout"]
        dout = dout_h.cuda()
        ref = ffa.bwd(q, k, v, out, lse, dout, plan, scale)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        code = call_noalloc(lib, q, k, v, out, lse, dout, plan, scale, dq, dk, dv)
        assert code == 0, f"call {call}: status {code}"
        plan.check_status()
        torch.cuda.synchronize()
        if call == 1:   # the first call may load the library's module (and its array); a warmed call allocates nothing
            assert torch.cuda.mem_get_info()[0] == free_before, "the warmed call changed the device's free memory"
        for name, got, want in (("dq", dq, ref[0]), ("dk", dk, ref[1]), ("dv", dv, ref[2])):
            check_grad(to_np(got), to_np(want).astype(np.float64), f"call {call} {name}")
        # and directly against the fp64 oracle
        r_dq, r_dk, r_dv = O.attention_backward(t["q"], t["k"], t["v"], dout_h, sl, scale)
        for name, got, want in (("dq", dq, r_dq), ("dk", dk, r_dk), ("dv", dv, r_dv)):
            check_grad(to_np(got), want, f"call {call} {name} vs oracle")


def test_noalloc_refuses_oversized_problems(ffa):
    import torch
    lib = ffa.load_library()
    limit = 64 << 20
    S, hq, d = 4096, 32, 128      # 64 MiB of fp32 dq accumulator alone
    assert ffa.bwd_workspace_size(S, S, hq, hq, d) > limit
    plan = ffa.Plan([], S, S)
    x = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    code = lib.ffa_bwd_noalloc(x.data_ptr(), x.data_ptr(), x.data_ptr(), x.data_ptr(), x.data_ptr(), x.data_ptr(),
                               S, S, hq, hq, d, plan.handle, ctypes.c_float(1.0), x.data_ptr(), x.data_ptr(),
                               x.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert code == 4   # FFA_ERR_UNSUPPORTED, nothing launched
