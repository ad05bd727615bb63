"""GB300 (sm_103a) Flex-Flash-Attention: fused softmax attention, forward and
backward, over AttnSlice masks, behind the C ABI of ``include/ffa.h``.

    plan = Plan(slices, seqlen_q, seqlen_k)      # block metadata on the GPU
    out, lse = fwd(q, k, v, plan, scale)
    dq, dk, dv = bwd(q, k, v, out, lse, dout, plan, scale)
    fwd_accumulate(q, k, v, plan_b, scale, out, lse)   # merge another key set in by LSE
    out, lse = lse_combine(out_a, lse_a, out_b, lse_b)
    out, lse = fwd_sink(q, k, v, plan, scale, sink)    # per-head attention-sink logits
    dq, dk, dv, dsink = bwd_sink(q, k, v, out, lse, dout, plan, scale, sink)
    bucket, chunk_area, bucket_area = dispatch_solve(slices, seqlen, seqlen, chunk_size, cp_size)   # host only
"""
from ._lib import (FFAError, MASK_BI_CAUSAL, MASK_CAUSAL, MASK_FULL, MASK_INV_CAUSAL, Plan, bwd,
                   bwd_sink, bwd_workspace_size, dispatch_solve, fwd, fwd_accumulate, fwd_sink, load_library,
                   lse_combine, range_gather, range_scatter_reduce, selftest_bounded_wait)

__all__ = ["FFAError", "Plan", "fwd", "fwd_accumulate", "fwd_sink", "lse_combine", "bwd", "bwd_sink",
           "bwd_workspace_size", "dispatch_solve", "range_gather", "range_scatter_reduce", "load_library",
           "selftest_bounded_wait",
           "MASK_FULL", "MASK_CAUSAL", "MASK_INV_CAUSAL", "MASK_BI_CAUSAL"]
