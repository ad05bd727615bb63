"""GB300 (sm_103a) Flex-Flash-Attention: fused softmax attention, forward and
backward, over AttnSlice masks, behind the C ABI of ``include/ffa.h``.

    plan = Plan(slices, seqlen_q, seqlen_k)      # block metadata on the GPU
    out, lse = fwd(q, k, v, plan, scale)
    dq, dk, dv = bwd(q, k, v, out, lse, dout, plan, scale)
"""
from ._lib import (FFAError, MASK_BI_CAUSAL, MASK_CAUSAL, MASK_FULL, MASK_INV_CAUSAL, Plan, bwd,
                   bwd_workspace_size, fwd, load_library)

__all__ = ["FFAError", "Plan", "fwd", "bwd", "bwd_workspace_size", "load_library", "MASK_FULL", "MASK_CAUSAL",
           "MASK_INV_CAUSAL", "MASK_BI_CAUSAL"]
