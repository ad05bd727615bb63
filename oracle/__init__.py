"""CPU oracle for the Flex-Flash-Attention hot path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The library in
``flexible_mask_flashattention_gb300`` never imports it and shares no code
with it; both sides only share the seeded input generators in ``workloads``.

Everything here is plain fp64 numpy written from the definitions on the
MagiAttention pages (AttnSlice masks, row softmax, the FLOP and mask-area
formulas, the Full/Partial/Empty block classes and their CSR form), plus
``rows_c``: the same attention definitions as plain C loops over one row at a
time and its allowed keys (``ffa_rows.c``), for sampled checks of 1M-token
problems over every head.
"""
from .ffa_oracle import *  # noqa: F401,F403
