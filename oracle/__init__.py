"""CPU oracle of the DFlash2 draft + select + verify step.

TEST INFRASTRUCTURE ONLY.  Plain, slow, FP64 (NumPy) restatement of what the
step computes, each function citing the page passage it follows.  Only the
tests, the smoke check in __graft_entry__ and the CPU-baseline leg of bench.py
may import it; the library and its Python binding never do, and share no code
with it.

Pin status: every function here is pinned by a `-m "not gpu"` test against
closed forms, brute force, textbook special cases or the cuRAND library (see
tests/test_oracle_*.py); no function is "parity unpinned".
"""
from . import philox  # noqa: F401
from .dflash2 import (  # noqa: F401
    STATUS_OK, STATUS_INVAL, STATUS_NONFINITE, bf16_to_f64, round_to_bf16, matrix_f64,
    rmsnorm, rope_neox, rope_inv_freq, dyn_conv, block_attention, visible_context_range,
    draft_block, topk, codebook_rows, selector_scores, selector_lattice, walk, verify, step,
    ddtree_build, ddtree_verify,
    advance, block_width, viterbi_path,
)
