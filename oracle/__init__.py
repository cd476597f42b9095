"""Plain, slow CPU oracle for causal grouped-query attention (TEST INFRASTRUCTURE).

Only the test-suite, the smoke check and the benchmark's CPU-baseline leg may
import this package.  The CUDA product path never calls it, and it shares no
code, table or helper with the CUDA path: both sides receive the same seeded
inputs from the ``synth`` package and nothing else.

Everything here is numpy in float64, written for a reader who checks it
against the pages by eye: the full score matrix is materialised, the causal
mask is an explicit boolean matrix, and grouped-query heads are expanded with
an explicit ``np.repeat``.  There is no blocking, fusion or reordering.

Every function is pinned by ``tests/test_oracle_pins.py`` against closed forms,
brute-force scalar loops, a library routine and hand-derived fixtures under
``tests/golden``; no part of the oracle is "parity unpinned".
"""

from .attention import (  # noqa: F401
    visible_mask,
    prefill,
    prefill_rows,
    attend,
    fp16_from_bits,
    unpack_coef_word,
    dequant_int4_row,
    dequant_int4_rows,
    fp8_e4m3_value,
    dequant_fp8_rows,
    paged_row_index,
    gather_paged_rows,
    num_splits,
    decode_split_partials,
    decode_unsplit,
    lse_merge,
    lse_merge_bwd,
    decode,
    decode_mq_split_partials,
    decode_mq,
    prefill_paged_varlen,
)
