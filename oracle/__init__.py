"""Float64 CPU oracle for exact softmax attention -- TEST INFRASTRUCTURE ONLY.

This package is the checker, not the product.  Only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may import
it.  It shares no code with the CUDA path (``exact_io_aware_37_gb300``) and
imports nothing from it; the two meet only through the seeded input
generators, which hold none of the method's arithmetic.

Sources (page title, section):
  [TT]  tensortonic.com "FlashAttention", sections 1-9 (the authority where the
        pages disagree).
  [AIE] wiki.ai-engineering.at "Flash Attention" (naive attention listing,
        online-softmax block, tiling loop -- the tiling loop is wrong as printed,
        see ``attention.tiled_forward_head``).
  [NON] nexusofnerds.com "FlashAttention" (claims only: exactness, causal and
        padding masks, variable-length packing, BF16/FP16).

Pin status of every public function: see the header of ``attention.py``.
"""

from .attention import (  # noqa: F401
    score_matrix,
    forward_head,
    backward_head,
    forward,
    backward,
    forward_varlen,
    backward_varlen,
    forward_rows,
    backward_dq_rows,
    backward_head_blocked,
    online_softmax_row,
    tiled_forward_head,
    cached_score_matrix,
    forward_cached_head,
    forward_cached,
    philox4x32_10,
    dropout_keep,
    forward_head_dropout,
    backward_head_dropout,
    forward_dropout,
    backward_dropout,
)
