"""CPU oracle for grouped-query attention over a KV cache (test infrastructure).

This package is test infrastructure, not product code.  Only the test suite,
``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl reference``
legs of ``bench.py`` may import it.  It shares no code with the CUDA library
and imports nothing from it.
"""

from .gqa_oracle import (  # noqa: F401
    repeat_kv,
    visible_mask,
    attention,
    dequant_q4,
    attention_q4,
    paged_to_contiguous,
    append_paged,
    attention_paged,
    quantize_q4,
    attention_q4_residual,
)
