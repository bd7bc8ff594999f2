"""CPU oracle for the block-causal attention path (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline and
reference legs may import this package.  It shares no code with the CUDA path.
"""
from .attention import (cache_append, masked_attention, prefill, prefill_piecewise,  # noqa: F401
                        prefix_decode, query_positions, visibility, visible_pairs)
