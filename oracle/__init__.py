"""fp64 CPU oracle for attention over a block-paged KV cache.

TEST INFRASTRUCTURE: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline / reference legs of ``bench.py`` may import this package.  The CUDA
library and its Python binding never do.
"""
from .paged_oracle import (  # noqa: F401
    attend, gather, kv_head_of, kv_write, merge_partials, paged_attention, partial_attend,
    visible_keys,
)
