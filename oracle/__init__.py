"""CPU oracle for DMS decode attention -- test infrastructure only.

Imported by ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py``; never by the product library or its binding.
"""
from .dms_oracle import (  # noqa: F401
    SlotSimulator,
    decode_attention,
    eviction_decisions,
    kv_token_reads,
    prefill_attention,
    retained_length,
    softmax_attention,
    visibility_mask,
)
