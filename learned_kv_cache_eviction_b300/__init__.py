"""DMS (Dynamic Memory Sparsification) decode attention for NVIDIA B300.

The compute lives in libdms.so (CUDA, sm_103a; C ABI in include/dms.h);
``dms`` is its Python binding and ``workload`` draws seeded synthetic inputs.
"""
from .dms import (  # noqa: F401
    DmsCache,
    DmsError,
    DmsStepGraph,
    dms_append,
    dms_append_chunk,
    dms_cache_create,
    dms_cache_create_ex,
    dms_cache_destroy,
    dms_cache_lengths,
    dms_cache_slot_positions,
    dms_cache_status,
    dms_decode_attention,
    dms_decode_attention_noalloc,
    dms_prefill,
    dms_step,
    dms_step_graph_create,
    dms_step_graph_destroy,
    dms_step_graph_launch,
    dms_step_host,
    dms_step_host_join,
    load_library,
)
