"""Generalized paged attention, cache append and block copy for one GB300 (sm_103a).

The work runs in ``libpagedkv.so`` (hand-written CUDA behind a C ABI, ``include/pagedkv.h``);
this package holds the in-tree build, a thin ctypes binding and the seeded workload generators.
Calls raise if the library has not been built: there is no CPU fallback.
"""
from .pagedkv import (PA_KV_E4M3, PA_KV_SAME, PagedKVError, block_copy, device_status,  # noqa: F401
                      forward_widen_bytes, forward_workspace_size, kitty_record_bytes, kitty_workspace_size, kv_append,
                      kv_quantize_pages,
                      library_path, load_library, pa_forward, pa_forward_kitty,
                      pa_forward_append, pa_forward_no_alloc, set_timing_events, status_names,
                      version)
