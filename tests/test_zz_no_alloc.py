"""pa_forward_no_alloc: attention for callers that cannot allocate device memory (a plug-in
inside an engine whose allocator owns all device memory, a loop that must not call cudaMalloc or
cudaFree).  The call uses the library's own fixed-size scratch; it must give the same results as
pa_forward with a caller-allocated workspace, call after call, and refuse batches whose scratch
would not fit.

This file is collected last on purpose: a run that stops at the first failure has run every
other test before it."""
import ctypes

import numpy as np
import pytest
import torch

import paged_kv_cache_generalized_gb300 as pkg
from paged_kv_cache_generalized_gb300 import pagedkv as pk
from paged_kv_cache_generalized_gb300 import workloads as W

from gpu_util import as_f64, assert_close, batch_to_dev


def _no_alloc_call(b, d, out):
    """Calls the C entry point directly with plain pointers."""
    lib = pk.load_library()
    dims = pk.forward_dims(d["q"], d["k"], d["bt"], d["ctx"])
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    ptr = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    return lib.pa_forward_no_alloc(ctypes.byref(dims), ptr(d["q"]), ptr(d["k"]), ptr(d["v"]),
                                   ptr(d["bt"]), ptr(d["ctx"]), ptr(d["ql"]),
                                   ctypes.c_float(b.scale), ptr(out), stream)


@pytest.mark.gpu
def test_no_alloc_matches_pa_forward_on_two_calls_in_a_row():
    batches = [
        W.make_attn_batch("na_decode", [700, 33, 2000, 0, 4096], [1] * 5, 16, 4, 128, 16, "bf16",
                          seed=101),
        W.make_attn_batch("na_mixed", [300, 90, 1500], [1, 40, 3], 8, 8, 128, 32, "bf16",
                          seed=102),
    ]
    for b in batches:
        d = batch_to_dev(b)
        ref = pkg.pa_forward(d["q"], d["k"], d["v"], d["bt"], d["ctx"], d["ql"], b.scale)
        out = torch.full_like(d["q"], float("nan"))
        rc = _no_alloc_call(b, d, out)
        torch.cuda.synchronize()
        assert rc == 0, pk.load_library().pa_status_string(rc)
        assert pkg.device_status() == 0
        assert_close(as_f64(out), as_f64(ref), b.dtype, f"no_alloc vs pa_forward ({b.name})")


def test_no_alloc_rejects_batches_that_do_not_fit():
    """Host-side check, before any device work: a batch whose scratch exceeds the library's
    fixed array is refused with PA_ERR_WORKSPACE."""
    lib = pk.load_library()
    big = pk.PaDims(1, 4096, 4096, 64, 64, 128, 16, 1 << 20, 4096, 0)
    assert lib.pa_forward_workspace_size(ctypes.byref(big)) > pk.NO_ALLOC_WORKSPACE_BYTES
    fake = ctypes.c_void_p(0x10000)
    rc = lib.pa_forward_no_alloc(ctypes.byref(big), fake, fake, fake, fake, fake, fake,
                                 ctypes.c_float(0.1), ctypes.c_void_p(0x20000), None)
    assert rc == 3
