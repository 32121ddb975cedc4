"""pa_forward_no_alloc: attention for callers that cannot allocate device memory (a plug-in
inside an engine whose allocator owns all device memory, a loop that must not call cudaMalloc or
cudaFree because they can synchronise the device).  The call uses the library's own fixed-size
scratch.  It must give the same bytes as pa_forward with a caller-allocated workspace (both run
the same planner and kernels, which are deterministic), call after call and batch after batch
(the scratch keeps the previous call's contents), within the bf16 tolerances of the float64
oracle; it must allocate no device memory; it must write nothing outside `out`; and it must
refuse batches whose scratch would not fit.

This file is collected last on purpose: a run that stops at the first failure has run every
other test before it."""
import ctypes

import pytest
import torch

import oracle
import paged_kv_cache_generalized_gb300 as pkg
from paged_kv_cache_generalized_gb300 import pagedkv as pk
from paged_kv_cache_generalized_gb300 import workloads as W

from gpu_util import as_f64, assert_close, batch_to_dev

GUARD = 4096


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
def test_no_alloc_matches_pa_forward_and_the_oracle_on_two_calls_in_a_row():
    batches = [
        # GQA decode with split-KV merges, and a mixed batch that takes the tensor-core
        # kernel (tile pairs and a split lone tile) beside the GQA decode kernel
        W.make_attn_batch("na_decode", [700, 33, 2000, 0, 4096], [1] * 5, 16, 4, 128, 16, "bf16",
                          seed=101),
        W.make_attn_batch("na_mixed", [300, 90, 1500, 2600], [1, 40, 3, 20], 8, 8, 128, 32, "bf16",
                          seed=102),
    ]
    state = []
    for b in batches:
        d = batch_to_dev(b)
        ref = pkg.pa_forward(d["q"], d["k"], d["v"], d["bt"], d["ctx"], d["ql"], b.scale)
        torch.cuda.synchronize()
        assert pkg.device_status() == 0
        want = oracle.paged_attention_batch(b, threads=8)
        assert_close(as_f64(ref), want, b.dtype, f"pa_forward ({b.name})")
        # out between two guards of NaN bit patterns
        n = d["q"].numel()
        buf = torch.full((2 * GUARD + n,), float("nan"), dtype=d["q"].dtype, device="cuda")
        out = buf[GUARD:GUARD + n].view(d["q"].shape)
        state.append((b, d, ref, want, buf, out))

    # the first call on a device looks up the scratch's address (and the driver may load the
    # library's module); free memory is compared from the second call on
    b, d, _, _, _, out = state[0]
    assert _no_alloc_call(b, d, out) == 0
    torch.cuda.synchronize()

    for rnd in range(2):                                # batch A, B, A, B: two calls of each in a row
        for b, d, ref, want, buf, out in state:
            out.fill_(float("nan"))
            torch.cuda.synchronize()
            free0 = torch.cuda.mem_get_info()[0]
            rc = _no_alloc_call(b, d, out)
            torch.cuda.synchronize()
            free1 = torch.cuda.mem_get_info()[0]
            assert rc == 0, pk.load_library().pa_status_string(rc)
            assert free1 == free0, f"{b.name}: device free memory changed by {free0 - free1} bytes"
            assert pkg.device_status() == 0
            assert torch.equal(out, ref), f"no_alloc differs from pa_forward ({b.name}, call {rnd + 1})"
            assert_close(as_f64(out), want, b.dtype, f"no_alloc vs oracle ({b.name}, call {rnd + 1})")
            assert torch.isnan(buf[:GUARD]).all() and torch.isnan(buf[GUARD + out.numel():]).all(), \
                f"{b.name}: bytes written outside out"
        # the same batch again at once: a second call in a row over the first one's scratch
        b, d, ref, want, buf, out = state[-1]
        out.fill_(float("nan"))
        assert _no_alloc_call(b, d, out) == 0
        torch.cuda.synchronize()
        assert torch.equal(out, ref), f"no_alloc repeated call differs ({b.name})"


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
