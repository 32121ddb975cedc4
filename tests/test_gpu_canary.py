"""Canary guard regions around every buffer the attention calls write (no memory checker runs on
the GPU here, so the guards carry the out-of-bounds-write check).

The output and the caller's workspace sit between 4 KiB guards filled with a seeded byte
pattern; after the call the guards must hold exactly the same bytes, so a write one byte past
either end of `out` or of the workspace fails.  The outputs are also compared with the float64
oracle, so the call did its work.  Cases: the mixed batch (tensor-core prefill tiles, lone
tiles, GQA decode on tensor-core fragments, split-KV merges), MHA decode with many splits, fp32
at head_dim 64, E4M3 caches, and decode over 2-bit pages."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_generalized_gb300 as pkg
from paged_kv_cache_generalized_gb300 import workloads as W

from gpu_util import TORCH_DTYPE, as_f64, assert_close, batch_to_dev

pytestmark = pytest.mark.gpu

GUARD = 4096


@pytest.fixture(autouse=True)
def _clean_status():
    pkg.device_status()
    yield


class Guarded:
    """`nbytes` of usable device memory between two guards of a seeded byte pattern; the usable
    region starts 4 KiB into the allocation (so it keeps the allocation's 256-byte alignment)."""

    def __init__(self, nbytes, seed):
        g = torch.Generator().manual_seed(seed)
        self.n = int(nbytes)
        host = torch.randint(0, 256, (GUARD + self.n + GUARD,), dtype=torch.uint8, generator=g)
        self.pattern = host.clone()
        self.buf = host.cuda()

    def view(self, dtype, shape):
        return self.buf[GUARD:GUARD + self.n].view(dtype).view(shape)

    def region(self):
        return self.buf[GUARD:GUARD + self.n]

    def check(self, what):
        torch.cuda.synchronize()
        got = self.buf.cpu()
        before, after = got[:GUARD], got[GUARD + self.n:]
        assert torch.equal(before, self.pattern[:GUARD]), f"{what}: bytes written before the buffer"
        assert torch.equal(after, self.pattern[GUARD + self.n:]), f"{what}: bytes written past the buffer"


def _forward_guarded(b, d, seed, **kw):
    dt = TORCH_DTYPE[b.dtype]
    out_g = Guarded(d["q"].numel() * d["q"].element_size(), seed)
    need = pkg.forward_workspace_size(d["q"], d["k"], d["bt"], d["ctx"])
    ws_g = Guarded(need, seed + 1)
    out = out_g.view(dt, tuple(d["q"].shape))
    pkg.pa_forward(d["q"], d["k"], d["v"], d["bt"], d["ctx"], d["ql"], b.scale, out=out,
                   workspace=ws_g.region(), **kw)
    out_g.check(f"{b.name} out")
    ws_g.check(f"{b.name} workspace")
    assert pkg.device_status() == 0
    return out


CASES = [
    ("canary_mixed_gqa", [500, 100, 3000, 33, 0, 700, 1500], [1, 130, 1, 17, 64, 1, 40], 32, 8, 128, 32, "bf16"),
    ("canary_decode_mha", [4096, 700, 33, 2000, 0, 513], [1] * 6, 16, 16, 128, 16, "bf16"),
    ("canary_prefill_lone", [2000, 9000], [20, 12], 16, 4, 128, 16, "f16"),
    ("canary_d64_f32", [250, 17, 90], [1, 33, 5], 4, 2, 64, 16, "f32"),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_pa_forward_writes_nothing_outside_out_and_workspace(case):
    name, ctx, ql, hq, hkv, d_, B, dtype = case
    b = W.make_attn_batch(name, ctx, ql, hq, hkv, d_, B, dtype, seed=len(name))
    d = batch_to_dev(b)
    out = _forward_guarded(b, d, seed=11)
    assert_close(as_f64(out), oracle.paged_attention_batch(b, threads=8), b.dtype, name)


def test_e4m3_caches_write_nothing_outside_out_and_workspace():
    b = W.make_attn_batch("canary_e4m3", [900, 60, 2048], [1, 1, 1], 8, 8, 128, 16, "bf16", seed=5,
                          poison=False)
    ks, vs = 1.0 / 32, 1.0 / 16
    kc = oracle.e4m3_encode(W.normal_f32(b.k_cache.shape, 6), np.float32(1.0) / np.float32(ks))
    vc = oracle.e4m3_encode(W.normal_f32(b.v_cache.shape, 7), np.float32(1.0) / np.float32(vs))
    d = batch_to_dev(b)
    d["k"], d["v"] = torch.from_numpy(kc).cuda(), torch.from_numpy(vc).cuda()
    out = _forward_guarded(b, d, seed=21, k_scale=ks, v_scale=vs)
    ref = oracle.paged_attention_batch(b, threads=8, kv=(kc, vc, ks, vs))
    assert_close(as_f64(out), ref, b.dtype, "e4m3 canary")


def test_kitty_decode_writes_nothing_outside_out_and_workspace():
    from test_gpu_kitty import gpu_state, oracle_rows

    b = W.make_kitty_batch("canary_kitty", [127, 128, 300, 1801, 4101], 8, 2, 32, dtype="bf16", seed=31)
    d = gpu_state(b)
    out_g = Guarded(d["q"].numel() * d["q"].element_size(), 41)
    need = pkg.kitty_workspace_size(d["q"], d["pages"], d["res_k"], d["bt"], b.promoted)
    ws_g = Guarded(need, 42)
    out = out_g.view(torch.bfloat16, tuple(d["q"].shape))
    pkg.pa_forward_kitty(d["q"], d["pages"], d["res_k"], d["res_v"], d["bt"], d["ctx"], d["ql"], b.promoted,
                         b.scale, out=out, workspace=ws_g.region())
    out_g.check("kitty out")
    ws_g.check("kitty workspace")
    assert pkg.device_status() == 0
    assert_close(as_f64(out), oracle_rows(b, list(range(b.num_seqs))), "bf16", "kitty canary")
