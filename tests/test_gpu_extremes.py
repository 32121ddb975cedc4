"""GPU parity at the edges of what pa_forward accepts (through the C ABI, against the float64
oracle): contexts past 100K tokens on both kernels, GQA groups of 16 and 128 query heads per KV
head, more sequences than the planner ranks by length, first tokens (c = 0, q = 1: the output is
the token's own V row), and zero and negative softmax scales."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_generalized_gb300 as pkg
from paged_kv_cache_generalized_gb300 import workloads as W

from gpu_util import as_f64, assert_close, batch_to_dev, gather_rows, run_forward, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clean_status():
    pkg.device_status()
    yield


def _tc_tiles(b, d):
    """Runs pa_forward with its own workspace and returns (out, number of tensor-core items)."""
    need = pkg.forward_workspace_size(d["q"], d["k"], d["bt"], d["ctx"])
    ws = torch.zeros(max(need, 256), dtype=torch.uint8, device="cuda")
    out = pkg.pa_forward(d["q"], d["k"], d["v"], d["bt"], d["ctx"], d["ql"], b.scale, workspace=ws)
    torch.cuda.synchronize()
    return out, int(ws[:64].view(torch.int32).cpu()[3])


def test_contexts_past_100k_tokens():
    """A 200K-token decode (split-KV at the 64-split cap) and a 300-token turn over 100K cached
    tokens on the tensor cores, GQA 8:1, sampled rows including every last token."""
    b = W.make_attn_batch("long_ctx", [200000, 100000, 5], [1, 300, 1], 8, 1, 128, 64, "bf16", seed=31,
                          poison=False)
    d = batch_to_dev(b)
    out, tc_items = _tc_tiles(b, d)
    assert tc_items > 0
    assert pkg.device_status() == 0
    rows = sample_rows(b, 24, seed=2)
    ref = oracle.paged_attention_batch(b, rows=rows, threads=16)
    assert_close(gather_rows(out, b, rows), ref, "bf16", "long contexts")


@pytest.mark.parametrize("hq,hkv,ql", [(32, 2, [1, 40, 3]), (128, 1, [1, 9, 2])])
def test_wide_gqa_groups(hq, hkv, ql):
    """g = 16 (a tile packs 8 tokens x 16 heads) and g = 128 (one token per tile): both kernels."""
    b = W.make_attn_batch(f"g{hq // hkv}", [300, 777, 64], ql, hq, hkv, 128, 16, "bf16", seed=hq)
    d = batch_to_dev(b)
    out, tc_items = _tc_tiles(b, d)
    assert tc_items > 0
    assert pkg.device_status() == 0
    assert_close(as_f64(out), oracle.paged_attention_batch(b, threads=16), "bf16", f"g={hq // hkv}")


def test_more_sequences_than_the_planner_ranks():
    """Past 4096 sequences the planner orders tensor-core sequences by index, not by length."""
    rng = np.random.default_rng(11)
    S = 4500
    ctx = rng.integers(0, 96, S)
    ql = np.where(rng.random(S) < 0.9, 1, rng.integers(4, 40, S))
    b = W.make_attn_batch("s4500", ctx, ql, 8, 2, 128, 16, "bf16", seed=12)
    d = batch_to_dev(b)
    out, tc_items = _tc_tiles(b, d)
    assert tc_items > 0
    assert pkg.device_status() == 0
    rows = sample_rows(b, 1500, seed=4)
    assert_close(gather_rows(out, b, rows), oracle.paged_attention_batch(b, rows=rows, threads=16),
                 "bf16", "4500 sequences")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_first_tokens_return_their_own_value_row(dtype):
    """c = 0, q = 1: the only visible key is the token itself, so out = its V row exactly."""
    b = W.make_attn_batch("first", [0] * 7, [1] * 7, 8, 2, 128, 16, dtype, seed=21)
    out = run_forward(b)
    assert pkg.device_status() == 0
    B = b.block_size
    for i in range(b.num_seqs):
        blk = b.block_tables[i, 0]
        for h in range(b.num_q_heads):
            v = b.v_cache[blk, h // 4, 0]
            want = v if dtype == "f32" else (v.astype(np.uint32) << 16).view(np.float32)
            np.testing.assert_array_equal(as_f64(out[i, h]), want.astype(np.float64))


@pytest.mark.parametrize("scale", [0.0, -0.09])
def test_zero_and_negative_scales(scale):
    """scale = 0 averages the visible V rows; a negative scale flips the weighting.  Both stay on
    the CUDA-core kernels (the tensor-core kernel takes positive scales)."""
    b = W.make_attn_batch("scale", [130, 0, 45], [1, 30, 17], 8, 2, 128, 16, "bf16", seed=23, scale=scale)
    out = run_forward(b)
    assert pkg.device_status() == 0
    assert_close(as_f64(out), oracle.paged_attention_batch(b, threads=8), "bf16", f"scale {scale}")
