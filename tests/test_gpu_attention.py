"""GPU parity of pa_forward against the float64 oracle (through the C ABI).

Small cases are compared row by row in full (several KV tiles, ragged tails, every dtype, head
dim, block size and GQA group the library supports).  The benchmark-sized configurations are
compared on sampled rows, including every sequence's last token (the longest causal range).
"""
import zlib

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_generalized_gb300 as pkg
from paged_kv_cache_generalized_gb300 import workloads as W

from gpu_util import (as_f64, assert_close, batch_to_dev, gather_rows, run_forward, sample_rows,
                      to_dev)

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clean_status():
    pkg.device_status()
    yield


def _full_parity(b, threads=8):
    out = run_forward(b)
    ref = oracle.paged_attention_batch(b, threads=threads)
    err = assert_close(as_f64(out), ref, b.dtype, b.name)
    assert pkg.device_status() == 0
    return err


def test_tiny_config():
    _full_parity(W.tiny())


CASES = [
    # name, ctx_lens, q_lens, Hq, Hkv, d, B, dtype, layout
    ("decode_mha_bf16", [512, 1000, 37, 4096, 15, 16], [1] * 6, 8, 8, 128, 16, "bf16", "shuffle"),
    ("decode_gqa4_bf16", [700, 33, 2000, 0], [1] * 4, 16, 4, 128, 32, "bf16", "shuffle"),
    ("decode_gqa8_f16", [300, 129, 64], [1] * 3, 16, 2, 128, 16, "f16", "shuffle"),
    ("decode_d64_f32", [250, 17, 1], [1] * 3, 4, 2, 64, 16, "f32", "shuffle"),
    ("prefill_mha_bf16", [300, 0, 129], [200, 150, 33], 4, 4, 128, 16, "bf16", "segments"),
    ("prefill_gqa4_bf16", [1024, 77, 5], [96, 300, 16], 8, 2, 128, 32, "bf16", "shuffle"),
    ("prefill_short_turns_bf16", [64, 200, 31], [2, 3, 15], 8, 8, 128, 16, "bf16", "shuffle"),
    ("prefill_d64_bf16", [100, 40], [70, 9], 4, 2, 64, 16, "bf16", "shuffle"),
    ("prefill_f32", [60, 0], [40, 33], 4, 4, 128, 16, "f32", "shuffle"),
    ("mixed_gqa_bf16", [500, 100, 2000, 33, 0, 700], [1, 130, 1, 17, 64, 1], 32, 8, 128, 32,
     "bf16", "shuffle"),
    ("block64_f16", [200, 70], [1, 90], 8, 4, 128, 64, "f16", "shuffle"),
    ("block128_bf16", [300, 5], [130, 1], 4, 1, 128, 128, "bf16", "shuffle"),
    ("exact_block_multiples_bf16", [16, 31, 32, 48], [16, 1, 32, 16], 4, 4, 128, 16, "bf16", "shuffle"),
    # CUDA-core GQA rows (2 or 4 query rows per KV head and item): short turns with ragged row
    # groups, a group of 3 (rows split 2 + 1), fp32 at d=128, d=64
    ("short_turns_gqa4_bf16", [100, 513, 0, 47], [3, 2, 1, 1], 16, 4, 128, 32, "bf16", "shuffle"),
    ("gqa3_f16", [300, 45, 1200], [5, 1, 1], 6, 2, 128, 16, "f16", "shuffle"),
    ("gqa4_f32_d128", [400, 90], [1, 3], 8, 2, 128, 16, "f32", "shuffle"),
    ("gqa2_d64_bf16", [1000, 5, 300], [1, 1, 7], 8, 4, 64, 16, "bf16", "segments"),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_small_cases_full_parity(case):
    name, ctx, ql, hq, hkv, d, B, dtype, layout = case
    b = W.make_attn_batch(name, ctx, ql, hq, hkv, d, B, dtype, seed=zlib.crc32(name.encode()) % 1000,
                          layout=layout, seg=(32, 160))
    _full_parity(b)


def test_many_sequences_exercise_the_planner():
    """More sequences than one planner pass (1024 threads) covers; mixed decode and turns."""
    rng = np.random.default_rng(7)
    S = 2500
    ctx = rng.integers(0, 120, S)
    ql = np.where(rng.random(S) < 0.8, 1, rng.integers(2, 40, S))
    b = W.make_attn_batch("many", ctx, ql, 8, 2, 64, 16, "bf16", seed=7)
    out = run_forward(b)
    rows = sample_rows(b, 3000, seed=1)
    ref = oracle.paged_attention_batch(b, rows=rows, threads=8)
    assert_close(gather_rows(out, b, rows), ref, "bf16", "many")
    assert pkg.device_status() == 0


def test_prefix_sharing_aliasing():
    b = W.make_attn_batch("prefix", [200, 150, 96], [1, 40, 1], 8, 8, 128, 16, "bf16", seed=3,
                          shared_prefix_blocks=5, slack=0.5)
    _full_parity(b)


def test_nan_poisoned_unread_slots_do_not_leak():
    """Free blocks and the tails of last blocks hold NaN; block-table padding holds garbage ids."""
    b = W.make_attn_batch("poison", [45, 0, 300, 17], [1, 37, 100, 1], 8, 2, 128, 16, "bf16",
                          seed=5, poison=True)
    bt = b.block_tables.copy()
    bt[bt < 0] = 2 ** 30
    b.block_tables = bt
    _full_parity(b)


def test_chunked_turn_matches_one_prefill():
    """ConvKV turn-level prefix extension: a turn attended in two chunks (append chunk, attend;
    append next chunk, attend) gives the rows of attending the whole turn at once."""
    b = W.make_attn_batch("chunked", [500], [200], 8, 2, 128, 16, "bf16", seed=11)
    d = batch_to_dev(b)
    full = as_f64(pkg.pa_forward(d["q"], d["k"], d["v"], d["bt"], d["ctx"], d["ql"], b.scale))
    parts = []
    for c0, n in ((500, 120), (620, 80)):
        qq = d["q"][c0 - 500:c0 - 500 + n].contiguous()
        o = pkg.pa_forward(qq, d["k"], d["v"], d["bt"], torch.tensor([c0], dtype=torch.int32, device="cuda"),
                           torch.tensor([n], dtype=torch.int32, device="cuda"), b.scale)
        parts.append(as_f64(o))
    torch.cuda.synchronize()
    ref = oracle.paged_attention_batch(b)
    assert_close(full, ref, "bf16", "whole turn")
    assert_close(np.concatenate(parts), ref, "bf16", "chunked turn")


def test_deterministic():
    b = W.make_attn_batch("det", [900, 30, 2000], [1, 64, 1], 16, 4, 128, 16, "bf16", seed=13)
    d = batch_to_dev(b)
    o1 = run_forward(b, d).clone()
    o2 = run_forward(b, d)
    assert torch.equal(o1, o2)


def test_bad_block_id_is_flagged_not_trapped():
    b = W.make_attn_batch("badblk", [100, 100], [1, 1], 4, 4, 128, 16, "bf16", seed=17)
    bt = b.block_tables.copy()
    bt[1, 2] = b.num_blocks + 1000
    b.block_tables = bt
    out = run_forward(b)
    flags = pkg.device_status()
    assert flags & 0x1, pkg.status_names(flags)
    # the other sequence is unaffected
    ref = oracle.paged_attention(b.q[:1], b.k_cache, b.v_cache, "bf16", b.block_tables[:1],
                                 b.ctx_lens[:1], b.q_lens[:1], 4, 4, 128, 16, b.scale)
    assert_close(as_f64(out[:1]), ref, "bf16", "unaffected sequence")


def test_inconsistent_lengths_are_flagged():
    b = W.make_attn_batch("badlen", [10, 20], [3, 2], 4, 4, 64, 16, "f32", seed=19)
    d = batch_to_dev(b)
    d["ql"] = torch.tensor([3, 9], dtype=torch.int32, device="cuda")     # sum != total_q
    out = torch.full_like(d["q"], 7.0)
    pkg.pa_forward(d["q"], d["k"], d["v"], d["bt"], d["ctx"], d["ql"], b.scale, out=out)
    flags = pkg.device_status()
    assert flags & 0x2
    assert torch.all(out == 7.0)               # nothing was written


# ------------------------------------------------------------------------------------------------
# Benchmark-sized configurations: sampled rows
# ------------------------------------------------------------------------------------------------

def _sampled(b, n_rows, seed=0, **kw):
    d = batch_to_dev(b)
    out = run_forward(b, d, **kw)
    rows = sample_rows(b, n_rows, seed=seed)
    ref = oracle.paged_attention_batch(b, rows=rows, threads=16)
    err = assert_close(gather_rows(out, b, rows), ref, b.dtype, b.name)
    assert pkg.device_status() == 0
    return out, err


def test_config_decode13b_full_size():
    _sampled(W.decode13b(), 512)


def test_config_mixed_gqa_full_size():
    _sampled(W.mixed_gqa(), 384)


def test_config_longprefill_full_size():
    _sampled(W.longprefill(), 128)


# ------------------------------------------------------------------------------------------------
# Tensor-core path (multi-token bf16/f16 turns, head_dim 128)
# ------------------------------------------------------------------------------------------------

def _forward_with_workspace(b):
    d = batch_to_dev(b)
    need = pkg.forward_workspace_size(d["q"], d["k"], d["bt"], d["ctx"])
    ws = torch.zeros(max(need, 256), dtype=torch.uint8, device="cuda")
    out = pkg.pa_forward(d["q"], d["k"], d["v"], d["bt"], d["ctx"], d["ql"], b.scale, workspace=ws)
    torch.cuda.synchronize()
    counters = ws[:64].view(torch.int32).cpu().numpy()
    return out, counters


TC_CASES = [
    # name, ctx, q, Hq, Hkv, B, dtype, scale
    ("tc_one_tile", [0], [128], 1, 1, 16, "bf16", None),
    ("tc_one_tile_tiny_scale", [0], [128], 1, 1, 16, "bf16", 1e-30),   # weights ~uniform
    ("tc_ctx_not_multiple", [77], [100], 2, 2, 16, "bf16", None),
    ("tc_gqa4_b32", [1000, 31], [64, 200], 16, 4, 32, "bf16", None),
    ("tc_gqa8_f16", [260], [40], 16, 2, 64, "f16", None),
    ("tc_b128", [300], [129], 2, 1, 128, "bf16", None),
    ("tc_long", [3000], [300], 1, 1, 16, "bf16", None),
    # lone query tiles (odd tile count per KV head: slot 0 alone, slot 1 passes its turns): 4 and
    # 5 KV tiles, a ragged last KV tile, partly filled query tiles, every block size, f16, MHA
    # and GQA, a lone tile next to a pair, a tiny scale
    ("lone_4_tiles", [400], [32], 8, 2, 32, "bf16", None),
    ("lone_5_tiles_f16", [520], [32], 8, 2, 16, "f16", None),
    ("lone_ragged_mha", [1000, 2222], [100, 77], 2, 2, 64, "bf16", None),
    ("lone_b128_gqa8", [5000], [16], 16, 2, 128, "bf16", None),
    ("lone_beside_pair", [3000, 700], [96, 48], 8, 2, 16, "bf16", None),
    ("lone_tiny_scale", [1500], [32], 4, 1, 32, "bf16", 1e-30),
    # few items over long contexts (200+ KV tiles per lone tile)
    ("lone_long_context", [30000, 17000, 25000], [16, 16, 48], 64, 8, 32, "bf16", None),
    # more items than CTAs (24 sequences x 8 KV heads of lone tiles, some beside pairs)
    ("lone_many_items", [600 + 37 * i for i in range(24)], [16] * 20 + [48, 32, 16, 48], 64, 8, 16,
     "bf16", None),
]

# Launches with fewer pair items than CTAs: each pair's key range runs as chunks on separate CTAs,
# merged by the logsumexp rule (rows that see no key in some chunk, pairs whose tiles end in
# different chunks, lone tiles, GQA 8, f16, block sizes 16-128)
TC_CHUNK_CASES = [
    ("chunk_one_turn_gqa8", [60000], [16], 16, 2, 32, "bf16", None),
    ("chunk_two_turns_100k", [100000, 99000], [32, 32], 16, 4, 32, "bf16", None),
    ("chunk_pairs_f16_b16", [16000], [256], 32, 8, 16, "f16", None),
    ("chunk_ragged_mix", [30000, 17000, 25000, 900], [16, 16, 48, 130], 64, 8, 64, "bf16", None),
    ("chunk_mha_b128", [20000], [200], 4, 4, 128, "bf16", None),
    ("chunk_short_context", [1000], [40], 8, 2, 16, "bf16", None),
]


@pytest.mark.parametrize("case", TC_CHUNK_CASES, ids=[c[0] for c in TC_CHUNK_CASES])
def test_tensor_core_key_range_chunks(case):
    name, ctx, ql, hq, hkv, B, dtype, scale = case
    b = W.make_attn_batch(name, ctx, ql, hq, hkv, 128, B, dtype, seed=zlib.crc32(name.encode()) % 1000,
                          scale=scale)
    out, counters = _forward_with_workspace(b)
    assert counters[3] > 0, "no tile went to the tensor-core kernel"
    assert counters[6] > 0, "the pairs were not chunked"
    assert pkg.device_status() == 0
    ref = oracle.paged_attention_batch(b, threads=8)
    assert_close(as_f64(out), ref, b.dtype, name)
    out2, _ = _forward_with_workspace(b)
    assert torch.equal(out, out2)                      # the merge order does not depend on timing


@pytest.mark.parametrize("case", TC_CASES, ids=[c[0] for c in TC_CASES])
def test_tensor_core_path(case):
    name, ctx, ql, hq, hkv, B, dtype, scale = case
    b = W.make_attn_batch(name, ctx, ql, hq, hkv, 128, B, dtype, seed=zlib.crc32(name.encode()) % 1000,
                          scale=scale)
    out, counters = _forward_with_workspace(b)
    assert counters[3] > 0, "no tile went to the tensor-core kernel"
    assert pkg.device_status() == 0
    ref = oracle.paged_attention_batch(b, threads=8)
    assert_close(as_f64(out), ref, b.dtype, name)


# ------------------------------------------------------------------------------------------------
# Block-first pools ("KVキャッシュ管理の教科書" 第14章: all layers of a block contiguous): one
# layer's K and V are strided views [num_blocks, Hkv, B, d] with a block stride of L * 2 * Hkv*B*d
# ------------------------------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
def test_block_first_pool_every_layer(dtype):
    ctx, ql = [700, 90, 1500, 33, 2000], [40, 3, 1, 200, 1]
    b = W.make_attn_batch("block_first", ctx, ql, 8, 2, 128, 16, dtype, seed=77)
    L = 3
    kv = [(b.k_cache, b.v_cache)] + [(W.random_values(b.k_cache.shape, dtype, 90 + 2 * l),
                                      W.random_values(b.v_cache.shape, dtype, 91 + 2 * l)) for l in range(1, L)]
    # [num_blocks, L, 2, Hkv, B, d]
    pool = torch.stack([torch.stack([to_dev(k, dtype), to_dev(v, dtype)], 1) for k, v in kv], 1)
    d = batch_to_dev(b)
    for layer, (k, v) in enumerate(kv):
        kc, vc = pool[:, layer, 0], pool[:, layer, 1]
        assert kc.stride(0) == L * 2 * kc[0].numel()
        out = pkg.pa_forward(d["q"], kc, vc, d["bt"], d["ctx"], d["ql"], b.scale)
        torch.cuda.synchronize()
        assert pkg.device_status() == 0
        import dataclasses
        ref = oracle.paged_attention_batch(dataclasses.replace(b, k_cache=k, v_cache=v), threads=8)
        assert_close(as_f64(out), ref, dtype, f"block-first layer {layer}")
