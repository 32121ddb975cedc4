"""GPU tests of the layer-by-layer swap-in schedule ("Stateful Large Language Model Serving with
Pensieve", section "パイプライン化されたswap-in") and of swap-out, through the C ABI.

Before every schedule runs, the device blocks that the swap-in refills are overwritten with NaN
bit patterns, so a layer whose attention started before its own blocks landed shows up as a
non-finite or wrong output.  Every layer holds different values, so a transfer that landed in
the wrong layer is caught as well.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_generalized_gb300 as pkg
from paged_kv_cache_generalized_gb300 import swap as S
from paged_kv_cache_generalized_gb300 import workloads as W

from gpu_util import as_f64, assert_close, bits, to_dev

pytestmark = pytest.mark.gpu

NAN_BF16 = 0x7FC0


@pytest.fixture(autouse=True)
def _clean_status():
    pkg.device_status()
    yield


def _layers(L=3):
    """One small mixed GQA batch (resumed turns on the tensor-core and CUDA-core paths, decode
    steps) and L layers of K/V values for it (layer 0 = the batch's own)."""
    ctx = [700, 90, 1500, 33, 400, 2000]
    ql = [40, 3, 1, 200, 1, 17]
    b = W.make_attn_batch("swap", ctx, ql, 8, 2, 128, 16, "bf16", seed=40, poison=False)
    kv = [(b.k_cache, b.v_cache)] + [
        (W.random_values(b.k_cache.shape, "bf16", 500 + 2 * l), W.random_values(b.v_cache.shape, "bf16", 501 + 2 * l))
        for l in range(1, L)]
    return b, kv


def _setup(b, kv, frac=0.5):
    L = len(kv)
    blocks = W.swap_plan(b, frac)
    assert len(blocks) > 4
    pool = torch.stack([torch.stack([to_dev(k, "bf16"), to_dev(v, "bf16")]) for k, v in kv])
    host = torch.empty((L, 2, len(blocks)) + tuple(b.k_cache.shape[1:]), dtype=torch.bfloat16).pin_memory()
    dblocks = torch.from_numpy(blocks).cuda()
    for layer in range(L):
        host[layer].copy_(pool[layer][:, dblocks])
    return pool, host, dblocks


def _poison(pool, dblocks):
    pool.view(torch.int16)[:, :, dblocks] = NAN_BF16


def _schedule(b, pool, host, dblocks, mode, serial):
    q, bt, ctx, ql = to_dev(b.q, "bf16"), to_dev(b.block_tables), to_dev(b.ctx_lens), to_dev(b.q_lens)
    outs = [torch.empty_like(q) for _ in range(pool.shape[0])]
    cur = torch.cuda.current_stream()
    sw = S.LayerSwapIn(host, pool, dblocks, mode=mode, max_ctas=8,
                       copy_stream=cur if serial else torch.cuda.Stream(priority=-1))

    def attention(layer):
        pkg.pa_forward(q, pool[layer, 0], pool[layer, 1], bt, ctx, ql, b.scale, out=outs[layer])

    _poison(pool, dblocks)
    sw.run(attention)
    torch.cuda.synchronize()
    assert pkg.device_status() == 0
    return outs


@pytest.mark.parametrize("mode", ["staged", "gather"])
def test_pipelined_swap_in_matches_oracle_per_layer(mode):
    b, kv = _layers()
    pool, host, dblocks = _setup(b, kv)
    outs = _schedule(b, pool, host, dblocks, mode, serial=False)
    for layer, (k, v) in enumerate(kv):
        ref = oracle.paged_attention_batch(dataclasses.replace(b, k_cache=k, v_cache=v), threads=8)
        assert_close(as_f64(outs[layer]), ref, "bf16", f"{mode} layer {layer}")


def test_pipelined_equals_serial_bit_for_bit():
    b, kv = _layers()
    pool, host, dblocks = _setup(b, kv)
    ref = [bits(o) for o in _schedule(b, pool, host, dblocks, "staged", serial=True)]
    for mode in ("staged", "gather"):
        got = _schedule(b, pool, host, dblocks, mode, serial=False)
        for layer in range(len(kv)):
            assert bits(got[layer]).tobytes() == ref[layer].tobytes(), f"{mode} layer {layer}"


def test_swap_out_to_host_bit_exact():
    b, kv = _layers(2)
    pool, host, dblocks = _setup(b, kv)
    back = torch.zeros_like(host).pin_memory()
    S.swap_out(pool, back, S.swap_out_pairs(dblocks), max_ctas=4)
    torch.cuda.synchronize()
    assert pkg.device_status() == 0
    expect = pool[:, :, dblocks].cpu()
    assert bits(back).tobytes() == bits(expect).tobytes()


def test_swap_out_beside_swap_in_on_two_streams():
    """Eviction of some blocks on a low-priority stream while others come back on a high-priority
    one: both land bit for bit."""
    b, kv = _layers(2)
    pool, host, dblocks = _setup(b, kv)
    half = dblocks.numel() // 2
    ins, outs_ = dblocks[:half], dblocks[half:]
    host_in = host[:, :, :half].contiguous().pin_memory()
    evict = torch.zeros((2, 2, dblocks.numel() - half) + tuple(host.shape[3:]), dtype=host.dtype).pin_memory()
    expect_out = pool[:, :, outs_].cpu()
    _poison(pool, ins)
    hi, lo = torch.cuda.Stream(priority=-1), torch.cuda.Stream(priority=0)
    lo.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(lo):
        S.swap_out(pool, evict, S.swap_out_pairs(outs_), stream=lo, max_ctas=16)
    sw = S.LayerSwapIn(host_in, pool, ins, mode="gather", max_ctas=16, copy_stream=hi)
    sw.run(None)
    torch.cuda.synchronize()
    assert pkg.device_status() == 0
    assert bits(evict).tobytes() == bits(expect_out).tobytes()
    assert bits(pool[:, :, ins]).tobytes() == bits(host_in).tobytes()
