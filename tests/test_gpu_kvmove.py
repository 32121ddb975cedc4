"""GPU bit-exactness of kv_append and block_copy against the oracle (through the C ABI):
append into partially filled blocks, copy-on-write copies inside a device pool, swap-in from a
page-locked host pool and swap-out to one, multi-layer pools, and device-side flagging of bad
slots and pairs."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_generalized_gb300 as pkg
from paged_kv_cache_generalized_gb300 import workloads as W

from gpu_util import bits, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clean_status():
    pkg.device_status()
    yield


def _u16(t):
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("dtype,B,d,hkv", [("f16", 32, 128, 40), ("bf16", 16, 128, 8),
                                           ("f16", 16, 64, 3), ("bf16", 128, 64, 2)])
def test_append_single_layer_bit_exact(dtype, B, d, hkv):
    b = W.make_attn_batch("app", [0, 5, B - 1, B, 3 * B + 2], [3, B + 4, 1, 2 * B, 7], hkv, hkv,
                          d, B, dtype, seed=B + d, poison=False)
    kc0 = W.random_bits16(b.k_cache.shape, 1)
    vc0 = W.random_bits16(b.v_cache.shape, 2)
    kn = W.random_bits16(b.k_new.shape, 3)
    vn = W.random_bits16(b.v_new.shape, 4)
    slots = b.slot_mapping.copy()
    slots[1] = -1                                     # one padding token
    kc, vc = to_dev(kc0, dtype), to_dev(vc0, dtype)
    pkg.kv_append(to_dev(kn, dtype), to_dev(vn, dtype), to_dev(slots), kc, vc)
    ek, ev = oracle.kv_append(kn, vn, slots, kc0, vc0, B)
    assert _u16(kc).tobytes() == ek.tobytes()
    assert _u16(vc).tobytes() == ev.tobytes()
    assert pkg.device_status() == 0


def test_append_multi_layer_pool_bit_exact():
    """Pool [L, 2 (K,V), num_blocks, Hkv, B, d]: K and V of each layer are strided views."""
    plan = W.kvmove_plan(num_layers=3, num_sessions=6, swap_sessions=1, lens=(40, 300), new=(1, 70))
    L, nb, hkv, B, d = plan.num_layers, plan.num_blocks, plan.num_kv_heads, plan.block_size, plan.head_dim
    pool0 = W.random_bits16((L, 2, nb, hkv, B, d), 5)
    T = len(plan.slot_mapping)
    new0 = W.random_bits16((L, 2, T, hkv, d), 6)
    pool = to_dev(pool0, "f16")
    new = to_dev(new0, "f16")
    pkg.kv_append(new[:, 0], new[:, 1], to_dev(plan.slot_mapping), pool[:, 0], pool[:, 1])
    got = _u16(pool)
    for l in range(L):
        ek, ev = oracle.kv_append(new0[l, 0], new0[l, 1], plan.slot_mapping, pool0[l, 0],
                                  pool0[l, 1], B)
        assert got[l, 0].tobytes() == ek.tobytes()
        assert got[l, 1].tobytes() == ev.tobytes()
    assert pkg.device_status() == 0


def test_append_bad_slot_is_flagged_and_skipped():
    kc0 = W.random_bits16((4, 2, 16, 64), 7)
    kn = W.random_bits16((2, 2, 64), 8)
    kc, vc = to_dev(kc0, "bf16"), to_dev(kc0, "bf16")
    pkg.kv_append(to_dev(kn, "bf16"), to_dev(kn, "bf16"), to_dev(np.array([3, 4 * 16 + 5])), kc, vc)
    assert pkg.device_status() & 0x4
    ek, _ = oracle.kv_append(kn[:1], kn[:1], [3], kc0, kc0, 16)
    assert _u16(kc).tobytes() == ek.tobytes()


def test_copy_on_write_in_device_pool_bit_exact():
    plan = W.kvmove_plan(num_layers=2, num_sessions=10, swap_sessions=1, lens=(64, 900))
    L, nb = plan.num_layers, plan.num_blocks
    shape = (L * 2, nb, plan.num_kv_heads, plan.block_size, plan.head_dim)
    pool0 = W.random_bits16(shape, 9)                # NaN/Inf payloads included
    pool = to_dev(pool0, "f16")
    pkg.block_copy(pool, pool, to_dev(plan.cow_pairs))
    expect = oracle.block_copy(pool0, pool0, plan.cow_pairs)
    assert _u16(pool).tobytes() == expect.tobytes()
    assert pkg.device_status() == 0


def test_swap_in_from_pinned_host_and_out_again():
    plan = W.kvmove_plan(num_layers=2, num_sessions=4, swap_sessions=3, lens=(64, 700))
    L, nb, nh = plan.num_layers, plan.num_blocks, plan.num_host_blocks
    blk = (plan.num_kv_heads, plan.block_size, plan.head_dim)
    host0 = W.random_bits16((2 * L, nh, *blk), 10)
    dev0 = W.random_bits16((2 * L, nb, *blk), 11)
    host = to_dev(host0, "f16", pin=True)
    pool = to_dev(dev0, "f16")
    pairs = to_dev(plan.swap_pairs)
    pkg.block_copy(host, pool, pairs)                 # swap-in: host -> device
    torch.cuda.synchronize()
    expect = oracle.block_copy(host0, dev0, plan.swap_pairs)
    assert _u16(pool).tobytes() == expect.tobytes()
    # swap-out of the same blocks to a fresh pinned host pool
    back = torch.zeros_like(host).pin_memory()
    rev = np.ascontiguousarray(plan.swap_pairs[:, ::-1])
    pkg.block_copy(pool, back, to_dev(rev))
    torch.cuda.synchronize()
    assert bits(back).tobytes() == host0.view(np.uint8).tobytes()
    assert pkg.device_status() == 0


def test_copy_bad_pair_is_flagged_and_skipped():
    pool0 = W.random_bits16((2, 6, 4, 16, 32), 12)
    pool = to_dev(pool0, "bf16")
    pairs = np.array([[0, 5], [1, 99], [2, 4]], dtype=np.int64)
    pkg.block_copy(pool, pool, to_dev(pairs))
    assert pkg.device_status() & 0x8
    expect = oracle.block_copy(pool0, pool0, pairs[[0, 2]])
    assert _u16(pool).tobytes() == expect.tobytes()


def test_config_kvmove_one_layer_full_size():
    """KV-movement configuration at full session count and block geometry, one layer resident:
    append, copy-on-write and swap-in, compared on every touched block."""
    plan = W.kvmove_plan(num_layers=1)
    nb, nh = plan.num_blocks, plan.num_host_blocks
    blk = (plan.num_kv_heads, plan.block_size, plan.head_dim)
    pool0 = W.random_bits16((2, nb, *blk), 20)
    pool = to_dev(pool0, "f16")
    T = len(plan.slot_mapping)
    new0 = W.random_bits16((2, T, plan.num_kv_heads, plan.head_dim), 21)
    host0 = W.random_bits16((2, nh, *blk), 22)
    host = to_dev(host0, "f16", pin=True)
    pkg.block_copy(pool, pool, to_dev(plan.cow_pairs))
    pkg.kv_append(to_dev(new0[0], "f16"), to_dev(new0[1], "f16"), to_dev(plan.slot_mapping),
                  pool[0], pool[1])
    pkg.block_copy(host, pool, to_dev(plan.swap_pairs))
    torch.cuda.synchronize()
    assert pkg.device_status() == 0
    exp = oracle.block_copy(pool0, pool0, plan.cow_pairs)
    ek, ev = oracle.kv_append(new0[0], new0[1], plan.slot_mapping, exp[0], exp[1], plan.block_size)
    exp = np.stack([ek, ev])
    exp = oracle.block_copy(host0, exp, plan.swap_pairs)
    got = _u16(pool)
    touched = np.unique(np.concatenate([plan.cow_pairs[:, 1], plan.swap_pairs[:, 1],
                                        plan.slot_mapping // plan.block_size]))
    assert got[:, touched].tobytes() == exp[:, touched].tobytes()
    untouched = np.setdiff1d(np.arange(nb), touched)[:500]
    assert got[:, untouched].tobytes() == pool0[:, untouched].tobytes()
