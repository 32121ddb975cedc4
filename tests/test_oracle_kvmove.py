"""Pins for the cache-append and block-copy oracles and for the sizing formulas (CPU only).

Append and copy move bits, so their pins are structural: what the pages say must hold after a
write (the token lands at its logical position as seen through the block table; nothing else
changes; copy-on-write leaves the other sharer's view intact; a swap out and back in is the
identity), checked with code written independently of the oracle's scatter.  Sizing is pinned
to the numbers the pages print (``tests/golden/sizing.json``).
"""
import json
import os

import numpy as np
import pytest

from paged_kv_cache_generalized_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "sizing.json")


def _gather(cache, bt_row, pos, B):
    """Logical position -> the [Hkv, d] slice it lives in, through one block-table row."""
    return cache[bt_row[pos // B], :, pos % B, :]


@pytest.mark.parametrize("dtype,B", [("f16", 32), ("bf16", 16), ("f32", 8)])
def test_append_lands_at_logical_positions(oracle_mod, dtype, B):
    rng = np.random.default_rng(1)
    ctx = np.array([0, 5, B - 1, B, 3 * B + 2])
    new = np.array([3, B + 4, 1, 2 * B, 7])
    n = ctx + new
    need = (n + B - 1) // B
    pool = int(need.sum()) + 6
    perm = rng.permutation(pool)
    bt = np.full((len(n), int(need.max())), -1, np.int64)
    pos = 0
    for i, k in enumerate(need):
        bt[i, :k] = perm[pos:pos + k]
        pos += k
    Hkv, d = 3, 16
    kc = W.random_bits16((pool, Hkv, B, d), 7) if dtype != "f32" else W.normal_f32((pool, Hkv, B, d), 7)
    vc = W.random_bits16((pool, Hkv, B, d), 8) if dtype != "f32" else W.normal_f32((pool, Hkv, B, d), 8)
    T = int(new.sum())
    kn = W.random_bits16((T, Hkv, d), 9) if dtype != "f32" else W.normal_f32((T, Hkv, d), 9)
    vn = W.random_bits16((T, Hkv, d), 10) if dtype != "f32" else W.normal_f32((T, Hkv, d), 10)
    slots, owners = [], []
    for i in range(len(n)):
        for p in range(ctx[i], n[i]):
            slots.append(bt[i, p // B] * B + p % B)
            owners.append((i, p))
    k2, v2 = oracle_mod.kv_append(kn, vn, slots, kc, vc, B)
    written = np.zeros((pool, B), bool)
    for t, (i, p) in enumerate(owners):
        assert _gather(k2, bt[i], p, B).tobytes() == kn[t].tobytes()
        assert _gather(v2, bt[i], p, B).tobytes() == vn[t].tobytes()
        written[bt[i, p // B], p % B] = True
    # every other slot keeps its bytes
    keep = ~written
    assert k2.transpose(0, 2, 1, 3)[keep].tobytes() == kc.transpose(0, 2, 1, 3)[keep].tobytes()
    assert v2.transpose(0, 2, 1, 3)[keep].tobytes() == vc.transpose(0, 2, 1, 3)[keep].tobytes()
    # internal waste: each sequence leaves at most B - 1 unused slots in its last block
    assert ((need * B - n) <= B - 1).all()


def test_append_skips_padding_slots(oracle_mod):
    kc = W.random_bits16((4, 2, 16, 8), 1)
    vc = W.random_bits16((4, 2, 16, 8), 2)
    kn = W.random_bits16((3, 2, 8), 3)
    vn = W.random_bits16((3, 2, 8), 4)
    k2, v2 = oracle_mod.kv_append(kn, vn, [-1, 17, -1], kc, vc, 16)
    exp_k = kc.copy()
    exp_k[1, :, 1, :] = kn[1]
    assert k2.tobytes() == exp_k.tobytes()


def test_append_then_attend_first_token(oracle_mod):
    """Write a first token into an empty pool through the append oracle, then attend it: the
    attention output is that token's V row exactly (closed form of softmax over one key)."""
    B, Hkv, d = 16, 2, 64
    kc = np.full((3, Hkv, B, d), np.nan, np.float32)
    vc = kc.copy()
    kn = W.normal_f32((1, Hkv, d), 5)
    vn = W.normal_f32((1, Hkv, d), 6)
    k2, v2 = oracle_mod.kv_append(kn, vn, [2 * B + 0], kc, vc, B)
    q = W.normal_f32((1, 4, d), 7)
    out = oracle_mod.paged_attention(q, k2, v2, "f32", [[2]], [0], [1], 4, Hkv, d, B, 0.125)
    np.testing.assert_array_equal(out[0], np.repeat(vn[0].astype(np.float64), 2, axis=0))


def test_block_copy_moves_every_plane_bit_for_bit(oracle_mod):
    planes, pool = 6, 20
    src = W.random_bits16((planes, pool, 4, 16, 8), 11)          # NaN/Inf payloads included
    dst = W.random_bits16((planes, pool, 4, 16, 8), 12)
    pairs = np.array([[3, 7], [3, 8], [0, 19], [12, 2]])
    out = oracle_mod.block_copy(src, dst, pairs)
    for s, t in pairs:
        assert out[:, t].tobytes() == src[:, s].tobytes()
    untouched = [b for b in range(pool) if b not in set(pairs[:, 1])]
    assert out[:, untouched].tobytes() == dst[:, untouched].tobytes()
    # the copy is of bits: NaN payloads survive
    nanlike = (src[:, pairs[:, 0]] & 0x7C00) == 0x7C00
    assert nanlike.any()


def test_copy_on_write_keeps_the_other_sharer_intact(oracle_mod):
    """Sequences A and B share their last block (refcount 2).  B writes a token: CoW copies the
    block to a fresh one, B's table is remapped, then B appends.  A's view is unchanged, and B
    sees the shared prefix plus its new token."""
    B, Hkv, d = 16, 2, 8
    pool = W.random_bits16((1, 6, Hkv, B, d), 21)                 # one plane
    bt_a = [4, 1]
    bt_b = [4, 1]                                                 # block 1 holds 10 tokens
    before_a = [_gather(pool[0], bt_a, p, B).copy() for p in range(26)]
    pool2 = oracle_mod.block_copy(pool, pool, [[1, 5]])
    bt_b = [4, 5]
    kn = W.random_bits16((1, Hkv, d), 22)
    k2, _ = oracle_mod.kv_append(kn, kn, [5 * B + 10], pool2[0], pool2[0], B)
    for p in range(26):
        assert _gather(k2, bt_a, p, B).tobytes() == before_a[p].tobytes()
        if p < 26:
            assert _gather(k2, bt_b, p, B).tobytes() == before_a[p].tobytes()
    assert _gather(k2, bt_b, 26, B).tobytes() == kn[0].tobytes()


def test_swap_out_and_in_is_identity(oracle_mod):
    dev = W.random_bits16((4, 10, 2, 32, 16), 31)
    host = np.zeros((4, 5, 2, 32, 16), np.uint16)
    out_pairs = [[2, 0], [7, 1], [9, 4]]
    host = oracle_mod.block_copy(dev, host, out_pairs)
    fresh = np.zeros_like(dev)
    back = oracle_mod.block_copy(host, fresh, [[0, 1], [1, 3], [4, 8]])
    for (d_src, h), d_dst in zip(out_pairs, [1, 3, 8]):
        assert back[:, d_dst].tobytes() == dev[:, d_src].tobytes()


# --------------------------------------------------------------------------------------------
# Sizing, pinned to the pages' printed numbers
# --------------------------------------------------------------------------------------------

def _golden():
    with open(GOLDEN) as f:
        return json.load(f)


def test_kv_bytes_per_token_matches_pages(oracle_mod):
    for case in _golden()["kv_bytes_per_token"]:
        got = oracle_mod.kv_bytes_per_token(case["layers"], case["hidden"], case["bytes_per_elem"])
        if "expected_bytes" in case and case.get("exact"):
            assert got == case["expected_bytes"], case["cite"]
        if "expected_mb_approx" in case:
            assert abs(got / 2**20 - case["expected_mb_approx"]) <= case["rel_tol"] * case["expected_mb_approx"]
        if "expected_kb_approx" in case:
            assert abs(got / 1024 - case["expected_kb_approx"]) <= case["rel_tol"] * case["expected_kb_approx"]


def test_request_and_budget_sizes_match_pages(oracle_mod):
    g = _golden()
    for case in g["tokens_per_request"]:
        b = oracle_mod.kv_bytes_per_token(case["layers"], case["hidden"], case["bytes_per_elem"])
        gb = b * case["tokens"] / 1e9
        assert abs(gb - case["expected_gb_approx"]) <= case["rel_tol"] * case["expected_gb_approx"], case["cite"]
    for case in g["tokens_in_budget"]:
        b = oracle_mod.kv_bytes_per_token(case["layers"], case["hidden"], case["bytes_per_elem"])
        toks = case["budget_bytes"] / b
        assert abs(toks - case["expected_tokens_approx"]) <= case["rel_tol"] * case["expected_tokens_approx"], case["cite"]


def test_element_count_formula_matches_pages(oracle_mod):
    for case in _golden()["kv_elements"]:
        el = oracle_mod.kv_elements(case["batch"], case["layers"], case["seq"], case["head_dim"],
                                    case["heads"])
        assert el * case["bytes_per_elem"] == case["expected_gib"] * 2**30, case["cite"]


def test_gqa_fraction_matches_pages(oracle_mod):
    for case in _golden()["gqa_fraction"]:
        full = oracle_mod.kv_bytes_per_token(40, 5120, 2)
        grouped = oracle_mod.kv_bytes_per_token(40, 5120 // case["group"], 2)
        assert grouped / full == case["expected_fraction"], case["cite"]


def test_workload_sizes_follow_from_the_formula(oracle_mod):
    """The KV-movement workload's per-token bytes (all layers, K and V) equal M_kv."""
    plan = W.kvmove_plan(num_layers=40, num_sessions=2, swap_sessions=1)
    per_token_all_layers = plan.num_layers * 2 * plan.num_kv_heads * plan.head_dim * W.ELEM_BYTES[plan.dtype]
    assert per_token_all_layers == oracle_mod.kv_bytes_per_token(40, 5120, 2)
