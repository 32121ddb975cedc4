"""Pins for the float64 attention oracle (CPU only).

Each test checks the oracle against something other than itself:
  * torch's scaled_dot_product_attention (float64, explicit causal mask, GQA through the
    library's own ``enable_gqa`` convention) on caches written by an independent placement;
  * closed forms (first token, zero scale, one dominant key);
  * invariances the pages fix (block ids are only addresses; chunked turns equal one prefill;
    a decode step equals the single-query formula; GQA equals MHA with replicated K/V heads;
    prefix sharing equals copied blocks; unread slots never matter).
A final test plants mistakes in copies of the oracle source and checks the pins catch each one.
"""
import os
import subprocess
import tempfile

import numpy as np
import pytest
import torch

from paged_kv_cache_generalized_gb300 import workloads as W

pytestmark = pytest.mark.filterwarnings("ignore")


def _as_f64(x, dtype):
    """Storage array -> float64 through torch's own dtype conversion (independent of the oracle's
    hand-written bf16/f16 decoding)."""
    if dtype == "f32":
        return torch.from_numpy(np.asarray(x, dtype=np.float32)).double()
    t = torch.from_numpy(np.asarray(x).view(np.int16))
    return t.view(torch.bfloat16 if dtype == "bf16" else torch.float16).double()


def _place(seqs_k, seqs_v, bt, pool, Hkv, B, d, dtype):
    """Writes each sequence's contiguous K/V [n, Hkv, d] into a pool [pool, Hkv, B, d]: logical
    block lb of sequence i goes to physical block bt[i, lb]."""
    if dtype == "f32":
        kc = np.full((pool, Hkv, B, d), np.nan, dtype=np.float32)
    else:
        kc = np.full((pool, Hkv, B, d), W.NAN_BITS[dtype], dtype=np.uint16)
    vc = kc.copy()
    for i, (k, v) in enumerate(zip(seqs_k, seqs_v)):
        n = k.shape[0]
        for lb in range((n + B - 1) // B):
            lo, hi = lb * B, min(n, lb * B + B)
            kc[bt[i, lb], :, : hi - lo, :] = np.transpose(k[lo:hi], (1, 0, 2))
            vc[bt[i, lb], :, : hi - lo, :] = np.transpose(v[lo:hi], (1, 0, 2))
    return kc, vc


def _sdpa_case(ctx, ql, Hq, Hkv, d, B, dtype, seed, scale=None):
    rng = np.random.default_rng(seed)
    n = [c + q for c, q in zip(ctx, ql)]
    nb = [(x + B - 1) // B for x in n]
    pool = sum(nb) + 3
    perm = rng.permutation(pool)
    bt = np.full((len(n), max(nb)), -1, dtype=np.int32)
    pos = 0
    for i, k in enumerate(nb):
        bt[i, :k] = perm[pos:pos + k]
        pos += k
    ks = [W.random_values((x, Hkv, d), dtype, seed * 10 + 2 * i) for i, x in enumerate(n)]
    vs = [W.random_values((x, Hkv, d), dtype, seed * 10 + 2 * i + 1) for i, x in enumerate(n)]
    kc, vc = _place(ks, vs, bt, pool, Hkv, B, d, dtype)
    T = sum(ql)
    q = W.random_values((T, Hq, d), dtype, seed * 10 + 99)
    sc = 1.0 / np.sqrt(d) if scale is None else scale
    return dict(q=q, kc=kc, vc=vc, bt=bt, ks=ks, vs=vs, ctx=np.array(ctx, np.int32),
                ql=np.array(ql, np.int32), Hq=Hq, Hkv=Hkv, d=d, B=B, dtype=dtype, scale=sc)


def _run_oracle(oracle_mod, c, **over):
    args = dict(c)
    args.update(over)
    return oracle_mod.paged_attention(args["q"], args["kc"], args["vc"], args["dtype"], args["bt"],
                                      args["ctx"], args["ql"], args["Hq"], args["Hkv"], args["d"],
                                      args["B"], args["scale"])


def _sdpa_reference(c):
    """torch SDPA per sequence on the contiguous K/V, mask[j, p] = p <= ctx + j."""
    outs = []
    qt = _as_f64(c["q"], c["dtype"])
    cu = 0
    for i, (ctx, ql) in enumerate(zip(c["ctx"], c["ql"])):
        n = int(ctx) + int(ql)
        qi = qt[cu:cu + ql].permute(1, 0, 2).unsqueeze(0)            # [1, Hq, ql, d]
        ki = _as_f64(c["ks"][i], c["dtype"]).permute(1, 0, 2).unsqueeze(0)  # [1, Hkv, n, d]
        vi = _as_f64(c["vs"][i], c["dtype"]).permute(1, 0, 2).unsqueeze(0)
        mask = torch.arange(n)[None, :] <= (int(ctx) + torch.arange(int(ql)))[:, None]
        o = torch.nn.functional.scaled_dot_product_attention(
            qi, ki, vi, attn_mask=mask, scale=float(c["scale"]), enable_gqa=True)
        outs.append(o[0].permute(1, 0, 2))
        cu += ql
    return torch.cat(outs).numpy()


SDPA_CASES = [
    # ctx, q_lens, Hq, Hkv, d, B, dtype
    ([37, 50], [5, 1], 4, 4, 64, 16, "f32"),
    ([0, 1, 15, 16, 17], [1, 3, 2, 16, 40], 8, 2, 64, 16, "f32"),
    ([100, 33], [30, 7], 6, 3, 32, 32, "bf16"),
    ([70, 0], [1, 20], 4, 1, 128, 16, "f16"),
    ([5], [90], 2, 2, 16, 8, "f32"),
]


@pytest.mark.parametrize("case", SDPA_CASES)
def test_matches_torch_sdpa(oracle_mod, case):
    ctx, ql, Hq, Hkv, d, B, dtype = case
    c = _sdpa_case(ctx, ql, Hq, Hkv, d, B, dtype, seed=len(ctx) * 7 + d)
    got = _run_oracle(oracle_mod, c)
    ref = _sdpa_reference(c)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


def test_first_token_is_its_value_row(oracle_mod):
    """c = 0, q = 1: the only visible key is the token itself, so out = V_0 exactly."""
    c = _sdpa_case([0, 0], [1, 1], 4, 2, 64, 16, "bf16", seed=3)
    got = _run_oracle(oracle_mod, c)
    for i in range(2):
        v0 = _as_f64(c["vs"][i], "bf16")[0].numpy()          # [Hkv, d]
        np.testing.assert_array_equal(got[i], np.repeat(v0, 2, axis=0))


def test_zero_scale_is_mean_of_visible_values(oracle_mod):
    c = _sdpa_case([20, 3], [4, 2], 2, 2, 16, 8, "f32", seed=5, scale=0.0)
    got = _run_oracle(oracle_mod, c)
    cu = 0
    for i, (ctx, ql) in enumerate(zip(c["ctx"], c["ql"])):
        v = c["vs"][i].astype(np.float64)
        for j in range(ql):
            mean = v[: ctx + j + 1].mean(axis=0)                 # [Hkv, d]
            np.testing.assert_allclose(got[cu + j], mean, rtol=0, atol=1e-13)
        cu += ql


def test_one_dominant_key_selects_its_value(oracle_mod):
    """q aligned with one visible key (times a large factor): softmax is one-hot on it."""
    c = _sdpa_case([40], [1], 1, 1, 64, 16, "f32", seed=11)
    target = 17
    k = c["ks"][0][target, 0].astype(np.float64)
    q = (1.0e3 * k).astype(np.float32).reshape(1, 1, 64)
    got = _run_oracle(oracle_mod, c, q=q)
    np.testing.assert_allclose(got[0, 0], c["vs"][0][target, 0], rtol=0, atol=1e-12)


def test_block_id_permutation_invariance(oracle_mod):
    b = W.make_attn_batch("perm", [45, 3, 64], [7, 1, 33], 8, 4, 64, 16, "bf16", seed=21)
    ref = oracle_mod.paged_attention_batch(b)
    rng = np.random.default_rng(0)
    perm = rng.permutation(b.num_blocks)
    k2 = np.empty_like(b.k_cache)
    v2 = np.empty_like(b.v_cache)
    k2[perm] = b.k_cache
    v2[perm] = b.v_cache
    bt2 = np.where(b.block_tables >= 0, perm[np.maximum(b.block_tables, 0)], -1).astype(np.int32)
    got = oracle_mod.paged_attention(b.q, k2, v2, b.dtype, bt2, b.ctx_lens, b.q_lens, 8, 4, 64,
                                     16, b.scale)
    np.testing.assert_array_equal(got, ref)


def test_chunked_turn_equals_one_prefill(oracle_mod):
    """A new turn of q tokens attended at once equals the same turn attended in two chunks
    (q' then q'' with the context advanced by q'), and each token equals a q_len = 1 decode
    at context c + j (ConvKV turn-level prefix extension; causality)."""
    b = W.make_attn_batch("chunk", [29, 80], [19, 6], 4, 2, 64, 16, "f32", seed=31)
    full = oracle_mod.paged_attention_batch(b)
    args = (b.q, b.k_cache, b.v_cache, b.dtype)
    hd = (4, 2, 64, 16, b.scale)
    # chunks of sequence 0: 19 = 11 + 8 ; sequence 1 kept whole
    q0 = b.q[:19]
    part1 = oracle_mod.paged_attention(q0[:11], *args[1:], b.block_tables[:1], [29], [11], *hd)
    part2 = oracle_mod.paged_attention(q0[11:], *args[1:], b.block_tables[:1], [40], [8], *hd)
    np.testing.assert_array_equal(np.concatenate([part1, part2]), full[:19])
    # every token as a single-query decode
    for j in range(6):
        dec = oracle_mod.paged_attention(b.q[19 + j:20 + j], *args[1:], b.block_tables[1:2],
                                         [80 + j], [1], *hd)
        np.testing.assert_array_equal(dec[0], full[19 + j])


def test_gqa_equals_mha_with_replicated_kv_heads(oracle_mod):
    g = 4
    b = W.make_attn_batch("gqa", [23, 70], [9, 1], 8, 2, 64, 16, "bf16", seed=41)
    got = oracle_mod.paged_attention_batch(b)
    k_rep = np.repeat(b.k_cache, g, axis=1)    # KV head kh -> query heads kh*g .. kh*g+g-1
    v_rep = np.repeat(b.v_cache, g, axis=1)
    mha = oracle_mod.paged_attention(b.q, k_rep, v_rep, b.dtype, b.block_tables, b.ctx_lens,
                                     b.q_lens, 8, 8, 64, 16, b.scale)
    np.testing.assert_array_equal(got, mha)


def test_prefix_sharing_equals_copied_blocks(oracle_mod):
    b = W.make_attn_batch("prefix", [40, 50, 33], [4, 1, 2], 4, 4, 32, 8, "f32", seed=51,
                          shared_prefix_blocks=3, slack=1.0)
    got = oracle_mod.paged_attention_batch(b)
    assert (b.block_tables[1:, :3] == b.block_tables[0, :3]).all()
    # give sequences 1 and 2 private copies of the shared blocks
    used = set(int(x) for x in b.block_tables.ravel() if x >= 0)
    free = [x for x in range(b.num_blocks) if x not in used]
    k2, v2, bt2 = b.k_cache.copy(), b.v_cache.copy(), b.block_tables.copy()
    for i in (1, 2):
        for lb in range(3):
            dst = free.pop()
            k2[dst], v2[dst] = b.k_cache[bt2[i, lb]], b.v_cache[bt2[i, lb]]
            bt2[i, lb] = dst
    sep = oracle_mod.paged_attention(b.q, k2, v2, "f32", bt2, b.ctx_lens, b.q_lens, 4, 4, 32, 8,
                                     b.scale)
    np.testing.assert_array_equal(got, sep)


def test_unread_slots_do_not_matter(oracle_mod):
    """Free blocks, tail slots past each sequence's length and block-table padding may hold
    anything (NaN here); the output is unchanged and finite."""
    kw = dict(ctx_lens=[13, 60, 0], q_lens=[3, 1, 17], num_q_heads=4, num_kv_heads=2,
              head_dim=64, block_size=16, dtype="bf16", seed=61)
    clean = W.make_attn_batch("clean", poison=False, **kw)
    dirty = W.make_attn_batch("dirty", poison=True, **kw)
    assert np.isnan(W.to_storage(np.zeros(1, np.float32), "f32")).sum() == 0
    bt = dirty.block_tables.copy()
    bt[bt < 0] = 2 ** 30                            # padding past each sequence: garbage ids
    a = oracle_mod.paged_attention_batch(clean)
    bb = oracle_mod.paged_attention(dirty.q, dirty.k_cache, dirty.v_cache, "bf16", bt,
                                    dirty.ctx_lens, dirty.q_lens, 4, 2, 64, 16, dirty.scale)
    assert np.isfinite(a).all()
    np.testing.assert_array_equal(a, bb)


def test_row_subset_equals_full(oracle_mod):
    b = W.make_attn_batch("rows", [31, 5], [4, 9], 6, 2, 64, 16, "f16", seed=71)
    full = oracle_mod.paged_attention_batch(b)
    rows = np.array([[0, 0, 0], [0, 3, 5], [1, 8, 2], [1, 0, 4]])
    sub = oracle_mod.paged_attention_batch(b, rows=rows)
    cu = b.cu_q
    for r, (i, j, h) in enumerate(rows):
        np.testing.assert_array_equal(sub[r], full[cu[i] + j, h])


def test_threads_do_not_change_results(oracle_mod):
    b = W.make_attn_batch("thr", [100, 7, 64], [12, 1, 5], 8, 2, 64, 16, "bf16", seed=81)
    one = oracle_mod.paged_attention_batch(b, threads=1)
    many = oracle_mod.paged_attention_batch(b, threads=4)
    np.testing.assert_array_equal(one, many)


def test_out_of_range_block_is_an_error(oracle_mod):
    b = W.make_attn_batch("bad", [20], [2], 2, 2, 16, 16, "f32", seed=91)
    bt = b.block_tables.copy()
    bt[0, 1] = b.num_blocks + 5
    with pytest.raises(ValueError):
        oracle_mod.paged_attention(b.q, b.k_cache, b.v_cache, "f32", bt, b.ctx_lens, b.q_lens,
                                   2, 2, 16, 16, b.scale)


# --------------------------------------------------------------------------------------------
# Planted mistakes: each mutated copy of the oracle source must fail at least one pin.
# --------------------------------------------------------------------------------------------
MUTATIONS = {
    "gqa_map_modulo": ("const int64_t kh = h / group;", "const int64_t kh = h % num_kv_heads;"),
    "scale_dropped": ("s[p] = scale * dot;", "s[p] = dot;"),
    "slot_head_transposed": ("int64_t kbase = phys * block_stride + (kh * B + k) * d;",
                             "int64_t kbase = phys * block_stride + (k * num_kv_heads + kh) * d;"),
    "causal_off_by_one": ("const int64_t n = P + 1;", "const int64_t n = P;"),
    "causal_sees_next": ("const int64_t P = (int64_t)ctx_lens[i] + j;",
                         "const int64_t P = (int64_t)ctx_lens[i] + j + (j + 1 < q_lens[i]);"),
    "softmax_sign": ("s[p] = exp(s[p] - mx);", "s[p] = exp(mx - s[p]);"),
    "logical_block_ignored": ("int64_t phys = block_tables[i * (int64_t)max_blocks_per_seq + jb];\n            if (phys < 0",
                              "int64_t phys = block_tables[i * (int64_t)max_blocks_per_seq + 0];\n            if (phys < 0"),
}


def _build_mutant(src_text, name, tmpdir):
    c = os.path.join(tmpdir, f"{name}.c")
    so = os.path.join(tmpdir, f"lib{name}.so")
    with open(c, "w") as f:
        f.write(src_text)
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", c, "-o", so,
                    "-lm"], check=True, capture_output=True)
    return so


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(oracle_mod, name, monkeypatch):
    import ctypes

    src = open(os.path.join(os.path.dirname(oracle_mod.__file__), "attention.c")).read()
    old, new = MUTATIONS[name]
    assert src.count(old) >= 1, name
    mutated = src.replace(old, new, 1)
    with tempfile.TemporaryDirectory() as tmp:
        so = _build_mutant(mutated, name, tmp)
        lib = oracle_mod.declare(ctypes.CDLL(so))
        monkeypatch.setattr(oracle_mod, "_lib", lib)
        caught = False
        for case in SDPA_CASES:
            ctx, ql, Hq, Hkv, d, B, dtype = case
            c = _sdpa_case(ctx, ql, Hq, Hkv, d, B, dtype, seed=len(ctx) * 7 + d)
            try:
                got = _run_oracle(oracle_mod, c)
            except ValueError:
                caught = True
                break
            ref = _sdpa_reference(c)
            if not np.allclose(got, ref, rtol=0, atol=1e-12, equal_nan=False):
                caught = True
                break
        assert caught, f"planted mistake {name!r} passed every SDPA pin"
