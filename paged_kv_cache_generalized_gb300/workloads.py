"""Seeded synthetic inputs for generalized paged attention, cache append and block copy.

This module is shared by the CUDA path's tests and benchmark and by the oracle's tests.  It holds
none of the method's arithmetic: it draws sequence lengths, lays out physical blocks, writes block
tables and slot maps, and fills tensors with N(0, 1) values (or raw 16-bit patterns).

Storage conventions (numpy has no bfloat16):
  * ``f32`` tensors are ``np.float32``;
  * ``bf16`` and ``f16`` tensors are ``np.uint16`` arrays holding the raw bit patterns.

Cache layout: ``[num_blocks, num_kv_heads, block_size, head_dim]`` per cache (K and V separate).
Query/output layout: packed ragged ``[total_q, num_q_heads, head_dim]`` in sequence order.

The shapes mirror the multi-turn serving batches on the pages (Pensieve's resumed conversations
with a new turn of several tokens, vLLM-style decode batches, ConvKV's non-contiguous turn
segments).  No dataset items are reproduced; lengths are drawn from uniform ranges.
"""
from __future__ import annotations

import concurrent.futures as _cf
import os
from dataclasses import dataclass, field

import numpy as np

DTYPES = ("f32", "bf16", "f16")
ELEM_BYTES = {"f32": 4, "bf16": 2, "f16": 2}
# quiet-NaN bit patterns used to poison slots that no sequence may read
NAN_BITS = {"bf16": 0x7FC0, "f16": 0x7E00}

_CHUNK = 1 << 24


def _rngs(seed: int, n: int):
    return [np.random.Generator(np.random.PCG64(s)) for s in np.random.SeedSequence(seed).spawn(n)]


def _threads() -> int:
    try:
        return max(1, min(16, len(os.sched_getaffinity(0))))
    except AttributeError:  # pragma: no cover
        return max(1, min(16, os.cpu_count() or 1))


def normal_f32(shape, seed: int) -> np.ndarray:
    """N(0,1) float32 values; chunked over independent child streams so the result depends only
    on (shape, seed), whatever the thread count."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.float32)
    nchunks = max(1, (n + _CHUNK - 1) // _CHUNK)
    gens = _rngs(seed, nchunks)

    def fill(i):
        lo, hi = i * _CHUNK, min(n, (i + 1) * _CHUNK)
        gens[i].standard_normal(hi - lo, dtype=np.float32, out=out[lo:hi])

    if nchunks == 1:
        fill(0)
    else:
        with _cf.ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(fill, range(nchunks)))
    return out.reshape(shape)


def random_bits16(shape, seed: int) -> np.ndarray:
    """Uniform random 16-bit patterns (NaN and Inf payloads included)."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    nchunks = max(1, (n + _CHUNK - 1) // _CHUNK)
    gens = _rngs(seed, nchunks)

    def fill(i):
        lo, hi = i * _CHUNK, min(n, (i + 1) * _CHUNK)
        out[lo:hi] = gens[i].integers(0, 1 << 16, hi - lo, dtype=np.uint16)

    if nchunks == 1:
        fill(0)
    else:
        with _cf.ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(fill, range(nchunks)))
    return out.reshape(shape)


def to_storage(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round float32 values to the storage dtype (round-to-nearest-even) and return the storage
    array (float32 for f32, uint16 bit patterns for bf16/f16)."""
    if dtype == "f32":
        return np.ascontiguousarray(x, dtype=np.float32)
    if dtype == "f16":
        return np.ascontiguousarray(x.astype(np.float16)).view(np.uint16)
    if dtype == "bf16":
        import torch  # the conversion routine only

        t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
        out = np.empty(x.shape, dtype=np.uint16)
        flat_in, flat_out = t.reshape(-1), out.reshape(-1)
        step = 1 << 26
        for lo in range(0, flat_in.numel(), step):
            flat_out[lo:lo + step] = flat_in[lo:lo + step].to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        return out
    raise ValueError(dtype)


def random_values(shape, dtype: str, seed: int) -> np.ndarray:
    return to_storage(normal_f32(shape, seed), dtype)


def nan_value(dtype: str):
    return np.float32(np.nan) if dtype == "f32" else np.uint16(NAN_BITS[dtype])


@dataclass
class AttnBatch:
    """One batch of generalized paged attention.

    Sequence i has ``ctx_lens[i]`` tokens cached before this step and ``q_lens[i]`` new query
    tokens.  The new tokens' K/V already sit in the cache at logical positions
    ``ctx_lens[i] .. ctx_lens[i] + q_lens[i] - 1`` (``k_new``/``v_new`` hold the same values and
    ``slot_mapping`` their physical slots, for the append step).
    """

    name: str
    dtype: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    ctx_lens: np.ndarray
    q_lens: np.ndarray
    block_tables: np.ndarray
    q: np.ndarray
    k_cache: np.ndarray
    v_cache: np.ndarray
    slot_mapping: np.ndarray
    k_new: np.ndarray
    v_new: np.ndarray
    scale: float
    seed: int
    meta: dict = field(default_factory=dict)

    @property
    def num_seqs(self) -> int:
        return int(self.ctx_lens.shape[0])

    @property
    def total_q(self) -> int:
        return int(self.q_lens.sum())

    @property
    def num_blocks(self) -> int:
        return int(self.k_cache.shape[0])

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def seq_lens(self) -> np.ndarray:
        return (self.ctx_lens.astype(np.int64) + self.q_lens.astype(np.int64))

    @property
    def cu_q(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.q_lens.astype(np.int64))])


def _blocks_needed(n_tokens: np.ndarray, B: int) -> np.ndarray:
    return (n_tokens.astype(np.int64) + B - 1) // B


def layout_shuffled(n_tokens: np.ndarray, B: int, slack: float, rng, pool_blocks: int | None = None):
    """Physical blocks drawn from one global shuffle of a pool sized for the batch plus ``slack``
    (or of exactly ``pool_blocks`` blocks)."""
    need = _blocks_needed(n_tokens, B)
    used = int(need.sum())
    pool = int(np.ceil((1.0 + slack) * used)) if pool_blocks is None else int(pool_blocks)
    assert pool >= used
    perm = rng.permutation(pool).astype(np.int32)
    max_blocks = max(1, int(need.max()))
    bt = np.full((len(n_tokens), max_blocks), -1, dtype=np.int32)
    pos = 0
    for i, nb in enumerate(need):
        bt[i, :nb] = perm[pos:pos + nb]
        pos += nb
    return bt, pool


def layout_segments(n_tokens: np.ndarray, B: int, seg_lo: int, seg_hi: int, slack: float, rng):
    """ConvKV-style turn segments: each sequence's tokens are cut into segments of
    U{seg_lo..seg_hi} tokens (rounded up to whole blocks); every segment occupies a contiguous
    physical run, and the runs of all sequences (plus free runs) are shuffled through the pool."""
    need = _blocks_needed(n_tokens, B)
    segs = []  # (seq, first logical block, nblocks)
    for i, nb in enumerate(need):
        lb = 0
        while lb < nb:
            t = int(rng.integers(seg_lo, seg_hi + 1))
            s = max(1, (t + B - 1) // B)
            s = min(s, int(nb) - lb)
            segs.append((i, lb, s))
            lb += s
    used = int(need.sum())
    free = int(np.ceil(slack * used))
    runs = list(segs)
    while free > 0:  # free runs, also segment-sized
        s = min(free, max(1, int(rng.integers(seg_lo, seg_hi + 1)) // B))
        runs.append((-1, 0, s))
        free -= s
    order = rng.permutation(len(runs))
    bt = np.full((len(n_tokens), max(1, int(need.max()))), -1, dtype=np.int32)
    pos = 0
    for k in order:
        i, lb, s = runs[k]
        if i >= 0:
            bt[i, lb:lb + s] = np.arange(pos, pos + s, dtype=np.int32)
        pos += s
    return bt, pos


def make_attn_batch(name, ctx_lens, q_lens, num_q_heads, num_kv_heads, head_dim, block_size,
                    dtype, seed, layout="shuffle", slack=0.1, seg=(64, 1024), poison=True,
                    shared_prefix_blocks=0, scale=None, pool_blocks=None) -> AttnBatch:
    """Build a batch: lengths as given, block tables by ``layout``, values N(0,1) rounded to
    ``dtype``.  ``shared_prefix_blocks`` > 0 makes every sequence alias the first blocks of
    sequence 0 (prefix sharing; those sequences must have at least that many full blocks)."""
    assert dtype in DTYPES
    rng = np.random.Generator(np.random.PCG64(seed))
    ctx = np.asarray(ctx_lens, dtype=np.int32)
    ql = np.asarray(q_lens, dtype=np.int32)
    assert (ql >= 1).all() and (ctx >= 0).all()
    n = ctx.astype(np.int64) + ql
    B = block_size
    if layout == "shuffle":  # one seeded permutation of the whole pool
        bt, pool = layout_shuffled(n, B, slack, rng, pool_blocks)
    elif layout == "segments":
        bt, pool = layout_segments(n, B, seg[0], seg[1], slack, rng)
    else:
        raise ValueError(layout)
    if shared_prefix_blocks:
        k = shared_prefix_blocks
        assert (n >= k * B).all()
        bt[1:, :k] = bt[0, :k]
    Hq, Hkv, d = num_q_heads, num_kv_heads, head_dim
    T = int(ql.sum())
    k_cache = random_values((pool, Hkv, B, d), dtype, seed * 1000 + 1)
    v_cache = random_values((pool, Hkv, B, d), dtype, seed * 1000 + 2)
    q = random_values((T, Hq, d), dtype, seed * 1000 + 3)
    if poison:
        live = np.zeros(pool, dtype=bool)
        nan = nan_value(dtype)
        for i in range(len(n)):
            nb = int((n[i] + B - 1) // B)
            live[bt[i, :nb]] = True
        k_cache[~live] = nan
        v_cache[~live] = nan
        # unused tail slots of each sequence's last block (unless another sequence reads them)
        readers = {}
        for i in range(len(n)):
            nb = int((n[i] + B - 1) // B)
            for lb in range(nb):
                used = min(B, int(n[i]) - lb * B)
                pb = int(bt[i, lb])
                readers[pb] = max(readers.get(pb, 0), used)
        for pb, used in readers.items():
            if used < B:
                k_cache[pb, :, used:, :] = nan
                v_cache[pb, :, used:, :] = nan
    # the step's new tokens: their K/V (already in the cache) and their slots
    cu = np.concatenate([[0], np.cumsum(ql.astype(np.int64))])
    slots = np.empty(T, dtype=np.int64)
    for i in range(len(n)):
        for j in range(int(ql[i])):
            p = int(ctx[i]) + j
            slots[cu[i] + j] = int(bt[i, p // B]) * B + p % B
    blk, off = slots // B, slots % B
    k_new = np.ascontiguousarray(k_cache[blk, :, off, :])
    v_new = np.ascontiguousarray(v_cache[blk, :, off, :])
    sc = float(1.0 / np.sqrt(d)) if scale is None else float(scale)
    return AttnBatch(name, dtype, Hq, Hkv, d, B, ctx, ql, bt, q, k_cache, v_cache, slots,
                     k_new, v_new, sc, seed, {"layout": layout, "pool_blocks": pool})


# ---------------------------------------------------------------------------------------------
# The five workloads (sizes as stated for the benchmark configurations).
# ---------------------------------------------------------------------------------------------

def tiny(seed: int = 1) -> AttnBatch:
    """1 layer, 4 query / 4 KV heads, head_dim 64, fp32, block size 16, a 16-block pool drawn as a
    seeded permutation; two sequences with 37 and 50 cached tokens and 5 and 1 new tokens."""
    return make_attn_batch("tiny", [37, 50], [5, 1], 4, 4, 64, 16, "f32", seed,
                           layout="shuffle", pool_blocks=16)


def decode13b_lengths(seed: int = 2, num_seqs: int = 64, lo: int = 512, hi: int = 4096):
    rng = np.random.Generator(np.random.PCG64(seed + 100))
    return rng.integers(lo, hi + 1, num_seqs).astype(np.int32)


def decode13b(seed: int = 2, num_seqs: int = 64, lo: int = 512, hi: int = 4096, **kw) -> AttnBatch:
    """Llama-2-13B-shaped decode batch: 40 MHA heads, head_dim 128, bf16, block size 16,
    q_len 1, cached context U{lo..hi}, blocks shuffled through a pool with 10% free."""
    ctx = decode13b_lengths(seed, num_seqs, lo, hi)
    return make_attn_batch("decode13b", ctx, np.ones_like(ctx), 40, 40, 128, 16, "bf16", seed,
                           layout="shuffle", slack=0.1, **kw)


def mixed_gqa_lengths(seed: int = 3, n_resume: int = 32, n_decode: int = 32,
                      hist=(1024, 16384), turn=(16, 512), dec=(256, 8192)):
    rng = np.random.Generator(np.random.PCG64(seed + 100))
    c_r = rng.integers(hist[0], hist[1] + 1, n_resume)
    q_r = rng.integers(turn[0], turn[1] + 1, n_resume)
    c_d = rng.integers(dec[0], dec[1] + 1, n_decode)
    ctx = np.concatenate([c_r, c_d]).astype(np.int32)
    ql = np.concatenate([q_r, np.ones(n_decode, dtype=np.int64)]).astype(np.int32)
    order = rng.permutation(len(ctx))
    return ctx[order], ql[order]


def mixed_gqa(seed: int = 3, n_resume: int = 32, n_decode: int = 32, hist=(1024, 16384),
              turn=(16, 512), dec=(256, 8192), **kw) -> AttnBatch:
    """Pensieve-style mixed batch: GQA 32 query / 8 KV heads, head_dim 128, bf16, block size 32;
    resumed conversations (history U{hist}, new turn U{turn}) mixed with decode sequences."""
    ctx, ql = mixed_gqa_lengths(seed, n_resume, n_decode, hist, turn, dec)
    return make_attn_batch("mixed_gqa", ctx, ql, 32, 8, 128, 32, "bf16", seed,
                           layout="shuffle", slack=0.1, **kw)


def longprefill(seed: int = 4, num_seqs: int = 8, ctx: int = 16384, q: int = 2048, **kw) -> AttnBatch:
    """Prefill-heavy batch: 40 MHA heads, head_dim 128, bf16, block size 16; every sequence has
    ``ctx`` cached and ``q`` new tokens; block tables made of ConvKV-style turn segments
    (64..1024 tokens) on shuffled physical runs."""
    return make_attn_batch("longprefill", [ctx] * num_seqs, [q] * num_seqs, 40, 40, 128, 16,
                           "bf16", seed, layout="segments", slack=0.05, seg=(64, 1024), **kw)


# ---------------------------------------------------------------------------------------------
# KV movement (append into partially filled blocks, copy-on-write copies, swap-in scatter).
# ---------------------------------------------------------------------------------------------

@dataclass
class KVMovePlan:
    """Structure of a KV-movement step (no tensor values: those are drawn separately).

    Pool layout on the device: ``[num_layers, 2 (K,V), num_blocks, num_kv_heads, block_size,
    head_dim]``; one *plane* is one (layer, K|V) slice, so a block copy moves every plane.
    """

    num_layers: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    dtype: str
    num_blocks: int
    seq_lens: np.ndarray          # tokens cached before the append
    new_lens: np.ndarray          # tokens appended this step
    block_tables: np.ndarray      # after CoW remapping and growth, covers seq_lens + new_lens
    slot_mapping: np.ndarray      # int64 [T_new]
    cow_pairs: np.ndarray         # int64 [P, 2] (src block, dst block), both on the device pool
    swap_pairs: np.ndarray        # int64 [S, 2] (host block, device block)
    num_host_blocks: int
    seed: int

    @property
    def block_bytes(self) -> int:  # one plane
        return self.num_kv_heads * self.block_size * self.head_dim * ELEM_BYTES[self.dtype]


def kvmove_plan(seed: int = 5, num_layers: int = 8, num_sessions: int = 64, lens=(512, 8192),
                new=(1, 256), num_kv_heads: int = 40, head_dim: int = 128, block_size: int = 32,
                cow_frac: float = 0.10, refs=(2, 4), swap_sessions: int = 8) -> KVMovePlan:
    """KV movement at the Llama-2-13B shape (40 layers x 5120 hidden, fp16, 32-token blocks).

    * ``num_sessions`` sessions of U{lens} cached tokens; each appends U{new} tokens, first into
      its partially filled last block, then into fresh blocks.
    * ``cow_frac`` of the sessions' blocks are shared by U{refs} sequences: each such block gets
      (r - 1) copy-on-write copies into free blocks.
    * ``swap_sessions`` further sessions live in a host-pinned pool and are swapped in, block by
      block, into free device blocks.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    B = block_size
    L = rng.integers(lens[0], lens[1] + 1, num_sessions).astype(np.int64)
    add = rng.integers(new[0], new[1] + 1, num_sessions).astype(np.int64)
    have = (L + B - 1) // B
    need = (L + add + B - 1) // B
    resident = int(have.sum())
    cow_src = rng.choice(resident, int(round(cow_frac * resident)), replace=False)
    r = rng.integers(refs[0], refs[1] + 1, len(cow_src))
    n_cow = int((r - 1).sum())
    grow = int((need - have).sum())
    Ls = rng.integers(lens[0], lens[1] + 1, swap_sessions).astype(np.int64)
    n_swap = int(((Ls + B - 1) // B).sum())
    pool = resident + n_cow + grow + n_swap
    pool = int(np.ceil(pool * 1.02))
    perm = rng.permutation(pool).astype(np.int64)
    cursor = 0

    def take(k):
        nonlocal cursor
        out = perm[cursor:cursor + k]
        cursor += k
        return out

    bt = np.full((num_sessions, int(need.max())), -1, dtype=np.int32)
    for i in range(num_sessions):
        bt[i, :have[i]] = take(int(have[i]))
    flat_res = np.concatenate([bt[i, :have[i]] for i in range(num_sessions)]).astype(np.int64)
    src = np.repeat(flat_res[cow_src], r - 1)
    dst = take(n_cow)
    cow_pairs = np.stack([src, dst], axis=1).astype(np.int64)
    slots = []
    for i in range(num_sessions):
        bt[i, have[i]:need[i]] = take(int(need[i] - have[i]))
        for p in range(int(L[i]), int(L[i] + add[i])):
            slots.append(int(bt[i, p // B]) * B + p % B)
    swap_dst = take(n_swap)
    swap_pairs = np.stack([np.arange(n_swap, dtype=np.int64), swap_dst], axis=1)
    return KVMovePlan(num_layers, num_kv_heads, head_dim, B, "f16", pool, L.astype(np.int32),
                      add.astype(np.int32), bt, np.asarray(slots, dtype=np.int64), cow_pairs,
                      swap_pairs, n_swap, seed)


def shrink_plan_layers(plan: KVMovePlan, num_layers: int) -> KVMovePlan:
    from dataclasses import replace
    return replace(plan, num_layers=num_layers)


# ---------------------------------------------------------------------------------------------
# Layer-pipelined swap-in (a batch whose resumed conversations left part of their history on the
# CPU tier).
# ---------------------------------------------------------------------------------------------

def swap_plan(batch: AttnBatch, frac: float = 0.125) -> np.ndarray:
    """Device blocks whose contents come back from the CPU tier before this step's attention: the
    earliest ``frac`` of every resumed conversation's cached history (Pensieve evicts a
    conversation's chunks from its earlier end), whole blocks only.  Host block i of the returned
    list goes to device block ``out[i]``; a session's blocks are consecutive on the host, so each
    layer's swapped blocks form one contiguous host region per plane."""
    B = batch.block_size
    out = []
    for i in range(batch.num_seqs):
        if int(batch.q_lens[i]) <= 1:
            continue                                   # decode steps stayed resident
        k = int(frac * int(batch.ctx_lens[i])) // B
        out.extend(int(x) for x in batch.block_tables[i, :k])
    return np.asarray(out, dtype=np.int64)


@dataclass
class KittyBatch:
    """A decode batch over 2-bit pages with promoted key channels ("KVキャッシュ管理の教科書"
    第22章, Kitty), before quantisation: every full 128-token page's tokens sit in a staging pool
    in the residual-page format (``stage_k``/``stage_v`` [num_full, Hkv, 128, d]); ``pairs`` maps
    staging page s to its record id t in a pool of ``num_pages`` records.  Each sequence's last
    n % 128 tokens sit in residual page ``block_tables[i][n // 128]`` of ``res_k``/``res_v`` (later
    slots NaN-poisoned: never read).  Sequence i has n_i = ctx_lens[i] + 1 tokens; q is
    [S, Hq, d]."""
    name: str
    dtype: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    promoted: int
    scale: float
    q: np.ndarray
    ctx_lens: np.ndarray
    q_lens: np.ndarray
    stage_k: np.ndarray
    stage_v: np.ndarray
    pairs: np.ndarray
    num_pages: int
    res_k: np.ndarray
    res_v: np.ndarray
    block_tables: np.ndarray
    page_of: list = field(default_factory=list)   # per sequence: staging ids of its full pages

    @property
    def num_seqs(self) -> int:
        return len(self.ctx_lens)


def make_kitty_batch(name, ctx_lens, num_q_heads, num_kv_heads, promoted, dtype="bf16", seed=7,
                     slack=0.1, head_dim=128):
    T = 128
    rng = np.random.Generator(np.random.PCG64(seed + 300))
    ctx = np.asarray(ctx_lens, dtype=np.int32)
    n = ctx.astype(np.int64) + 1
    nfull = n // T
    num_full = int(nfull.sum())
    has_tail = (n % T) > 0
    num_res = int(has_tail.sum()) + 2
    num_pages = int(np.ceil(num_full * (1 + slack))) + 1
    S = len(ctx)
    maxp = int(((n + T - 1) // T).max())
    stage_k = random_values((num_full, num_kv_heads, T, head_dim), dtype, seed * 1000 + 1)
    stage_v = random_values((num_full, num_kv_heads, T, head_dim), dtype, seed * 1000 + 2)
    rec_ids = rng.permutation(num_pages)[:num_full]
    pairs = np.stack([np.arange(num_full), rec_ids], axis=1).astype(np.int64)
    res_k = random_values((num_res, num_kv_heads, T, head_dim), dtype, seed * 1000 + 3)
    res_v = random_values((num_res, num_kv_heads, T, head_dim), dtype, seed * 1000 + 4)
    res_ids = rng.permutation(num_res)
    bt = np.full((S, maxp), -1, dtype=np.int32)
    page_of = []
    j = r = 0
    for i in range(S):
        page_of.append(list(range(j, j + int(nfull[i]))))
        bt[i, :nfull[i]] = rec_ids[j:j + nfull[i]]
        j += int(nfull[i])
        if has_tail[i]:
            rid = int(res_ids[r])
            r += 1
            bt[i, nfull[i]] = rid
            tail = int(n[i] % T)
            res_k[rid, :, tail:] = nan_value(dtype)
            res_v[rid, :, tail:] = nan_value(dtype)
    q = random_values((S, num_q_heads, head_dim), dtype, seed * 1000 + 5)
    return KittyBatch(name, dtype, num_q_heads, num_kv_heads, head_dim, promoted,
                      1.0 / float(np.sqrt(head_dim)), q, ctx, np.ones(S, np.int32), stage_k,
                      stage_v, pairs, num_pages, res_k, res_v, bt, page_of)


def decode13b_kitty(seed: int = 2, num_seqs: int = 64, lo: int = 512, hi: int = 4096, promoted: int = 32,
                    **kw) -> KittyBatch:
    """The decode13b batch (40 MHA heads, head_dim 128, bf16, context U{lo..hi}) over 2-bit pages
    with ``promoted`` 4-bit key channels."""
    ctx = decode13b_lengths(seed, num_seqs, lo, hi)
    return make_kitty_batch("decode13b_kitty", ctx, 40, 40, promoted, seed=seed, **kw)
