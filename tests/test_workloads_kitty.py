"""Layout invariants of the generator's 2-bit page batches (host logic, no arithmetic of the
method): every full page of every sequence maps to its own record, the residual page of a
sequence with a partial page is its own, table padding is never a valid id, and residual slots
past a sequence's tail hold NaN (so a kernel that read them would be caught by the parity tests)."""
import numpy as np

from paged_kv_cache_generalized_gb300 import workloads as W

T = 128


def check(b):
    n = b.ctx_lens.astype(np.int64) + 1
    nfull = n // T
    assert len(b.pairs) == int(nfull.sum()) == b.stage_k.shape[0]
    assert len(np.unique(b.pairs[:, 1])) == len(b.pairs)                 # distinct records
    assert b.pairs[:, 1].min() >= 0 and b.pairs[:, 1].max() < b.num_pages
    res_ids = []
    for i in range(b.num_seqs):
        assert len(b.page_of[i]) == nfull[i]
        for p, sid in enumerate(b.page_of[i]):
            assert b.block_tables[i, p] == b.pairs[sid, 1]              # table -> record of page p
        width = b.block_tables.shape[1]
        used = int(nfull[i]) + (1 if n[i] % T else 0)
        assert np.all(b.block_tables[i, used:width] == -1)              # padding
        if n[i] % T:
            rid = int(b.block_tables[i, nfull[i]])
            res_ids.append(rid)
            tail = int(n[i] % T)
            slots = b.res_k[rid, :, tail:].reshape(-1)
            assert np.all((slots & 0x7FFF) > 0x7F80)                     # bf16 NaN patterns
            assert np.all((b.res_v[rid, :, tail:].reshape(-1) & 0x7FFF) > 0x7F80)
            assert np.all((b.res_k[rid, :, :tail].reshape(-1) & 0x7F80) != 0x7F80)   # finite tokens
    assert len(set(res_ids)) == len(res_ids)                            # distinct residual pages
    assert b.q.shape == (b.num_seqs, b.num_q_heads, 128) and np.all(b.q_lens == 1)


def test_small_batches():
    for lens, hq, hkv, P in (([0, 127, 128, 129, 255, 256, 4100], 4, 2, 32), ([300, 5], 8, 8, 16)):
        check(W.make_kitty_batch("t", lens, hq, hkv, P, seed=3))


def test_deterministic_by_seed():
    a = W.make_kitty_batch("t", [300, 700], 4, 2, 32, seed=8)
    b = W.make_kitty_batch("t", [300, 700], 4, 2, 32, seed=8)
    assert np.array_equal(a.stage_k, b.stage_k) and np.array_equal(a.block_tables, b.block_tables)
    assert np.array_equal(a.res_v, b.res_v) and np.array_equal(a.q, b.q)
