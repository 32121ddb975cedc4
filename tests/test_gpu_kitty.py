"""GPU parity of the 2-bit page format with promoted 4-bit key channels ("KVキャッシュ管理の教科書"
第22章, Kitty) against the oracle, through the C ABI: the page quantiser bit for bit, decode
attention over quantised pages plus residual pages within the bf16 tolerances (every row of small
batches with ragged tails, exact page boundaries, tail-only sequences, MHA and GQA, bf16 and f16,
P = 16 and 32; sampled sequences of the full decode batch), bad lengths and ids flagged.

The oracle quantises the same bf16/f16 tokens itself: no expected value comes from the GPU."""
import numpy as np
import pytest
import torch

import oracle
from oracle import kitty
import paged_kv_cache_generalized_gb300 as pkg
from paged_kv_cache_generalized_gb300 import workloads as W

from gpu_util import as_f64, assert_close, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clean_status():
    pkg.device_status()
    yield


def gpu_state(b):
    R = kitty.record_bytes(b.promoted)
    d = dict(q=to_dev(b.q, b.dtype), stage_k=to_dev(b.stage_k, b.dtype), stage_v=to_dev(b.stage_v, b.dtype),
             res_k=to_dev(b.res_k, b.dtype), res_v=to_dev(b.res_v, b.dtype),
             pairs=to_dev(b.pairs), bt=to_dev(b.block_tables), ctx=to_dev(b.ctx_lens),
             ql=to_dev(b.q_lens))
    d["pages"] = torch.full((b.num_pages, b.num_kv_heads, R), 0xAB, dtype=torch.uint8, device="cuda")
    if len(b.pairs):
        pkg.kv_quantize_pages(d["stage_k"], d["stage_v"], d["pairs"], d["pages"], b.promoted)
    return d


def gpu_forward(b, d, **kw):
    out = pkg.pa_forward_kitty(d["q"], d["pages"], d["res_k"], d["res_v"], d["bt"], d["ctx"], d["ql"],
                               b.promoted, b.scale, **kw)
    torch.cuda.synchronize()
    return out


def oracle_rows(b, seqs):
    """Oracle outputs [len(seqs), Hq, d] of the given sequences: their pages quantised by the
    oracle from the same staging tokens, then the oracle's decode attention."""
    R = kitty.record_bytes(b.promoted)
    recs = []
    bt = np.full((len(seqs), b.block_tables.shape[1]), -1, np.int32)
    for si, i in enumerate(seqs):
        n = int(b.ctx_lens[i]) + 1
        for p, sid in enumerate(b.page_of[i]):
            rec = np.empty((b.num_kv_heads, R), np.uint8)
            for h in range(b.num_kv_heads):
                f = kitty.quantize_page(oracle.widen_f32(b.stage_k[sid, h], b.dtype),
                                        oracle.widen_f32(b.stage_v[sid, h], b.dtype), b.promoted)
                rec[h] = kitty.pack_record(f)
            bt[si, p] = len(recs)
            recs.append(rec)
        if n % 128:
            bt[si, n // 128] = b.block_tables[i, n // 128]
    pages = np.stack(recs) if recs else np.zeros((1, b.num_kv_heads, R), np.uint8)
    seqs = np.asarray(seqs)
    return kitty.paged_attention(b.q[seqs], pages, b.res_k, b.res_v, b.dtype, bt, b.ctx_lens[seqs],
                                 b.q_lens[seqs], b.num_q_heads, b.num_kv_heads, b.promoted, b.scale,
                                 threads=oracle.max_threads())


@pytest.mark.parametrize("dtype,P", [("bf16", 32), ("bf16", 16), ("f16", 32)])
def test_quantised_records_are_bit_exact(dtype, P):
    b = W.make_kitty_batch("q", [127, 128, 300, 700], 4, 2, P, dtype=dtype, seed=21)
    d = gpu_state(b)
    got = d["pages"].cpu().numpy()
    want = kitty.quantize_pages(b.stage_k, b.stage_v, b.pairs,
                                np.full(got.shape, 0xAB, np.uint8), P, dtype)
    assert np.array_equal(got, want)
    assert pkg.device_status() == 0


@pytest.mark.parametrize("hq,hkv,dtype,P", [(4, 4, "bf16", 32), (8, 2, "bf16", 16),
                                            (4, 4, "f16", 16), (8, 1, "f16", 32)])
def test_decode_matches_oracle_every_row(hq, hkv, dtype, P):
    # tail only (c = 0), one token short of a page, exactly one and two pages (no residual page),
    # one past a page, several items of eight pages with a tail, a long sequence
    lens = [0, 126, 127, 128, 255, 511, 700, 1800, 4100]
    b = W.make_kitty_batch("every_row", lens, hq, hkv, P, dtype=dtype, seed=hq + hkv + P)
    d = gpu_state(b)
    out = gpu_forward(b, d)
    assert pkg.device_status() == 0
    ref = oracle_rows(b, list(range(b.num_seqs)))
    assert_close(as_f64(out), ref, dtype, f"kitty {hq}/{hkv} {dtype} P={P}")


def test_deterministic_and_workspace_reuse():
    b = W.make_kitty_batch("det", [3000, 129, 640], 8, 8, 32, seed=5)
    d = gpu_state(b)
    ws = torch.empty(1 << 24, dtype=torch.uint8, device="cuda")
    a = gpu_forward(b, d, workspace=ws).clone()
    c = gpu_forward(b, d, workspace=ws)
    assert torch.equal(a.view(torch.int16), c.view(torch.int16))


def test_bad_lengths_and_ids_are_flagged():
    b = W.make_kitty_batch("bad", [300, 400], 4, 4, 16, seed=9)
    d = gpu_state(b)
    ql = d["ql"].clone()
    ql[1] = 2
    out = torch.zeros_like(d["q"])
    pkg.pa_forward_kitty(d["q"], d["pages"], d["res_k"], d["res_v"], d["bt"], d["ctx"], ql,
                         b.promoted, b.scale, out=out)
    torch.cuda.synchronize()
    assert pkg.device_status() & 0x2
    ref = oracle_rows(b, [0])
    assert_close(as_f64(out[:1]), ref, "bf16", "valid row beside a bad one")
    assert torch.count_nonzero(out[1].float()) == 0            # the bad row is not written
    bt = d["bt"].clone()
    bt[0, 0] = b.num_pages + 5
    pkg.pa_forward_kitty(d["q"], d["pages"], d["res_k"], d["res_v"], bt, d["ctx"], d["ql"],
                         b.promoted, b.scale)
    torch.cuda.synchronize()
    assert pkg.device_status() & 0x1
    pairs = d["pairs"][:1].clone()
    pairs[0, 1] = -3
    pkg.kv_quantize_pages(d["stage_k"], d["stage_v"], pairs, d["pages"], b.promoted)
    assert pkg.device_status() & 0x8


def test_refused_arguments():
    b = W.make_kitty_batch("arg", [300], 4, 4, 16, seed=3)
    d = gpu_state(b)
    with pytest.raises(pkg.PagedKVError):
        pkg.pa_forward_kitty(d["q"], d["pages"], d["res_k"], d["res_v"], d["bt"], d["ctx"], d["ql"],
                             24, b.scale)                      # P must be 16 or 32
    with pytest.raises(pkg.PagedKVError):
        pkg.pa_forward_kitty(d["q"], d["pages"], d["res_k"], d["res_v"], d["bt"], d["ctx"], d["ql"],
                             b.promoted, b.scale, workspace=torch.empty(256, dtype=torch.uint8, device="cuda"))


def test_full_decode_batch_sampled_sequences():
    b = W.decode13b_kitty()
    d = gpu_state(b)
    out = gpu_forward(b, d)
    assert pkg.device_status() == 0
    n = b.ctx_lens.astype(np.int64) + 1
    seqs = sorted({int(np.argmax(n)), int(np.argmin(n)), 7, 33})
    ref = oracle_rows(b, seqs)
    assert_close(as_f64(out[seqs]), ref, "bf16", "decode13b_kitty sampled sequences")
    # records of sampled pages, bit for bit
    pages = d["pages"]
    for sid in (0, len(b.pairs) // 2, len(b.pairs) - 1):
        t = int(b.pairs[sid, 1])
        for h in (0, 17, 39):
            f = kitty.quantize_page(oracle.widen_f32(b.stage_k[sid, h], "bf16"),
                                    oracle.widen_f32(b.stage_v[sid, h], "bf16"), b.promoted)
            assert np.array_equal(pages[t, h].cpu().numpy(), kitty.pack_record(f))


def test_long_sequence_merges_many_splits():
    # 60,001 tokens: 468 quantised pages in 59 items of 8 pages plus the residual page, so the
    # row's merge combines 60 split records (more than one warp-width of records)
    b = W.make_kitty_batch("long", [60000, 300], 4, 2, 32, seed=31)
    d = gpu_state(b)
    out = gpu_forward(b, d)
    assert pkg.device_status() == 0
    ref = oracle_rows(b, [0, 1])
    assert_close(as_f64(out), ref, "bf16", "kitty long sequence")
