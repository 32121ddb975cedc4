"""GPU parity of the 8-bit cache path (FP8 E4M3 codes, one scale for K and one for V) against the
float64 oracle, through the C ABI: the quantising append bit for bit, attention on E4M3 caches
within the bf16 tolerances (every row of small cases, sampled rows of the full decode batch).

Cache contents are N(0,1) values (the generator module's) encoded by the oracle's E4M3 encoder,
so the codes span the format's normal and subnormal range the way real K/V do."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_generalized_gb300 as pkg
from paged_kv_cache_generalized_gb300 import workloads as W

from gpu_util import as_f64, assert_close, gather_rows, sample_rows, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clean_status():
    pkg.device_status()
    yield


def _codes(shape, scale, seed):
    x = W.normal_f32(shape, seed)
    return oracle.e4m3_encode(x, np.float32(1.0) / np.float32(scale))


def _fp8_batch(name, ctx, ql, hq, hkv, B, dtype, ks, vs, seed, **kw):
    b = W.make_attn_batch(name, ctx, ql, hq, hkv, 128, B, dtype, seed=seed, poison=False, **kw)
    kc = _codes(b.k_cache.shape, ks, seed + 1)
    vc = _codes(b.v_cache.shape, vs, seed + 2)
    return b, kc, vc


def _run(b, kc, vc, ks, vs):
    q = to_dev(b.q, b.dtype)
    out = pkg.pa_forward(q, torch.from_numpy(kc).cuda(), torch.from_numpy(vc).cuda(),
                         to_dev(b.block_tables), to_dev(b.ctx_lens), to_dev(b.q_lens), b.scale,
                         k_scale=ks, v_scale=vs)
    torch.cuda.synchronize()
    assert pkg.device_status() == 0
    return out


CASES = [
    # name, ctx, q, Hq, Hkv, B, dtype, k_scale, v_scale
    ("decode_mha", [512, 1000, 37, 4096, 15], [1] * 5, 8, 8, 16, "bf16", 1 / 32, 1 / 16),
    ("decode_gqa4", [700, 33, 2000, 0], [1] * 4, 16, 4, 32, "bf16", 0.05, 0.02),
    ("decode_gqa2_f16", [300, 129, 64], [1] * 3, 8, 4, 16, "f16", 1 / 64, 1 / 64),
    ("turns_widened_gqa4", [300, 0, 129], [40, 33, 5], 8, 2, 16, "bf16", 0.03, 0.03),
    ("mha_turns", [100, 7], [20, 3], 4, 4, 64, "bf16", 1.0 / 8, 0.25),
    ("long_split", [16000, 9000], [1, 1], 8, 8, 32, "bf16", 1 / 32, 1 / 32),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_attention_on_e4m3_caches(case):
    name, ctx, ql, hq, hkv, B, dtype, ks, vs = case
    b, kc, vc = _fp8_batch(name, ctx, ql, hq, hkv, B, dtype, ks, vs, seed=len(name) * 13)
    out = _run(b, kc, vc, ks, vs)
    ref = oracle.paged_attention_batch(b, threads=8, kv=(kc, vc, ks, vs))
    assert_close(as_f64(out), ref, dtype, name)


def _uniform_codes(shape, seed):
    """Codes drawn uniformly over the 254 non-NaN codes (fast at full size)."""
    c = (W.random_bits16(shape, seed) & 0xFF).astype(np.uint8)
    c[(c & 0x7F) == 0x7F] ^= 0x01                       # S.1111.111 -> S.1111.110 (+-448)
    return c


def test_attention_on_e4m3_caches_decode13b_full_size():
    b = W.decode13b(poison=False)
    ks, vs = 1 / 512, 1 / 256                           # |values| <= 0.875, 1.75
    kc, vc = _uniform_codes(b.k_cache.shape, 71), _uniform_codes(b.v_cache.shape, 72)
    out = _run(b, kc, vc, ks, vs)
    rows = sample_rows(b, 256, seed=3)
    ref = oracle.paged_attention_batch(b, rows=rows, threads=16, kv=(kc, vc, ks, vs))
    assert_close(gather_rows(out, b, rows), ref, b.dtype, "decode13b e4m3")


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
def test_append_quantises_bit_exact(dtype):
    b = W.make_attn_batch("fp8app", [20, 3, 45], [5, 2, 17], 4, 2, 128, 16, dtype, seed=19, poison=False)
    ks, vs = 0.02, 0.5
    k0 = W.random_bits16(b.k_cache.shape, 4).astype(np.uint8)
    v0 = W.random_bits16(b.v_cache.shape, 5).astype(np.uint8)
    kn = W.normal_f32(b.k_new.shape, 6) * 3
    vn = W.normal_f32(b.v_new.shape, 7) * 300          # some values saturate
    kn_s, vn_s = W.to_storage(kn, dtype), W.to_storage(vn, dtype)
    kc, vc = torch.from_numpy(k0).cuda(), torch.from_numpy(v0).cuda()
    pkg.kv_append(to_dev(kn_s, dtype), to_dev(vn_s, dtype), to_dev(b.slot_mapping), kc, vc,
                  k_scale=ks, v_scale=vs)
    torch.cuda.synchronize()
    assert pkg.device_status() == 0
    ek, ev = oracle.kv_append_e4m3(kn_s, vn_s, b.slot_mapping, k0, v0, b.block_size, ks, vs, dtype)
    assert np.array_equal(kc.cpu().numpy(), ek)
    assert np.array_equal(vc.cpu().numpy(), ev)


def test_append_then_attend_matches_oracle():
    """The whole 8-bit step: bf16 new tokens quantised into the caches, then attention over them."""
    b = W.make_attn_batch("fp8step", [300, 64, 1000], [1, 40, 1], 16, 4, 128, 16, "bf16", seed=23,
                          poison=False)
    ks, vs = 1 / 40, 1 / 20
    k0, v0 = _codes(b.k_cache.shape, ks, 24), _codes(b.v_cache.shape, vs, 25)
    kc, vc = torch.from_numpy(k0).cuda(), torch.from_numpy(v0).cuda()
    pkg.kv_append(to_dev(b.k_new, "bf16"), to_dev(b.v_new, "bf16"), to_dev(b.slot_mapping), kc, vc,
                  k_scale=ks, v_scale=vs)
    out = pkg.pa_forward(to_dev(b.q, "bf16"), kc, vc, to_dev(b.block_tables), to_dev(b.ctx_lens),
                         to_dev(b.q_lens), b.scale, k_scale=ks, v_scale=vs)
    torch.cuda.synchronize()
    assert pkg.device_status() == 0
    ek, ev = oracle.kv_append_e4m3(b.k_new, b.v_new, b.slot_mapping, k0, v0, b.block_size, ks, vs, "bf16")
    assert np.array_equal(kc.cpu().numpy(), ek) and np.array_equal(vc.cpu().numpy(), ev)
    ref = oracle.paged_attention_batch(b, threads=8, kv=(ek, ev, ks, vs))
    assert_close(as_f64(out), ref, "bf16", "append then attend")


def test_append_quantises_every_layer_of_a_pool():
    """A [L, 2, num_blocks, Hkv, B, d] pool of E4M3 codes: one call quantises every layer's new
    tokens into that layer's K and V planes (strided views)."""
    b = W.make_attn_batch("fp8layers", [30, 7], [4, 3], 4, 2, 128, 16, "bf16", seed=29, poison=False)
    L, ks, vs = 3, 0.05, 0.2
    pool0 = (W.random_bits16((L, 2) + b.k_cache.shape, 30) & 0xFF).astype(np.uint8)
    new = [W.to_storage(W.normal_f32((2,) + b.k_new.shape, 31 + l), "bf16") for l in range(L)]
    pool = torch.from_numpy(pool0).cuda()
    kn = torch.stack([to_dev(x[0], "bf16") for x in new])
    vn = torch.stack([to_dev(x[1], "bf16") for x in new])
    pkg.kv_append(kn, vn, to_dev(b.slot_mapping), pool[:, 0], pool[:, 1], k_scale=ks, v_scale=vs)
    torch.cuda.synchronize()
    assert pkg.device_status() == 0
    got = pool.cpu().numpy()
    for l in range(L):
        ek, ev = oracle.kv_append_e4m3(new[l][0], new[l][1], b.slot_mapping, pool0[l, 0], pool0[l, 1],
                                       b.block_size, ks, vs, "bf16")
        assert np.array_equal(got[l, 0], ek) and np.array_equal(got[l, 1], ev), f"layer {l}"


def test_no_alloc_entry_point_on_e4m3_caches():
    b, kc, vc = _fp8_batch("fp8noalloc", [600, 31, 2000], [1, 1, 1], 16, 4, 32, "bf16", 1 / 16, 1 / 16, seed=41)
    q = to_dev(b.q, "bf16")
    args = (q, torch.from_numpy(kc).cuda(), torch.from_numpy(vc).cuda(), to_dev(b.block_tables),
            to_dev(b.ctx_lens), to_dev(b.q_lens), b.scale)
    a = pkg.pa_forward(*args, k_scale=1 / 16, v_scale=1 / 16)
    c = pkg.pa_forward_no_alloc(*args, k_scale=1 / 16, v_scale=1 / 16)
    torch.cuda.synchronize()
    assert pkg.device_status() == 0
    assert torch.equal(a, c)
    ref = oracle.paged_attention_batch(b, threads=8, kv=(kc, vc, 1 / 16, 1 / 16))
    assert_close(as_f64(c), ref, "bf16", "no-alloc e4m3")


# ---- multi-token turns on the tensor-core kernel: blocks widened into workspace scratch ----

def _up(x):
    return (x + 255) // 256 * 256


def _dev_args(b, kc, vc):
    return (to_dev(b.q, b.dtype), torch.from_numpy(kc).cuda(), torch.from_numpy(vc).cuda(),
            to_dev(b.block_tables), to_dev(b.ctx_lens), to_dev(b.q_lens))


def _forward_ws(b, kc, vc, ks, vs, extra=None):
    """pa_forward with a workspace of the required size plus ``extra`` widening bytes (None: the
    size the library asks for); returns (out, the planner's counters)."""
    q, k, v, bt, ctx, ql = _dev_args(b, kc, vc)
    full = pkg.forward_workspace_size(q, k, bt, ctx)
    widen = pkg.forward_widen_bytes(q, k, bt, ctx)
    nbytes = full if extra is None else full - widen + extra
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    out = pkg.pa_forward(q, k, v, bt, ctx, ql, b.scale, workspace=ws, k_scale=ks, v_scale=vs)
    torch.cuda.synchronize()
    return out, ws[:64].view(torch.int32).cpu().numpy()


TC_CASES = [
    # name, ctx, q, Hq, Hkv, B, dtype, k_scale, v_scale
    ("gqa4_bf16", [300, 0, 1000, 77], [130, 40, 257, 1], 16, 4, 16, "bf16", 0.03, 0.05),
    ("gqa8_f16_b32", [129, 513, 0], [64, 3, 300], 32, 4, 32, "f16", 1 / 64, 1 / 32),
    ("mha_b128", [200, 5, 640], [17, 16, 70], 4, 4, 128, "bf16", 0.25, 0.125),
    ("gqa2_b64_ragged", [1, 64, 127, 1500], [33, 100, 15, 9], 8, 4, 64, "bf16", 0.02, 0.02),
]


@pytest.mark.parametrize("case", TC_CASES, ids=[c[0] for c in TC_CASES])
def test_e4m3_turns_take_the_tensor_core_kernel(case):
    name, ctx, ql, hq, hkv, B, dtype, ks, vs = case
    b, kc, vc = _fp8_batch(name, ctx, ql, hq, hkv, B, dtype, ks, vs, seed=len(name) * 17)
    out, counters = _forward_ws(b, kc, vc, ks, vs)
    assert pkg.device_status() == 0
    g = hq // hkv
    cand = [i for i in range(len(ctx)) if ql[i] * g >= 16]
    blocks = sum((ctx[i] + ql[i] + B - 1) // B for i in cand)
    assert counters[7] == blocks, "widened blocks"
    assert counters[3] > 0, "no tile went to the tensor-core kernel"
    ref = oracle.paged_attention_batch(b, threads=8, kv=(kc, vc, ks, vs))
    assert_close(as_f64(out), ref, dtype, name)


def test_e4m3_scratch_capacity_decides_which_turns_widen():
    """Scratch for the first candidate's blocks only: it takes the tensor-core kernel, the later
    candidates run on CUDA cores; with no scratch every turn runs on CUDA cores.  Same results."""
    ctx, ql, B, hq, hkv = [700, 300, 50], [60, 200, 20], 16, 16, 4
    b, kc, vc = _fp8_batch("fp8cap", ctx, ql, hq, hkv, B, "bf16", 1 / 32, 1 / 16, seed=57)
    ref = oracle.paged_attention_batch(b, threads=8, kv=(kc, vc, 1 / 32, 1 / 16))
    S, mb = len(ctx), b.block_tables.shape[1]
    nb0 = (ctx[0] + ql[0] + B - 1) // B
    header = _up(4 * (S + 1)) + _up(4 * S * mb)
    blk = hkv * B * 128 * 2
    outs = []
    for extra, widened in ((header + nb0 * 2 * blk, nb0), (header + nb0 * 2 * blk + 2 * blk - 1, nb0), (0, None)):
        out, counters = _forward_ws(b, kc, vc, 1 / 32, 1 / 16, extra=extra)
        assert pkg.device_status() == 0
        if widened is None:
            assert counters[3] == 0
        else:
            assert counters[7] == widened and counters[3] > 0
        assert_close(as_f64(out), ref, "bf16", f"extra={extra}")
        outs.append(out)
    assert torch.equal(outs[0], outs[1])


def test_e4m3_widened_equals_bf16_caches_with_power_of_two_scales():
    """With power-of-two scales, bf16 caches holding code * scale give the tensor-core kernel
    operands that differ from the widened codes by exact powers of two, so the outputs agree bit
    for bit.  20 sequences x 8 KV heads of one tile pair each: 160 pair items, more than the SMs,
    so neither call cuts key ranges into chunks."""
    S, hq, hkv, B = 20, 32, 8, 16
    ctx = [int(x) for x in np.random.default_rng(5).integers(0, 700, S)]
    ql = [int(x) for x in np.random.default_rng(6).integers(4, 64, S)]
    ks, vs = 1 / 32, 1 / 8
    b, kc, vc = _fp8_batch("fp8pow2", ctx, ql, hq, hkv, B, "bf16", ks, vs, seed=61)
    out8, counters = _forward_ws(b, kc, vc, ks, vs)
    assert pkg.device_status() == 0 and counters[3] == S * hkv and counters[6] == 0
    k16 = (torch.from_numpy(kc).cuda().view(torch.float8_e4m3fn).float() * ks).to(torch.bfloat16)
    v16 = (torch.from_numpy(vc).cuda().view(torch.float8_e4m3fn).float() * vs).to(torch.bfloat16)
    q, _, _, bt, c, qlen = _dev_args(b, kc, vc)
    ws = torch.zeros(pkg.forward_workspace_size(q, k16, bt, c), dtype=torch.uint8, device="cuda")
    out16 = pkg.pa_forward(q, k16, v16, bt, c, qlen, b.scale, workspace=ws)
    torch.cuda.synchronize()
    assert pkg.device_status() == 0
    assert ws[:64].view(torch.int32)[6].item() == 0, "the bf16 call was chunked"
    assert torch.equal(out8, out16)


def test_e4m3_widening_flags_a_bad_block_id():
    """A bad id in a widened sequence's table is flagged; the other sequences' rows are unharmed."""
    b, kc, vc = _fp8_batch("fp8bad", [400, 90, 1000], [50, 30, 1], 16, 4, 16, "bf16", 1 / 32, 1 / 32, seed=67)
    ref = oracle.paged_attention_batch(b, threads=8, kv=(kc, vc, 1 / 32, 1 / 32))
    b.block_tables[0, 3] = b.k_cache.shape[0] + 5
    out, counters = _forward_ws(b, kc, vc, 1 / 32, 1 / 32)
    assert pkg.device_status() & 0x1                   # PA_DEV_BAD_BLOCK_ID
    assert counters[3] > 0
    keep = slice(int(b.q_lens[0]), int(b.q_lens.sum()))
    assert_close(as_f64(out)[keep], ref[keep], "bf16", "other sequences")


def test_e4m3_mixed_gqa_full_size():
    """The mixed GQA batch (32 resumed turns of 16-512 new tokens over 1K-16K histories + 32
    decodes) on E4M3 caches: turns widened onto the tensor-core kernel, sampled rows."""
    b = W.mixed_gqa(poison=False)
    ks, vs = 1 / 512, 1 / 256
    kc, vc = _uniform_codes(b.k_cache.shape, 73), _uniform_codes(b.v_cache.shape, 74)
    out, counters = _forward_ws(b, kc, vc, ks, vs)
    assert pkg.device_status() == 0
    assert counters[3] > 0 and counters[7] > 0
    rows = sample_rows(b, 192, seed=5)
    ref = oracle.paged_attention_batch(b, rows=rows, threads=16, kv=(kc, vc, ks, vs))
    assert_close(gather_rows(out, b, rows), ref, b.dtype, "mixed_gqa e4m3")


def test_e4m3_turns_on_a_block_first_pool():
    """Every layer of a block-first pool of E4M3 codes ([num_blocks, L, K|V, Hkv, B, d]): the
    widening reads each layer's blocks through the pool's block stride."""
    ctx, ql, ks, vs = [700, 90, 1500, 33], [40, 3, 130, 1], 1 / 32, 1 / 16
    b = W.make_attn_batch("fp8blockfirst", ctx, ql, 8, 2, 128, 16, "bf16", seed=81, poison=False)
    L = 3
    codes = [(_codes(b.k_cache.shape, ks, 82 + 2 * l), _codes(b.v_cache.shape, vs, 83 + 2 * l)) for l in range(L)]
    pool = torch.stack([torch.stack([torch.from_numpy(k), torch.from_numpy(v)], 1) for k, v in codes], 1).cuda()
    q, bt, c, qlen = to_dev(b.q, "bf16"), to_dev(b.block_tables), to_dev(b.ctx_lens), to_dev(b.q_lens)
    for layer, (k, v) in enumerate(codes):
        kc, vc = pool[:, layer, 0], pool[:, layer, 1]
        assert kc.stride(0) == L * 2 * kc[0].numel()
        ws = torch.zeros(pkg.forward_workspace_size(q, kc, bt, c), dtype=torch.uint8, device="cuda")
        out = pkg.pa_forward(q, kc, vc, bt, c, qlen, b.scale, workspace=ws, k_scale=ks, v_scale=vs)
        torch.cuda.synchronize()
        assert pkg.device_status() == 0
        assert ws[:64].view(torch.int32)[7].item() > 0, "no block was widened"
        ref = oracle.paged_attention_batch(b, threads=8, kv=(k, v, ks, vs))
        assert_close(as_f64(out), ref, "bf16", f"block-first e4m3 layer {layer}")


def test_no_alloc_entry_point_widens_e4m3_turns():
    """pa_forward_no_alloc on E4M3 turns: its fixed scratch past the required workspace holds this
    batch's widened blocks, so it runs the same kernels as pa_forward with the full widening
    workspace and returns the same bits."""
    ks, vs = 1 / 16, 1 / 32
    b, kc, vc = _fp8_batch("fp8noalloc_turns", [600, 31, 2000], [50, 1, 70], 16, 4, 32, "f16", ks, vs, seed=43)
    args = _dev_args(b, kc, vc) + (b.scale,)
    a = pkg.pa_forward(*args, k_scale=ks, v_scale=vs)
    c = pkg.pa_forward_no_alloc(*args, k_scale=ks, v_scale=vs)
    torch.cuda.synchronize()
    assert pkg.device_status() == 0
    assert torch.equal(a, c)
    ref = oracle.paged_attention_batch(b, threads=8, kv=(kc, vc, ks, vs))
    assert_close(as_f64(c), ref, "f16", "no-alloc e4m3 turns")


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_e4m3_few_turns_run_as_key_range_chunks(dtype):
    """One 64-token turn over a 20K-token history beside a decode row (GQA 16/2): 2 pair items,
    so with the whole widening workspace the key ranges run as chunks.  Within the oracle's bar,
    and (power-of-two scales) bit for bit the result of 16-bit caches holding code * scale, which
    chunk the same way."""
    ks, vs = 1 / 32, 1 / 16
    b, kc, vc = _fp8_batch("fp8chunks", [20000, 300], [64, 1], 16, 2, 16, dtype, ks, vs, seed=91)
    out8, counters = _forward_ws(b, kc, vc, ks, vs)
    assert pkg.device_status() == 0
    assert counters[3] > 0 and counters[6] > 0, "the pairs were not chunked"
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float16
    k16 = (torch.from_numpy(kc).cuda().view(torch.float8_e4m3fn).float() * ks).to(tdt)
    v16 = (torch.from_numpy(vc).cuda().view(torch.float8_e4m3fn).float() * vs).to(tdt)
    q, _, _, bt, c, qlen = _dev_args(b, kc, vc)
    ws = torch.zeros(pkg.forward_workspace_size(q, k16, bt, c), dtype=torch.uint8, device="cuda")
    out16 = pkg.pa_forward(q, k16, v16, bt, c, qlen, b.scale, workspace=ws)
    torch.cuda.synchronize()
    assert pkg.device_status() == 0
    assert ws[:64].view(torch.int32)[6].item() == counters[6]
    # the decode row runs on different CUDA-core kernels for the two cache types: compare the turn
    assert torch.equal(out8[:64], out16[:64])
    ref = oracle.paged_attention_batch(b, threads=16, kv=(kc, vc, ks, vs))
    assert_close(as_f64(out8), ref, dtype, f"e4m3 chunks {dtype}")
