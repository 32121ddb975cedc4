"""GPU: pa_forward_append (the step's cache append written by extra blocks of the planner's
launch, then the attention) against the oracle's append and attention, and bit for bit against
kv_append followed by pa_forward on the same inputs.

The new tokens' slots start out NaN (or random E4M3 codes), so a token the fused append failed to
write shows as a cache mismatch and as NaN in every output row that attends to it."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_generalized_gb300 as pkg
from paged_kv_cache_generalized_gb300 import workloads as W

from gpu_util import as_f64, assert_close, bits, gather_rows, sample_rows, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clean_status():
    pkg.device_status()
    yield


def _scrub(cache, slots, B, fill):
    """A copy of ``cache`` ([num_blocks, Hkv, B, d]) with every slot in ``slots`` set to ``fill``."""
    c = cache.copy()
    for s in np.asarray(slots, dtype=np.int64):
        if s >= 0:
            c[s // B, :, s % B, :] = fill
    return c


def _both_paths(b, kc0, vc0, kn, vn, slots, **kw):
    """(out, k, v) of kv_append + pa_forward and of pa_forward_append, each from copies of
    kc0 / vc0 on the device."""
    q = to_dev(b.q, b.dtype)
    bt, ctx, ql = to_dev(b.block_tables), to_dev(b.ctx_lens), to_dev(b.q_lens)
    cdt = None if kc0.dtype == np.uint8 else b.dtype
    kn_d, vn_d, sm = to_dev(kn, b.dtype), to_dev(vn, b.dtype), to_dev(slots)
    k1, v1 = to_dev(kc0, cdt), to_dev(vc0, cdt)
    pkg.kv_append(kn_d, vn_d, sm, k1, v1, **kw)
    ref = pkg.pa_forward(q, k1, v1, bt, ctx, ql, b.scale, **kw)
    k2, v2 = to_dev(kc0, cdt), to_dev(vc0, cdt)
    out = pkg.pa_forward_append(q, kn_d, vn_d, sm, k2, v2, bt, ctx, ql, b.scale, **kw)
    torch.cuda.synchronize()
    return (ref, k1, v1), (out, k2, v2)


CASES = [
    # name, ctx_lens, q_lens, Hq, Hkv, d, B, dtype
    ("decode_gqa4_bf16", [700, 33, 2000, 0, 31], [1] * 5, 16, 4, 128, 32, "bf16"),
    ("mixed_tensor_core_bf16", [500, 100, 2000, 33, 0, 700], [1, 130, 1, 17, 64, 1], 32, 8, 128, 32,
     "bf16"),
    ("prefill_mha_f16", [300, 0, 129], [200, 150, 33], 4, 4, 128, 16, "f16"),
    ("short_turns_gqa4_bf16", [100, 513, 0, 47], [3, 2, 1, 1], 16, 4, 128, 16, "bf16"),
    ("prefill_d64_f32", [60, 0, 17], [40, 33, 1], 4, 2, 64, 16, "f32"),
    ("block128_bf16", [300, 5], [130, 1], 4, 1, 128, 128, "bf16"),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_fused_append_matches_oracle_and_separate_calls(case):
    name, ctx, ql, hq, hkv, d, B, dtype = case
    b = W.make_attn_batch(name, ctx, ql, hq, hkv, d, B, dtype, seed=len(name) * 7 + B)
    nan = W.nan_value(dtype)
    kc0 = _scrub(b.k_cache, b.slot_mapping, B, nan)
    vc0 = _scrub(b.v_cache, b.slot_mapping, B, nan)
    (ref, k1, v1), (out, k2, v2) = _both_paths(b, kc0, vc0, b.k_new, b.v_new, b.slot_mapping)
    assert pkg.device_status() == 0
    ek, ev = oracle.kv_append(b.k_new, b.v_new, b.slot_mapping, kc0, vc0, B)
    assert bits(k2).tobytes() == ek.tobytes()
    assert bits(v2).tobytes() == ev.tobytes()
    assert bits(k1).tobytes() == ek.tobytes()
    assert torch.equal(out, ref)
    assert_close(as_f64(out), oracle.paged_attention_batch(b, threads=8), dtype, name)


def test_fused_append_e4m3_caches():
    """E4M3 caches: a quantising append, then the attention on the codes."""
    ks, vs = 1 / 32, 1 / 16
    b = W.make_attn_batch("app_e4m3", [512, 37, 1000, 0], [1, 40, 1, 3], 8, 2, 128, 16, "bf16",
                          seed=91, poison=False)
    # cached codes of N(0,1) values, as real K/V are (the new tokens' slots are overwritten)
    kc0 = oracle.e4m3_encode(W.normal_f32(b.k_cache.shape, 92), np.float32(1.0) / np.float32(ks))
    vc0 = oracle.e4m3_encode(W.normal_f32(b.v_cache.shape, 93), np.float32(1.0) / np.float32(vs))
    (ref, k1, v1), (out, k2, v2) = _both_paths(b, kc0, vc0, b.k_new, b.v_new, b.slot_mapping,
                                               k_scale=ks, v_scale=vs)
    assert pkg.device_status() == 0
    ek, ev = oracle.kv_append_e4m3(b.k_new, b.v_new, b.slot_mapping, kc0, vc0, 16, ks, vs, "bf16")
    assert bits(k2).tobytes() == ek.tobytes()
    assert bits(v2).tobytes() == ev.tobytes()
    assert torch.equal(out, ref)
    expect = oracle.paged_attention_batch(b, threads=8, kv=(ek, ev, ks, vs))
    assert_close(as_f64(out), expect, "bf16", "app_e4m3")


def test_fused_append_padding_and_bad_slot():
    """slot < 0 is skipped; a slot past the pool is skipped and flagged; the other tokens land."""
    B = 16
    b = W.make_attn_batch("app_bad", [40, 0, 70], [1, 20, 1], 4, 4, 128, B, "bf16", seed=17)
    slots = b.slot_mapping.copy()
    slots[0] = -1
    slots[5] = b.k_cache.shape[0] * B + 3
    rnd_k = W.random_bits16(b.k_cache.shape, 18)
    rnd_v = W.random_bits16(b.v_cache.shape, 19)
    (_, k1, v1), (_, k2, v2) = _both_paths(b, rnd_k, rnd_v, b.k_new, b.v_new, slots)
    assert pkg.device_status() & 0x4                  # PA_DEV_BAD_SLOT
    keep = slots.copy()
    keep[5] = -1
    ek, ev = oracle.kv_append(b.k_new, b.v_new, keep, rnd_k, rnd_v, B)
    assert bits(k2).tobytes() == ek.tobytes() == bits(k1).tobytes()
    assert bits(v2).tobytes() == ev.tobytes() == bits(v1).tobytes()


def test_fused_append_mixed_gqa_full_size():
    """The mixed GQA batch (32 resumed turns of 16-512 new tokens + 32 decodes), sampled rows."""
    b = W.mixed_gqa()
    kc0 = _scrub(b.k_cache, b.slot_mapping, b.block_size, W.nan_value(b.dtype))
    vc0 = _scrub(b.v_cache, b.slot_mapping, b.block_size, W.nan_value(b.dtype))
    (ref, k1, _), (out, k2, _) = _both_paths(b, kc0, vc0, b.k_new, b.v_new, b.slot_mapping)
    assert pkg.device_status() == 0
    assert torch.equal(k2.view(torch.int16), k1.view(torch.int16))   # bits: unread slots hold NaN
    assert torch.equal(out, ref)
    rows = sample_rows(b, 192, seed=11)
    assert_close(gather_rows(out, b, rows), oracle.paged_attention_batch(b, rows=rows, threads=16),
                 b.dtype, "mixed_gqa")


def test_timing_events_bracket_the_kernels():
    """The events the library records around its tensor-core and decode kernels lie inside the
    caller's bracket of the whole call, and the call's results are unchanged by them."""
    b = W.make_attn_batch("timed", [500, 100, 2000, 0], [1, 130, 1, 64], 32, 8, 128, 32, "bf16", seed=5)
    q = to_dev(b.q, b.dtype)
    k, v = to_dev(b.k_cache, b.dtype), to_dev(b.v_cache, b.dtype)
    bt, ctx, ql = to_dev(b.block_tables), to_dev(b.ctx_lens), to_dev(b.q_lens)
    ref = pkg.pa_forward(q, k, v, bt, ctx, ql, b.scale)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
    pkg.set_timing_events(tc=(ev[2], ev[3]), cc=(ev[4], ev[5]))
    try:
        ev[0].record()
        out = pkg.pa_forward(q, k, v, bt, ctx, ql, b.scale)
        ev[1].record()
    finally:
        pkg.set_timing_events()
    torch.cuda.synchronize()
    assert pkg.device_status() == 0
    assert torch.equal(out, ref)
    call = ev[0].elapsed_time(ev[1])
    tc = ev[2].elapsed_time(ev[3])
    cc = ev[4].elapsed_time(ev[5])
    assert 0 < tc <= call and 0 < cc <= call
    assert ev[0].elapsed_time(ev[2]) >= 0 and ev[3].elapsed_time(ev[1]) >= 0
