"""Pins of the oracle's 8-bit cache path (FP8 E4M3 codes with one scale for K and one for V).

The format's definition -- 1 sign bit, 4 exponent bits with bias 7, 3 fraction bits, subnormals at
exponent 0, no infinities, S.1111.111 = NaN -- is checked against an independent implementation
(PyTorch's float8_e4m3fn) and against values worked out by hand; the encoder against the same
library's round-to-nearest-even conversion, hand-made ties and the saturation rule; the attention
path against the already pinned float32 path on exactly representable values.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_generalized_gb300 import workloads as W


def test_decode_matches_an_independent_implementation_on_all_codes():
    c = np.arange(256, dtype=np.uint8)
    mine = oracle.e4m3_decode(c)
    ref = torch.from_numpy(c).view(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(np.isnan(mine), np.isnan(ref))
    assert np.array_equal(mine[~np.isnan(mine)], ref[~np.isnan(ref)])
    fin = ~np.isnan(mine)
    assert np.array_equal(np.signbit(mine[fin]), np.signbit(ref[fin]))


@pytest.mark.parametrize("code,value", [
    (0x00, 0.0), (0x01, 2.0 ** -9), (0x07, 7 * 2.0 ** -9), (0x08, 2.0 ** -6), (0x30, 0.5),
    (0x38, 1.0), (0x39, 1.125), (0x40, 2.0), (0x77, 240.0), (0x7E, 448.0), (0xB8, -1.0),
    (0xFE, -448.0)])
def test_decode_hand_values(code, value):
    assert oracle.e4m3_decode(np.array([code], np.uint8))[0] == value


def test_decode_nan_and_negative_zero():
    v = oracle.e4m3_decode(np.array([0x7F, 0xFF, 0x80], np.uint8))
    assert np.isnan(v[0]) and np.isnan(v[1])
    assert v[2] == 0.0 and np.signbit(v[2])


def test_encode_round_trips_every_finite_code():
    c = np.array([x for x in range(256) if x not in (0x7F, 0xFF)], dtype=np.uint8)
    assert np.array_equal(oracle.e4m3_encode(oracle.e4m3_decode(c), 1.0), c)


def test_encode_matches_an_independent_round_to_nearest_even():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.normal(0, 1, 20000), rng.normal(0, 60, 20000),
                        rng.uniform(-2 ** -6, 2 ** -6, 20000)]).astype(np.float32)
    x = x[np.abs(x) < 440]
    mine = oracle.e4m3_encode(x, 1.0)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(mine, ref)


def test_encode_ties_go_to_the_even_code():
    # midpoints between consecutive representable values
    x = np.array([1.0625, 1.1875, 2 ** -10, 3 * 2 ** -10, 240.0 + 8.0, -1.0625], np.float32)
    got = oracle.e4m3_encode(x, 1.0)
    # 1.0625 -> 1.0 (0x38, even); 1.1875 -> 1.25 (0x3A); 2^-10 -> 0 (0x00); 3*2^-10 -> 2*2^-9
    # (0x02); 248 -> 256 (0x78, even over 240 = 0x77); -1.0625 -> -1.0
    assert got.tolist() == [0x38, 0x3A, 0x00, 0x02, 0x78, 0xB8]


def test_encode_saturates_at_448_and_keeps_the_sign():
    x = np.array([448.0, 449.0, 464.0, 470.0, 1e6, -1e6, -500.0, -1e-12], np.float32)
    assert oracle.e4m3_encode(x, 1.0).tolist() == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE, 0x80]


def test_encode_scales_in_float32_before_rounding():
    x = np.array([3.0, -0.7, 100.0], np.float32)
    inv = np.float32(1.0) / np.float32(3.0)
    y = (x * inv).astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode(x, inv), oracle.e4m3_encode(y, 1.0))


@pytest.mark.parametrize("ks,vs", [(1.0, 1.0), (0.25, 8.0), (2.0 ** -7, 2.0 ** 5)])
def test_attention_on_codes_equals_the_float32_path_on_their_values(ks, vs):
    """With power-of-two scales, code value x scale is exact in float32, so the 8-bit path must give
    bit-for-bit the pinned float32 path's result on the decoded caches."""
    b = W.make_attn_batch("fp8", [37, 50, 130], [5, 1, 17], 8, 2, 64, 16, "f32", seed=11, poison=False)
    rng = np.random.default_rng(5)
    kc = rng.integers(0, 256, b.k_cache.shape).astype(np.uint8)
    vc = rng.integers(0, 256, b.v_cache.shape).astype(np.uint8)
    kc[(kc & 0x7F) == 0x7F] = 0x3C                       # no NaN codes
    vc[(vc & 0x7F) == 0x7F] = 0x3C
    got = oracle.paged_attention_batch(b, kv=(kc, vc, ks, vs))
    kf = (oracle.e4m3_decode(kc) * ks).astype(np.float32)
    vf = (oracle.e4m3_decode(vc) * vs).astype(np.float32)
    assert np.array_equal(kf.astype(np.float64), oracle.e4m3_decode(kc) * ks)
    ref = oracle.paged_attention(b.q, kf, vf, "f32", b.block_tables, b.ctx_lens, b.q_lens,
                                 b.num_q_heads, b.num_kv_heads, b.head_dim, b.block_size, b.scale)
    assert np.array_equal(got, ref)


def test_append_encodes_then_scatters():
    b = W.make_attn_batch("fp8a", [20, 3], [5, 2], 4, 2, 64, 16, "bf16", seed=9, poison=False)
    k0 = np.zeros(b.k_cache.shape, np.uint8)
    v0 = np.zeros(b.v_cache.shape, np.uint8)
    ks, vs = 0.5, 3.0
    kc, vc = oracle.kv_append_e4m3(b.k_new, b.v_new, b.slot_mapping, k0, v0, b.block_size, ks, vs, "bf16")
    B = b.block_size
    for t, slot in enumerate(b.slot_mapping):
        blk, off = slot // B, slot % B
        for h in range(b.num_kv_heads):
            x = oracle.widen_f32(b.k_new[t, h], "bf16")
            want = torch.from_numpy(x * np.float32(1 / np.float32(ks))).to(torch.float8_e4m3fn)
            assert np.array_equal(kc[blk, h, off], want.view(torch.uint8).numpy())
    untouched = np.ones(kc.shape[:3], bool)
    for slot in b.slot_mapping:
        untouched[slot // B, :, slot % B] = False
    assert (kc[untouched] == 0).all() and (vc[untouched] == 0).all()


# Planted mistakes in the C oracle's 8-bit path: each must break the equality with the pinned
# float32 path above.
FP8_MUTATIONS = {
    "bias_8": ("v = ldexp((double)(m + 8), e - 10);", "v = ldexp((double)(m + 8), e - 11);"),
    "subnormal_step": ("v = ldexp((double)m, -9);", "v = ldexp((double)m, -10);"),
    "v_scale_dropped": ("o[x] += w * (element(v_cache, kv_dtype, vbase + x) * v_scale);",
                        "o[x] += w * (element(v_cache, kv_dtype, vbase + x) * 1.0);"),
    "k_scale_dropped": ("(element(k_cache, kv_dtype, kbase + x) * k_scale);",
                        "(element(k_cache, kv_dtype, kbase + x) * 1.0);"),
}


@pytest.mark.parametrize("name", sorted(FP8_MUTATIONS))
def test_fp8_pins_catch_planted_mistake(name, monkeypatch):
    import ctypes
    import os
    import subprocess
    import tempfile

    src = open(os.path.join(os.path.dirname(oracle.__file__), "attention.c")).read()
    old, new = FP8_MUTATIONS[name]
    assert src.count(old) == 1, name
    with tempfile.TemporaryDirectory() as tmp:
        c, so = os.path.join(tmp, "m.c"), os.path.join(tmp, "libm.so")
        open(c, "w").write(src.replace(old, new))
        subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", c, "-o", so, "-lm"],
                       check=True, capture_output=True)
        monkeypatch.setattr(oracle, "_lib", oracle.declare(ctypes.CDLL(so)))
        caught = False
        for ks, vs in [(0.25, 8.0), (2.0 ** -7, 2.0 ** 5)]:
            try:
                test_attention_on_codes_equals_the_float32_path_on_their_values(ks, vs)
            except AssertionError:
                caught = True
                break
        assert caught, f"planted mistake {name!r} passed the 8-bit pins"
