"""Pins of the oracle's 2-bit page format with promoted 4-bit key channels (the Kitty row,
"KVキャッシュ管理の教科書" 第22章).

Every pin checks the oracle against something other than itself: pages built on the quantisation
grid (codes, scales and minimums chosen first, so the exact answer is known), hand-worked bytes of
the record, the promotion rule on pages where the mean-magnitude order is known by construction,
round-half-even ties, the error bound of min/max quantisation on random pages, and the already
pinned float attention oracle on caches holding exactly representable values.  Each pin takes
the oracle module as an argument so that the planted-mistake test can run the same pins against
copies of the module with one mistake written in.
"""
import os
import types

import numpy as np
import pytest

import oracle
from oracle import kitty

T, D = 128, 128


def bf16_bits(x):
    """bf16 storage (uint16) of float32 values that are exactly representable in bf16."""
    x = np.asarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    assert np.all((u & 0xFFFF) == 0), "value not exact in bf16"
    return (u >> 16).astype(np.uint16)


def grid_page(rng, promoted_ids):
    """A page whose K and V lie on the quantisation grid the format must find: K channel x holds
    m_x + c * s_x with c spanning 0..L_x (L = 15 on the promoted channels, 3 elsewhere), V token
    t holds m_t + c * s_t with c spanning 0..3.  Promoted channels get minimum 8 so that their
    mean magnitude is the largest; the others stay within [-2, 2)."""
    pset = set(int(i) for i in promoted_ids)
    kc = np.zeros((T, D), np.int64)
    ks = np.zeros(D, np.float32)
    km = np.zeros(D, np.float32)
    for x in range(D):
        L = 15 if x in pset else 3
        c = rng.integers(0, L + 1, T)
        i0, i1 = rng.choice(T, 2, replace=False)
        c[i0], c[i1] = 0, L                                    # both ends of the grid present
        kc[:, x] = c
        ks[x] = 0.125 if x in pset else 2.0 ** -int(rng.integers(1, 4))
        km[x] = 8.0 if x in pset else -float(rng.integers(0, 4)) * 0.5
    vc = rng.integers(0, 4, (T, D))
    vc[:, 0], vc[:, 1] = 0, 3
    vc = np.array([rng.permutation(r) for r in vc])
    vs = (2.0 ** -rng.integers(0, 3, T)).astype(np.float32)
    vm = (rng.integers(-4, 4, T) * 0.25).astype(np.float32)
    k = (kc * ks[None, :] + km[None, :]).astype(np.float32)
    v = (vc * vs[:, None] + vm[:, None]).astype(np.float32)
    return k, v, dict(k_codes=kc, ks=ks, km=km, v_codes=vc, vs=vs, vm=vm)


# ---- pins (each takes the oracle module under test) -------------------------------------------

def pin_grid_page_round_trips(K):
    rng = np.random.default_rng(11)
    for P in (16, 32):
        pid = np.sort(rng.choice(D, P, replace=False))
        k, v, want = grid_page(rng, pid)
        f = K.quantize_page(k, v, P)
        g = K.unpack_record(K.pack_record(f), P)
        assert np.array_equal(g["pid"], pid)
        for name in ("k_codes", "v_codes", "ks", "km", "vs", "vm"):
            assert np.array_equal(g[name], want[name]), name
        kd, vd = K.dequantize(g)
        assert np.array_equal(kd, k.astype(np.float64))
        assert np.array_equal(vd, v.astype(np.float64))


def pin_hand_worked_bytes(K):
    # Promoted set (P = 16): channels 100..115, the only ones with large magnitude.  Channel 100
    # runs 100..115 (scale 1) with code 13 = 1 + 4 * 3 at token 2; the others are constant 50
    # (scale 0).  Channel 5 (2 bits) runs 0..3 with code 2 at token 1.  V token 0, channels 0..3
    # hold codes 1, 2, 3, 0; V token 1, channels 0..3 codes 3, 0, 0, 3; V token 70 (second half
    # page), channel 2 code 3 and channel 3 code 1 (scale 1, minimum 0).  Every other value is 0.
    k = np.zeros((T, D), np.float32)
    v = np.zeros((T, D), np.float32)
    k[:, 100:116] = 50.0
    k[:, 100] = 100.0
    k[2, 100], k[4, 100] = 113.0, 115.0
    k[1, 5], k[3, 5] = 2.0, 3.0
    v[0, :4] = [1.0, 2.0, 3.0, 0.0]
    v[1, :4] = [3.0, 0.0, 0.0, 3.0]
    v[70, :4] = [0.0, 0.0, 3.0, 1.0]
    f = K.quantize_page(k, v, 16)
    rec = K.pack_record(f)
    assert len(rec) == 10784
    assert list(rec[2048:2064]) == list(range(100, 116)) and np.all(rec[2064:2080] == 0)
    assert rec[2080 + 32 * 1 + 1] == 0x08        # token 1, channel 5 (byte 1, bits 2-3): code 2
    assert rec[2080 + 32 * 2 + 25] == 0x01       # token 2, channel 100 (byte 25, bits 0-1): low 1
    assert rec[6176 + 4 * 2 + 0] == 0x03         # token 2, promoted slot 0 (byte 0, bits 0-1): high 3
    assert rec[2080 + 32 * 3 + 1] == 0x0C        # token 3, channel 5: code 3
    assert rec[2080 + 32 * 4 + 25] == 0x03 and rec[6176 + 4 * 4] == 0x03   # token 4, channel 100: 15
    assert np.count_nonzero(rec[2080:2080 + 4096]) == 4 and np.count_nonzero(rec[6176:6176 + 512]) == 2
    vc_off = 6176 + 32 * 16
    # V codes: half page, then channel (16 bytes each), then token (4 per byte, low bits first)
    assert rec[vc_off + 0] == 0x0D               # channel 0: token 0 code 1, token 1 code 3 (bits 2-3)
    assert rec[vc_off + 16] == 0x02              # channel 1: token 0 code 2
    assert rec[vc_off + 32] == 0x03              # channel 2: token 0 code 3
    assert rec[vc_off + 48] == 0x0C              # channel 3: token 1 code 3
    assert rec[vc_off + 2048 + 32 + 1] == 0x30   # half 1, channel 2: token 70 = 64 + 6 -> byte 1, bits 4-5
    assert rec[vc_off + 2048 + 48 + 1] == 0x10   # half 1, channel 3: token 70 code 1
    assert np.count_nonzero(rec[vc_off:vc_off + 4096]) == 6
    f32 = lambda off: np.frombuffer(rec[off:off + 4].tobytes(), "<f4")[0]
    assert f32(1024) == 1.0                      # V scale of token 0
    assert f32(4 * 5) == 1.0 and f32(4 * 100) == 1.0 and f32(4 * 101) == 0.0   # K scales
    assert f32(512 + 4 * 100) == 100.0 and f32(512 + 4 * 101) == 50.0          # K minimums


def pin_promotion_by_mean_not_max(K):
    rng = np.random.default_rng(3)
    k = rng.uniform(-0.5, 0.5, (T, D)).astype(np.float32)
    heavy = np.arange(2, 2 * 16 + 2, 2)            # 16 channels with mean magnitude about 4
    k[:, heavy] += 4.0
    k[7, 1] = 300.0                                # one spike: largest max, mean about 2.6
    v = np.zeros((T, D), np.float32)
    f = K.quantize_page(k, v, 16)
    assert np.array_equal(f["pid"], heavy)


def pin_ties_go_to_lower_channels(K):
    k = np.tile(np.array([[1.0], [-1.0]], np.float32), (T // 2, D))   # +-1 rows: equal magnitudes
    assert np.all(np.abs(k) == 1.0)
    for P in (16, 32):
        f = K.quantize_page(k, np.zeros((T, D), np.float32), P)
        assert np.array_equal(f["pid"], np.arange(P))


def pin_round_half_even_and_constant_groups(K):
    v = np.zeros((T, D), np.float32)
    v[0, :5] = [0.0, 3.0, 0.5, 1.5, 2.5]          # scale 1: halfway points -> 0, 2, 2
    v[1, :] = 7.0                                  # constant token: scale 0, every code 0
    k = np.zeros((T, D), np.float32)
    f = K.quantize_page(k, v, 16)
    assert list(f["v_codes"][0, :5]) == [0, 3, 0, 2, 2]
    assert f["vs"][1] == 0 and np.all(f["v_codes"][1] == 0) and f["vm"][1] == 7.0
    _, vd = K.dequantize(f)
    assert np.all(vd[1] == 7.0)


def pin_error_bound_on_random_pages(K):
    rng = np.random.default_rng(5)
    for P in (16, 32):
        k = rng.standard_normal((T, D)).astype(np.float32) * rng.uniform(0.1, 3.0, D).astype(np.float32)
        v = rng.standard_normal((T, D)).astype(np.float32)
        f = K.unpack_record(K.pack_record(K.quantize_page(k, v, P)), P)
        kd, vd = K.dequantize(f)
        ks = f["ks"].astype(np.float64)
        vs = f["vs"].astype(np.float64)
        assert np.all(np.abs(kd - k) <= ks[None, :] * (0.5 + 1e-5))
        assert np.all(np.abs(vd - v) <= vs[:, None] * (0.5 + 1e-5))
        # promoted channels carry 16 levels: their step is a fifth of a 2-bit step on the same range
        rng_k = k.max(0).astype(np.float64) - k.min(0)
        levels = np.where(np.isin(np.arange(D), f["pid"]), 15, 3)
        assert np.allclose(ks, rng_k / levels, rtol=1e-6)
        # the promoted set is the top P of the float64 mean magnitudes (gaps here are large)
        top = np.sort(np.argsort(-np.abs(k.astype(np.float64)).mean(0), kind="stable")[:P])
        assert np.array_equal(f["pid"], top)


def _kitty_case(rng, K, P, lens, num_q_heads=4, num_kv_heads=2, grid=True):
    """Pages and residual pages of a decode batch, and the same tokens as one bf16 cache with
    128-token blocks (for the plain oracle).  Returns (kitty args, plain args)."""
    S = len(lens)
    n = np.array(lens, np.int64)
    nfull = n // T
    npages = int(nfull.sum())
    nres = int((n % T > 0).sum())
    maxp = int(((n + T - 1) // T).max())
    pool_pages = npages + 3
    page_ids = rng.permutation(pool_pages)[:npages]
    res_ids = rng.permutation(nres + 2)[:nres]
    pages = rng.integers(0, 256, (pool_pages, num_kv_heads, K.record_bytes(P)), dtype=np.uint8)
    res_k = rng.integers(0, 1 << 16, (nres + 2, num_kv_heads, T, D), dtype=np.uint16)
    res_v = rng.integers(0, 1 << 16, (nres + 2, num_kv_heads, T, D), dtype=np.uint16)
    nb = npages + nres
    ck = np.zeros((nb + 1, num_kv_heads, T, D), np.uint16)
    cv = np.zeros((nb + 1, num_kv_heads, T, D), np.uint16)
    bt = np.full((S, maxp), -7, np.int32)
    bt_plain = np.full((S, maxp), -7, np.int32)
    pi = ri = blk = 0
    for i in range(S):
        for p in range(int(nfull[i])):
            for h in range(num_kv_heads):
                if grid:
                    k, v, _ = grid_page(rng, np.sort(rng.choice(D, P, replace=False)))
                else:
                    k = rng.standard_normal((T, D)).astype(np.float32)
                    v = rng.standard_normal((T, D)).astype(np.float32)
                f = K.quantize_page(k, v, P)
                pages[page_ids[pi], h] = K.pack_record(f)
                if grid:
                    kd, vd = K.dequantize(f)
                    ck[blk, h] = bf16_bits(kd.astype(np.float32))
                    cv[blk, h] = bf16_bits(vd.astype(np.float32))
            bt[i, p], bt_plain[i, p] = page_ids[pi], blk
            pi += 1
            blk += 1
        if n[i] % T:
            r = res_ids[ri]
            tail = int(n[i] % T)
            kk = bf16_bits(np.round(rng.standard_normal((num_kv_heads, T, D)) * 8) / 8)
            vv = bf16_bits(np.round(rng.standard_normal((num_kv_heads, T, D)) * 8) / 8)
            res_k[r, :, :tail], res_v[r, :, :tail] = kk[:, :tail], vv[:, :tail]
            ck[blk], cv[blk] = res_k[r], res_v[r]
            bt[i, nfull[i]], bt_plain[i, nfull[i]] = r, blk
            ri += 1
            blk += 1
    ctx = (n - 1).astype(np.int32)
    ql = np.ones(S, np.int32)
    q = bf16_bits(np.round(rng.standard_normal((S, num_q_heads, D)) * 16) / 16)
    scale = 1.0 / np.sqrt(D)
    kit = (q, pages, res_k, res_v, "bf16", bt, ctx, ql, num_q_heads, num_kv_heads, P, scale)
    plain = (q, ck, cv, "bf16", bt_plain, ctx, ql, num_q_heads, num_kv_heads, D, T, scale)
    return kit, plain


def pin_attention_equals_plain_oracle_on_exact_values(K):
    rng = np.random.default_rng(7)
    for P, lens in ((16, [1, 127, 128, 129, 300]), (32, [256, 385, 5, 640])):
        kit, plain = _kitty_case(rng, K, P, lens)
        got = K.paged_attention(*kit)
        want = oracle.paged_attention(*plain)
        assert np.array_equal(got, want)


def pin_page_permutation_invariance(K):
    rng = np.random.default_rng(9)
    kit, _ = _kitty_case(rng, K, 32, [200, 700, 129], grid=False)
    q, pages, res_k, res_v, dt, bt, ctx, ql, hq, hkv, P, scale = kit
    a = K.paged_attention(*kit)
    perm = rng.permutation(pages.shape[0])
    inv = np.argsort(perm)
    pages2 = pages[perm]
    bt2 = bt.copy()
    n = ctx.astype(np.int64) + 1
    for i in range(len(ctx)):
        for p in range(int(n[i] // T)):
            bt2[i, p] = inv[bt[i, p]]
    b = K.paged_attention(q, pages2, res_k, res_v, dt, bt2, ctx, ql, hq, hkv, P, scale)
    assert np.array_equal(a, b)


PINS = [pin_grid_page_round_trips, pin_hand_worked_bytes, pin_promotion_by_mean_not_max,
        pin_ties_go_to_lower_channels, pin_round_half_even_and_constant_groups,
        pin_error_bound_on_random_pages, pin_attention_equals_plain_oracle_on_exact_values,
        pin_page_permutation_invariance]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin(kitty)


def test_record_sizes_and_bits_per_element():
    assert kitty.record_bytes(16) == 10784 and kitty.record_bytes(32) == 11296
    # 2-bit codes for every K and V element, 2 more bits on 25 % of the key channels, float32
    # scales and minimums: 2.76 bits per cached element (5.8x fewer bytes than 16-bit elements)
    bits = kitty.record_bytes(32) * 8 / (2 * T * D)
    assert abs(bits - 2.7578125) < 1e-12


def test_quantize_pages_writes_each_pair_and_every_head():
    rng = np.random.default_rng(13)
    res_k = rng.integers(0, 1 << 16, (3, 2, T, D), dtype=np.uint16) & 0x3FFF | 0x3C00
    res_v = rng.integers(0, 1 << 16, (3, 2, T, D), dtype=np.uint16) & 0x3FFF | 0x3C00
    pages = np.zeros((4, 2, kitty.record_bytes(16)), np.uint8)
    out = kitty.quantize_pages(res_k, res_v, [[2, 0], [0, 3]], pages, 16, "bf16")
    assert np.all(out[1] == 0) and np.all(out[2] == 0)
    for s, t in ((2, 0), (0, 3)):
        for h in range(2):
            f = kitty.quantize_page(oracle.widen_f32(res_k[s, h], "bf16"),
                                    oracle.widen_f32(res_v[s, h], "bf16"), 16)
            assert np.array_equal(out[t, h], kitty.pack_record(f))


# ---- planted mistakes: each must make at least one pin fail -----------------------------------

PLANTED = {
    "high bits weighted 2": ("k_codes[:, pid] += 4 * hi", "k_codes[:, pid] += 2 * hi"),
    "4 levels for 2 bits": ("levels = np.full(HEAD_DIM, 3,", "levels = np.full(HEAD_DIM, 4,"),
    "promotion by max": ("mag = mag + np.abs(k[t])", "mag = np.maximum(mag, np.abs(k[t]))"),
    "ties to higher channels": ('order = np.argsort(-mag, kind="stable")',
                                'order = HEAD_DIM - 1 - np.argsort(-mag[::-1], kind="stable")'),
    "codes packed high bits first": ("c[..., 0] | (c[..., 1] << 2) | (c[..., 2] << 4) | (c[..., 3] << 6)",
                                     "c[..., 3] | (c[..., 2] << 2) | (c[..., 1] << 4) | (c[..., 0] << 6)"),
    "V per channel": ("vmin = v.min(axis=1)\n    vmax = v.max(axis=1)",
                      "vmin = v.min(axis=0)\n    vmax = v.max(axis=0)"),
    "V codes token-major": ("halves = [_pack2(v_codes[64 * h:64 * h + 64].T) for h in range(2)]",
                            "halves = [_pack2(v_codes[64 * h:64 * h + 64]) for h in range(2)]"),
    "V halves swapped": ("np.concatenate([x.reshape(-1) for x in halves])",
                         "np.concatenate([x.reshape(-1) for x in halves[::-1]])"),
    "round half up": ("r = np.rint((x - lo) / s)", "r = np.floor((x - lo) / s + np.float32(0.5))"),
    "last full page read as residual": ("nfull = n // PAGE_TOKENS",
                                        "nfull = (n - 1) // PAGE_TOKENS"),
    "residual page ignored": ("        if n[i] % PAGE_TOKENS:\n            r = int",
                              "        if False:\n            r = int"),
}


@pytest.mark.parametrize("name", sorted(PLANTED))
def test_pins_catch_planted_mistake(name):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "kitty.py")).read()
    a, b = PLANTED[name]
    assert src.count(a) == 1, name
    mod = types.ModuleType("kitty_planted")
    exec(compile(src.replace(a, b), "kitty_planted", "exec"), mod.__dict__)
    caught = []
    for pin in PINS:
        try:
            pin(mod)
        except (AssertionError, ValueError, IndexError):
            caught.append(pin.__name__)
    assert caught, f"planted mistake {name!r} passed every pin"
