"""Oracle of the 2-bit paged KV cache with promoted 4-bit key channels (the Kitty row).

TEST INFRASTRUCTURE ONLY, like the rest of this package: the CUDA library never imports it.

What the pages state ("KVキャッシュ管理の教科書", 第3章 and 第22章, on Kitty):

* the KV cache is quantised to 2 bits per element;
* for the keys, the channels whose mean magnitude along the token direction is among the top
  12.5 % to 25 % are promoted to 4 bits; the rest stay at 2 bits;
* storage is split into a dense tensor holding the low 2 bits of every channel and a sparse
  tensor holding only the high 2 bits of the promoted channels, so that reading stays uniform;
* one quantisation group is 128 tokens, which is one page of the paged cache; the heavy
  quantisation work runs once per 128 decode steps.

Readings taken where the pages leave a step open (each one is also stated in the library's
header, which defines the same record):

* quantisation is asymmetric min/max (the KIVI convention the chapter contrasts Kitty with): K per
  channel over the page's 128 tokens, V per token over the head's d channels; the code of x is
  round-half-even((x - min) / s) clamped to [0, L], s = (max - min) / L, L = 3 (2 bits) or 15
  (promoted 4-bit key channels); a constant group (s = 0) codes every element as 0;
* the decisions that produce integers (codes, the promoted set) are taken in float32, the
  precision of the inputs' widening: differences, divisions and the magnitude sums are float32
  operations rounded to nearest; the magnitude sum runs over the tokens in order;
* the promoted set is the P channels with the largest magnitude sum, ties going to the lower
  channel index; P is 16 (12.5 %) or 32 (25 %) of d = 128;
* tokens of a sequence's last, partly filled page stay unquantised in a residual page of the
  query's dtype until the page fills; a sequence of n tokens has floor(n / 128) quantised pages.

Record of one (page, KV head), little-endian, byte offsets (d = 128, P promoted channels):

    [0, 512)          K scale s_x, float32 per channel x
    [512, 1024)       K minimum m_x, float32 per channel
    [1024, 1536)      V scale, float32 per token
    [1536, 2048)      V minimum, float32 per token
    [2048, 2080)      promoted channel ids, uint8, ascending in slots 0..P-1, later slots 0
    [2080, 6176)      K low bits: token t, channel x -> byte 32 t + x / 4, bits 2 (x % 4)
    [6176, 6176+32P)  K high bits of promoted slot k: byte (P / 4) t + k / 4, bits 2 (k % 4)
    then 4096 bytes   V codes: token t, channel x -> byte 2048 (t / 64) + 16 x + (t % 64) / 4,
                      bits 2 (t % 4) (per half page, channel-major)

A cached element's value is code x scale + minimum (a promoted key code is low + 4 x high).

The byte layout is this implementation's own (the chapter fixes the dense/sparse split and the
bit widths, not the order of the bytes).  K codes are token-major and V codes channel-major within
each half page of 64 tokens, so that a 32-bit word of K codes holds 16 channels of one key and a
word of V codes holds 16 tokens of one channel.
"""
from __future__ import annotations

import numpy as np

PAGE_TOKENS = 128
HEAD_DIM = 128
_OFF_KS, _OFF_KM, _OFF_VS, _OFF_VM, _OFF_PID, _OFF_KLO = 0, 512, 1024, 1536, 2048, 2080


def record_bytes(promoted: int) -> int:
    """Bytes of one (page, KV head) record."""
    return 10272 + 32 * int(promoted)


def _offsets(promoted):
    khi = _OFF_KLO + 32 * PAGE_TOKENS
    vc = khi + (promoted // 4) * PAGE_TOKENS
    return khi, vc


def _codes(x, lo, s, levels):
    """round-half-even((x - lo) / s) clamped to [0, levels], in float32; 0 where s == 0."""
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.rint((x - lo) / s)
    r = np.where(s == np.float32(0), np.float32(0), r)
    return np.clip(r, 0, levels).astype(np.int64)


def quantize_page(k, v, promoted):
    """Quantises one page of one KV head.

    ``k``, ``v``: float32 [128 tokens, 128 channels] (the residual page's values, widened
    exactly).  Returns a dict of the record's fields: ``k_codes`` [128, 128] (0..15 on promoted
    channels, 0..3 elsewhere), ``pid`` (the P promoted channel ids, ascending), ``ks``, ``km``
    (float32 per channel), ``v_codes`` [128, 128] (0..3), ``vs``, ``vm`` (float32 per token).
    """
    k = np.asarray(k, dtype=np.float32)
    v = np.asarray(v, dtype=np.float32)
    assert k.shape == (PAGE_TOKENS, HEAD_DIM) and v.shape == (PAGE_TOKENS, HEAD_DIM)
    P = int(promoted)
    # per-channel magnitude along the token direction: float32 sum of |k| in token order
    mag = np.zeros(HEAD_DIM, dtype=np.float32)
    for t in range(PAGE_TOKENS):
        mag = mag + np.abs(k[t])
    # the P largest, ties to the lower channel index (a stable sort on -mag keeps index order)
    order = np.argsort(-mag, kind="stable")
    pid = np.sort(order[:P])
    levels = np.full(HEAD_DIM, 3, dtype=np.float32)
    levels[pid] = 15
    kmin = k.min(axis=0)
    kmax = k.max(axis=0)
    ks = (kmax - kmin) / levels
    k_codes = _codes(k, kmin[None, :], ks[None, :], levels[None, :])
    vmin = v.min(axis=1)
    vmax = v.max(axis=1)
    vs = (vmax - vmin) / np.float32(3)
    v_codes = _codes(v, vmin[:, None], vs[:, None], 3)
    return dict(k_codes=k_codes, pid=pid.astype(np.int64), ks=ks.astype(np.float32),
                km=kmin.astype(np.float32), v_codes=v_codes, vs=vs.astype(np.float32),
                vm=vmin.astype(np.float32), promoted=P)


def _pack2(codes):
    """[rows, n] codes 0..3 -> [rows, n / 4] bytes, code j at bits 2 (j % 4) of byte j / 4."""
    c = np.asarray(codes, dtype=np.int64).reshape(codes.shape[0], -1, 4)
    b = c[..., 0] | (c[..., 1] << 2) | (c[..., 2] << 4) | (c[..., 3] << 6)
    return b.astype(np.uint8)


def _unpack2(b, n):
    b = np.asarray(b, dtype=np.int64)
    out = np.stack([(b >> (2 * i)) & 3 for i in range(4)], axis=-1)
    return out.reshape(b.shape[0], n)


def _pack_v(v_codes):
    """[128 tokens, 128 channels] V codes -> 4096 bytes: for each half page h (tokens 64 h ..
    64 h + 63), channel x's 64 codes in 16 bytes at 2048 h + 16 x, token t at bits 2 (t % 4) of
    byte (t % 64) / 4."""
    halves = [_pack2(v_codes[64 * h:64 * h + 64].T) for h in range(2)]   # [channel, 16 bytes]
    return np.concatenate([x.reshape(-1) for x in halves])


def _unpack_v(b):
    b = np.asarray(b, dtype=np.uint8).reshape(2, HEAD_DIM, 16)
    return np.concatenate([_unpack2(b[h], 64).T for h in range(2)], axis=0)


def pack_record(f) -> np.ndarray:
    """The record's bytes (uint8 [record_bytes]) from ``quantize_page``'s fields."""
    P = f["promoted"]
    khi_off, vc_off = _offsets(P)
    rec = np.zeros(record_bytes(P), dtype=np.uint8)
    rec[_OFF_KS:_OFF_KM] = f["ks"].astype("<f4").view(np.uint8)
    rec[_OFF_KM:_OFF_VS] = f["km"].astype("<f4").view(np.uint8)
    rec[_OFF_VS:_OFF_VM] = f["vs"].astype("<f4").view(np.uint8)
    rec[_OFF_VM:_OFF_PID] = f["vm"].astype("<f4").view(np.uint8)
    rec[_OFF_PID:_OFF_PID + P] = f["pid"].astype(np.uint8)
    kc = f["k_codes"]
    rec[_OFF_KLO:khi_off] = _pack2(kc & 3).reshape(-1)
    rec[khi_off:vc_off] = _pack2(kc[:, f["pid"]] >> 2).reshape(-1)
    rec[vc_off:vc_off + 32 * PAGE_TOKENS] = _pack_v(f["v_codes"])
    return rec


def unpack_record(rec, promoted):
    """Inverse of ``pack_record``."""
    rec = np.asarray(rec, dtype=np.uint8).reshape(-1)
    P = int(promoted)
    khi_off, vc_off = _offsets(P)
    ks = rec[_OFF_KS:_OFF_KM].view("<f4").astype(np.float32)
    km = rec[_OFF_KM:_OFF_VS].view("<f4").astype(np.float32)
    vs = rec[_OFF_VS:_OFF_VM].view("<f4").astype(np.float32)
    vm = rec[_OFF_VM:_OFF_PID].view("<f4").astype(np.float32)
    pid = rec[_OFF_PID:_OFF_PID + P].astype(np.int64)
    k_codes = _unpack2(rec[_OFF_KLO:khi_off].reshape(PAGE_TOKENS, 32), HEAD_DIM)
    hi = _unpack2(rec[khi_off:vc_off].reshape(PAGE_TOKENS, P // 4), P)
    k_codes[:, pid] += 4 * hi
    v_codes = _unpack_v(rec[vc_off:vc_off + 32 * PAGE_TOKENS])
    return dict(k_codes=k_codes, pid=pid, ks=ks, km=km, v_codes=v_codes, vs=vs, vm=vm,
                promoted=P)


def dequantize(f):
    """float64 K and V [128 tokens, 128 channels] of one record: code x scale + minimum."""
    k = f["k_codes"].astype(np.float64) * f["ks"].astype(np.float64)[None, :] \
        + f["km"].astype(np.float64)[None, :]
    v = f["v_codes"].astype(np.float64) * f["vs"].astype(np.float64)[:, None] \
        + f["vm"].astype(np.float64)[:, None]
    return k, v


def quantize_pages(res_k, res_v, pairs, pages, promoted, dtype):
    """Returns a copy of the page pool with residual page s quantised into page t for every
    (s, t) in ``pairs``, every KV head.  ``res_k``/``res_v``: generator-module storage
    [num_res, Hkv, 128, 128] of ``dtype``; ``pages``: uint8 [num_pages, Hkv, record_bytes]."""
    from oracle import widen_f32
    out = np.array(pages, dtype=np.uint8, copy=True)
    for s, t in np.asarray(pairs, dtype=np.int64).reshape(-1, 2):
        for h in range(out.shape[1]):
            f = quantize_page(widen_f32(res_k[s, h], dtype), widen_f32(res_v[s, h], dtype), promoted)
            out[t, h] = pack_record(f)
    return out


def paged_attention(q, pages, res_k, res_v, dtype, block_tables, ctx_lens, q_lens, num_q_heads,
                    num_kv_heads, promoted, scale, rows=None, threads=1):
    """Float64 decode attention over Kitty pages.

    Sequence i has n_i = ctx_lens[i] + q_lens[i] tokens (q_lens[i] = 1); logical page p <
    floor(n_i / 128) is the quantised record ``pages[block_tables[i][p]]``, and, when n_i is not a
    multiple of 128, logical page floor(n_i / 128) is the residual page
    ``res_k/res_v[block_tables[i][floor(n_i / 128)]]`` of ``dtype``.  Every quantised page used is
    dequantised to float64 and, with the residual pages' values, laid out as one float64 cache
    with blocks of 128 tokens; attention is then the plain oracle's ``paged_attention`` on it.
    """
    import oracle
    pages = np.asarray(pages, dtype=np.uint8)
    bt = np.asarray(block_tables, dtype=np.int64)
    ctx = np.asarray(ctx_lens, dtype=np.int64)
    ql = np.asarray(q_lens, dtype=np.int64)
    S = len(ctx)
    Hkv = num_kv_heads
    n = ctx + ql
    nfull = n // PAGE_TOKENS
    blocks = []
    bt2 = np.zeros((S, int(bt.shape[1])), dtype=np.int32)
    for i in range(S):
        for p in range(int(nfull[i])):
            kv = [dequantize(unpack_record(pages[bt[i, p], h], promoted)) for h in range(Hkv)]
            bt2[i, p] = len(blocks)
            blocks.append((np.stack([a for a, _ in kv]), np.stack([b for _, b in kv])))
        if n[i] % PAGE_TOKENS:
            r = int(bt[i, nfull[i]])
            with np.errstate(invalid="ignore"):      # unread slots may hold NaN patterns
                k = oracle.widen_f32(res_k[r], dtype).astype(np.float64)
                v = oracle.widen_f32(res_v[r], dtype).astype(np.float64)
            bt2[i, nfull[i]] = len(blocks)
            blocks.append((k, v))
    if not blocks:
        raise ValueError("no tokens")
    kc = np.stack([a for a, _ in blocks])
    vc = np.stack([b for _, b in blocks])
    return oracle.paged_attention(q, kc, vc, dtype, bt2, ctx.astype(np.int32), ql.astype(np.int32),
                                  num_q_heads, Hkv, HEAD_DIM, PAGE_TOKENS, scale, rows=rows,
                                  threads=threads, kv_dtype="f64")
