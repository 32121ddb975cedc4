"""Oracle for generalized paged attention, cache append and block copy.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's
CPU-baseline leg (``bench.py``) may import or run anything in this package; the product path
(``paged_kv_cache_generalized_gb300``) never does and fails loudly without its CUDA library.

The oracle is deliberately plain and slow.  It shares no code, header, table or helper with the
CUDA library; the only thing both sides use is the seeded input generator module.

* ``paged_attention``  -- float64 C code (``attention.c``): per output row, gather K/V block by
  block through the block table, causal mask over cached-plus-new positions, softmax, weighted V
  sum.  Pages: "SOSP 2023論文解説: PagedAttention" (section "PagedAttentionアルゴリズム", both
  equations; "ブロックテーブルによるメモリ管理"), "Stateful Large Language Model Serving with
  Pensieve" (section "汎化PagedAttentionカーネル"), "KVキャッシュ管理の教科書" (第19章, GQA).
* ``kv_append``  -- the literal scatter of each new token's K/V into its physical slot
  (slot = physical block * B + offset).  Pages: the PagedAttention page, section
  "ブロックテーブルによるメモリ管理" (a new token goes into the current block while it has room,
  otherwise into a newly allocated block).
* ``block_copy`` -- a byte copy of whole blocks, every plane.  Pages: the PagedAttention page,
  section "Copy-on-Writeによるメモリ共有" (a shared block is copied before it is written);
  the Pensieve page, sections "GPU-CPU 2層キャッシュ構造" and "パイプライン化されたswap-in"
  (blocks moved between the CPU tier and the GPU tier).
* ``e4m3_decode`` / ``e4m3_encode`` and the 8-bit variants of attention and append -- K and V
  kept as FP8 E4M3 codes with one scale each ("KVキャッシュ管理の教科書" 第3章: fewer bits per
  element as the third way to shrink the cache; 第22章: quantising KV before decoding).  The
  format follows its published definition (1 sign, 4 exponent bits with bias 7, 3 fraction bits,
  no infinities, S.1111.111 = NaN); encoding rounds to nearest, ties to an even code, and
  saturates at +-448.
* ``oracle.kitty`` -- 2-bit pages with promoted 4-bit key channels ("KVキャッシュ管理の教科書"
  第22章, Kitty): the page quantiser, the record's bytes, and decode attention on the dequantised
  pages plus the unquantised residual page (float64, through ``paged_attention``).
* ``kv_bytes_per_token`` / ``kv_elements`` -- sizing formulas: the Pensieve page, section
  "KVキャッシュのメモリ管理" (M_kv = L x H x 2 x b), and "KVキャッシュ管理の教科書" 第3章
  (2 x batch x layers x seq x head_dim x heads elements).
"""
from __future__ import annotations

import ctypes
import os
import shutil
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attention.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lib = None

DTYPE_CODES = {"f32": 0, "bf16": 1, "f16": 2, "e4m3": 3, "f64": 4}


def build(force: bool = False) -> str:
    """Compile ``attention.c`` with gcc (OpenMP if the toolchain has it).  Strict IEEE double:
    no fast-math and no FMA contraction, so results do not depend on the host ISA."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    os.makedirs(_BUILD, exist_ok=True)
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        raise RuntimeError("oracle: no C compiler found")
    base = [cc, "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    try:
        subprocess.run(base + ["-fopenmp", _SRC, "-o", tmp, "-lm"], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base + [_SRC, "-o", tmp, "-lm"], check=True, capture_output=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def declare(lib):
    """Argument types of the C entry points on a loaded copy of ``attention.c``."""
    p, i32, i64, dbl = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_double
    lib.oracle_paged_attention.restype = ctypes.c_int
    lib.oracle_paged_attention.argtypes = [p, p, p, ctypes.c_int, p, p, p, i32, i32, i32, i32,
                                           i32, i64, i32, i64, dbl, p, i64, p, ctypes.c_int]
    lib.oracle_paged_attention_kv.restype = ctypes.c_int
    lib.oracle_paged_attention_kv.argtypes = [p, p, p, ctypes.c_int, ctypes.c_int, dbl, dbl, p, p, p,
                                              i32, i32, i32, i32, i32, i64, i32, i64, dbl, p, i64, p,
                                              ctypes.c_int]
    lib.oracle_max_threads.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    if _lib is None:
        _lib = declare(ctypes.CDLL(build()))
    return _lib


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def paged_attention(q, k_cache, v_cache, dtype, block_tables, ctx_lens, q_lens, num_q_heads,
                    num_kv_heads, head_dim, block_size, scale, rows=None, threads=1,
                    block_stride=None, kv_dtype=None, k_scale=1.0, v_scale=1.0):
    """Float64 attention rows.

    ``q``: [T, Hq, d]; ``k_cache``/``v_cache``: [num_blocks, Hkv, B, d] (or any array whose
    block ``b`` starts at element ``b * block_stride``); storage as in the generator module
    (float32, or uint16 bit patterns for bf16/f16).  ``kv_dtype="e4m3"``: the caches hold uint8
    E4M3 codes; a cached element's value is its code's value times ``k_scale`` / ``v_scale``.
    ``rows``: optional int array [R, 3] of (sequence, token within its new tokens, query head).
    Returns float64 [T, Hq, d] (all rows) or [R, d].
    """
    lib = _load()
    q = np.ascontiguousarray(q)
    k_cache = np.ascontiguousarray(k_cache)
    v_cache = np.ascontiguousarray(v_cache)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    ctx = np.ascontiguousarray(ctx_lens, dtype=np.int32)
    ql = np.ascontiguousarray(q_lens, dtype=np.int32)
    if num_q_heads % num_kv_heads:
        raise ValueError("num_q_heads must be a multiple of num_kv_heads")
    T = int(ql.sum())
    if block_stride is None:
        block_stride = num_kv_heads * block_size * head_dim
    num_blocks = k_cache.size // block_stride if block_stride else 0
    if rows is None:
        out = np.empty((T, num_q_heads, head_dim), dtype=np.float64)
        rows_p, n_rows = None, 0
    else:
        rows_a = np.ascontiguousarray(rows, dtype=np.int64).reshape(-1, 3)
        out = np.empty((rows_a.shape[0], head_dim), dtype=np.float64)
        rows_p, n_rows = _ptr(rows_a), rows_a.shape[0]
    kvd = DTYPE_CODES[kv_dtype or dtype]
    rc = lib.oracle_paged_attention_kv(_ptr(q), _ptr(k_cache), _ptr(v_cache), DTYPE_CODES[dtype], kvd,
                                       float(k_scale), float(v_scale), _ptr(bt), _ptr(ctx), _ptr(ql),
                                       len(ctx), num_q_heads, num_kv_heads, head_dim, block_size,
                                       num_blocks, bt.shape[1], block_stride, float(scale), rows_p,
                                       n_rows, _ptr(out), int(threads))
    if rc != 0:
        raise ValueError(f"oracle_paged_attention: invalid input (code {rc})")
    return out


def paged_attention_batch(batch, rows=None, threads=1, kv=None):
    """``paged_attention`` on a generator-module ``AttnBatch``; ``kv`` = (k_codes, v_codes,
    k_scale, v_scale) replaces the batch's caches with E4M3 ones."""
    if kv is not None:
        kc, vc, ks, vs = kv
        return paged_attention(batch.q, kc, vc, batch.dtype, batch.block_tables, batch.ctx_lens,
                               batch.q_lens, batch.num_q_heads, batch.num_kv_heads, batch.head_dim,
                               batch.block_size, batch.scale, rows=rows, threads=threads,
                               kv_dtype="e4m3", k_scale=ks, v_scale=vs)
    return paged_attention(batch.q, batch.k_cache, batch.v_cache, batch.dtype, batch.block_tables,
                           batch.ctx_lens, batch.q_lens, batch.num_q_heads, batch.num_kv_heads,
                           batch.head_dim, batch.block_size, batch.scale, rows=rows,
                           threads=threads)


def kv_append(k_new, v_new, slot_mapping, k_cache, v_cache, block_size):
    """Returns copies of the caches with new token t's K/V written at slot ``slot_mapping[t]``:
    physical block ``slot // B``, offset ``slot % B``, every KV head.  Slots < 0 are padding and
    are skipped.  Caches: [num_blocks, Hkv, B, d]; new: [T, Hkv, d].  Bit-level copy."""
    k_out, v_out = k_cache.copy(), v_cache.copy()
    B = int(block_size)
    for t, slot in enumerate(np.asarray(slot_mapping, dtype=np.int64)):
        if slot < 0:
            continue
        blk, off = int(slot) // B, int(slot) % B
        if blk >= k_out.shape[0]:
            raise ValueError(f"slot {slot} outside the pool")
        for h in range(k_out.shape[1]):
            k_out[blk, h, off, :] = k_new[t, h, :]
            v_out[blk, h, off, :] = v_new[t, h, :]
    return k_out, v_out


def e4m3_decode(codes) -> np.ndarray:
    """float64 value of every E4M3 code (uint8 array), from the format's definition."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where((c >> 7) & 1, -1.0, 1.0)
    e = (c >> 3) & 15
    m = c & 7
    normal = (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0)
    sub = (m / 8.0) * 2.0 ** -6
    v = np.where(e == 0, sub, normal)
    v = np.where((e == 15) & (m == 7), np.nan, v)
    return sign * v


def _e4m3_table():
    codes = np.arange(127, dtype=np.uint8)          # the non-negative finite codes, increasing
    return codes, e4m3_decode(codes)


def e4m3_encode(x, inv_scale) -> np.ndarray:
    """E4M3 codes of ``x * inv_scale``: x widened to float32, multiplied by float32(inv_scale) in
    float32 (one rounding), then rounded to the nearest E4M3 value, ties to the even code, with
    magnitudes beyond 448 saturated to 448 and the sign kept (also for results rounded to zero).
    Non-finite inputs are outside this function's domain."""
    y = (np.asarray(x, dtype=np.float32) * np.float32(inv_scale)).astype(np.float64)
    codes, vals = _e4m3_table()
    a = np.abs(y)
    hi = np.searchsorted(vals, a, side="left").clip(0, len(vals) - 1)   # first value >= a
    lo = (hi - 1).clip(0, None)
    d_hi = np.abs(vals[hi] - a)
    d_lo = np.abs(a - vals[lo])
    pick = np.where(d_lo < d_hi, lo, hi)
    tie = d_lo == d_hi
    pick = np.where(tie & (lo % 2 == 0), lo, np.where(tie, hi, pick))
    pick = np.where(a >= vals[-1], len(vals) - 1, pick)
    out = codes[pick].astype(np.uint8)
    return np.where(np.signbit(y), out | np.uint8(0x80), out).astype(np.uint8)


def widen_f32(x, dtype):
    """float32 values of generator-module storage: float32 itself, or uint16 bit patterns of bf16
    (the top half of a binary32) or f16 (IEEE binary16); both widen exactly."""
    x = np.asarray(x)
    if dtype == "f32":
        return x.astype(np.float32)
    if dtype == "bf16":
        return (x.astype(np.uint32) << 16).view(np.float32)
    return x.astype(np.uint16).view(np.float16).astype(np.float32)


def kv_append_e4m3(k_new, v_new, slot_mapping, k_codes, v_codes, block_size, k_scale, v_scale,
                   dtype):
    """``kv_append`` into E4M3 caches: new K (V) elements of ``dtype`` are widened to float32,
    encoded with ``e4m3_encode(x, 1 / scale)`` (the reciprocal rounded to float32) and scattered
    to their slots."""
    kq = e4m3_encode(widen_f32(k_new, dtype), np.float32(1.0) / np.float32(k_scale))
    vq = e4m3_encode(widen_f32(v_new, dtype), np.float32(1.0) / np.float32(v_scale))
    return kv_append(kq, vq, slot_mapping, k_codes, v_codes, block_size)


def block_copy(src, dst, pairs):
    """Returns a copy of ``dst`` where, for every (s, t) in ``pairs``, block t of every plane holds
    the bytes of block s of ``src``.  ``src``/``dst``: [planes, num_blocks, ...] arrays of the same
    per-block shape (src may be a different pool, e.g. a host tier)."""
    out = dst.copy()
    for s, t in np.asarray(pairs, dtype=np.int64).reshape(-1, 2):
        for plane in range(src.shape[0]):
            out[plane, int(t)] = src[plane, int(s)]
    return out


def kv_bytes_per_token(num_layers, hidden, bytes_per_elem):
    """M_kv = L x H x 2 x b: one token's K and V over all layers (Pensieve page)."""
    return int(num_layers) * int(hidden) * 2 * int(bytes_per_elem)


def kv_elements(batch, num_layers, seq_len, head_dim, num_heads):
    """2 x batch x layers x seq x head_dim x heads elements ("KVキャッシュ管理の教科書" 第3章)."""
    return 2 * int(batch) * int(num_layers) * int(seq_len) * int(head_dim) * int(num_heads)
