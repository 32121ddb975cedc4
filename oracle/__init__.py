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

DTYPE_CODES = {"f32": 0, "bf16": 1, "f16": 2}


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


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        p, i32, i64, dbl = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_double
        lib.oracle_paged_attention.restype = ctypes.c_int
        lib.oracle_paged_attention.argtypes = [p, p, p, ctypes.c_int, p, p, p, i32, i32, i32, i32,
                                               i32, i64, i32, i64, dbl, p, i64, p, ctypes.c_int]
        lib.oracle_max_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def paged_attention(q, k_cache, v_cache, dtype, block_tables, ctx_lens, q_lens, num_q_heads,
                    num_kv_heads, head_dim, block_size, scale, rows=None, threads=1,
                    block_stride=None):
    """Float64 attention rows.

    ``q``: [T, Hq, d]; ``k_cache``/``v_cache``: [num_blocks, Hkv, B, d] (or any array whose
    block ``b`` starts at element ``b * block_stride``); storage as in the generator module
    (float32, or uint16 bit patterns for bf16/f16).
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
    rc = lib.oracle_paged_attention(_ptr(q), _ptr(k_cache), _ptr(v_cache), DTYPE_CODES[dtype],
                                    _ptr(bt), _ptr(ctx), _ptr(ql), len(ctx), num_q_heads,
                                    num_kv_heads, head_dim, block_size, num_blocks, bt.shape[1],
                                    block_stride, float(scale), rows_p, n_rows, _ptr(out),
                                    int(threads))
    if rc != 0:
        raise ValueError(f"oracle_paged_attention: invalid input (code {rc})")
    return out


def paged_attention_batch(batch, rows=None, threads=1):
    """``paged_attention`` on a generator-module ``AttnBatch``."""
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
