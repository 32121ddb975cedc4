"""Thin Python binding of libpagedkv.so (ctypes): argument marshalling only.

Every computation runs in the library's CUDA kernels; PyTorch supplies device memory, the
workspace allocation and the current stream.  There is no CPU fallback: if the library has not
been built (``paged_kv_cache_generalized_gb300.build.build()``) every call raises.

The functions mirror the C ABI in ``include/pagedkv.h`` (same names and semantics).
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

_lib = None

PA_OK = 0
STATUS_BITS = {
    0x1: "PA_DEV_BAD_BLOCK_ID",
    0x2: "PA_DEV_BAD_LENGTHS",
    0x4: "PA_DEV_BAD_SLOT",
    0x8: "PA_DEV_BAD_PAIR",
    0x10: "PA_DEV_TIMEOUT",
}
_DTYPES = {torch.float32: 0, torch.bfloat16: 1, torch.float16: 2}
PA_KV_SAME, PA_KV_E4M3 = 0, 1
# K/V caches of one-byte E4M3 codes may be given as uint8 or as torch's float8_e4m3fn
_E4M3 = tuple(t for t in (torch.uint8, getattr(torch, "float8_e4m3fn", None)) if t is not None)
_ELEM = {torch.float32: 4, torch.bfloat16: 2, torch.float16: 2}

EXPORTED = ("pa_forward_workspace_size", "pa_forward_widen_bytes", "pa_forward", "pa_forward_no_alloc", "pa_forward_append", "pa_set_timing_events", "kv_append",
            "block_copy", "pa_get_device_status", "pa_status_string", "pa_version",
            "pa_kitty_record_bytes", "pa_kitty_workspace_size", "kv_quantize_pages",
            "pa_forward_kitty")
KITTY_PAGE_TOKENS = 128
NO_ALLOC_WORKSPACE_BYTES = 32 * 1024 * 1024


class PaDims(ctypes.Structure):
    _fields_ = [("dtype", ctypes.c_int32), ("num_seqs", ctypes.c_int32), ("total_q", ctypes.c_int64),
                ("num_q_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("num_blocks", ctypes.c_int64), ("max_blocks_per_seq", ctypes.c_int32),
                ("kv_block_stride", ctypes.c_int64), ("kv_dtype", ctypes.c_int32),
                ("k_scale", ctypes.c_float), ("v_scale", ctypes.c_float)]


class KvAppendDims(ctypes.Structure):
    _fields_ = [("dtype", ctypes.c_int32), ("num_tokens", ctypes.c_int64),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("block_size", ctypes.c_int32), ("num_blocks", ctypes.c_int64),
                ("kv_block_stride", ctypes.c_int64), ("num_layers", ctypes.c_int32),
                ("new_layer_stride", ctypes.c_int64), ("cache_layer_stride", ctypes.c_int64),
                ("kv_dtype", ctypes.c_int32), ("k_scale", ctypes.c_float), ("v_scale", ctypes.c_float)]


class BlockCopyDims(ctypes.Structure):
    _fields_ = [("block_bytes", ctypes.c_int64), ("num_planes", ctypes.c_int32),
                ("src_plane_stride", ctypes.c_int64), ("dst_plane_stride", ctypes.c_int64),
                ("src_block_stride", ctypes.c_int64), ("dst_block_stride", ctypes.c_int64),
                ("src_num_blocks", ctypes.c_int64), ("dst_num_blocks", ctypes.c_int64),
                ("num_pairs", ctypes.c_int64), ("max_ctas", ctypes.c_int32)]


class KittyDims(ctypes.Structure):
    _fields_ = [("dtype", ctypes.c_int32), ("num_seqs", ctypes.c_int32),
                ("num_q_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("promoted", ctypes.c_int32),
                ("num_pages", ctypes.c_int64), ("num_res_pages", ctypes.c_int64),
                ("max_pages_per_seq", ctypes.c_int32)]


class PagedKVError(RuntimeError):
    pass


def library_path() -> str:
    return _build.LIB_PATH


def load_library(path: str | None = None):
    """Loads libpagedkv.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or _build.LIB_PATH
    if not os.path.exists(path):
        raise PagedKVError(f"libpagedkv.so not found at {path}: build it first "
                           "(paged_kv_cache_generalized_gb300.build.build())")
    lib = ctypes.CDLL(path)
    P, sz = ctypes.c_void_p, ctypes.c_size_t
    lib.pa_forward_workspace_size.restype = sz
    lib.pa_forward_workspace_size.argtypes = [ctypes.POINTER(PaDims)]
    lib.pa_forward_widen_bytes.restype = sz
    lib.pa_forward_widen_bytes.argtypes = [ctypes.POINTER(PaDims)]
    lib.pa_forward.restype = ctypes.c_int
    lib.pa_forward.argtypes = [ctypes.POINTER(PaDims), P, P, P, P, P, P, ctypes.c_float, P, P, sz, P]
    lib.pa_forward_no_alloc.restype = ctypes.c_int
    lib.pa_forward_no_alloc.argtypes = [ctypes.POINTER(PaDims), P, P, P, P, P, P, ctypes.c_float,
                                        P, P]
    lib.pa_forward_append.restype = ctypes.c_int
    lib.pa_forward_append.argtypes = [ctypes.POINTER(PaDims), P, P, P, P, P, P, P, P, P,
                                      ctypes.c_float, P, P, sz, P]
    lib.pa_set_timing_events.restype = ctypes.c_int
    lib.pa_set_timing_events.argtypes = [P, P, P, P]
    lib.kv_append.restype = ctypes.c_int
    lib.kv_append.argtypes = [ctypes.POINTER(KvAppendDims), P, P, P, P, P, P]
    lib.block_copy.restype = ctypes.c_int
    lib.block_copy.argtypes = [ctypes.POINTER(BlockCopyDims), P, P, P, P]
    lib.pa_get_device_status.restype = ctypes.c_int
    lib.pa_get_device_status.argtypes = [ctypes.POINTER(ctypes.c_uint32), P]
    lib.pa_status_string.restype = ctypes.c_char_p
    lib.pa_status_string.argtypes = [ctypes.c_int]
    lib.pa_version.restype = ctypes.c_char_p
    lib.pa_kitty_record_bytes.restype = sz
    lib.pa_kitty_record_bytes.argtypes = [ctypes.c_int32, ctypes.c_int32]
    lib.pa_kitty_workspace_size.restype = sz
    lib.pa_kitty_workspace_size.argtypes = [ctypes.POINTER(KittyDims)]
    lib.kv_quantize_pages.restype = ctypes.c_int
    lib.kv_quantize_pages.argtypes = [ctypes.POINTER(KittyDims), P, P, P, ctypes.c_int64, P, P]
    lib.pa_forward_kitty.restype = ctypes.c_int
    lib.pa_forward_kitty.argtypes = [ctypes.POINTER(KittyDims), P, P, P, P, P, P, P, ctypes.c_float,
                                     P, P, sz, P]
    _lib = lib
    return lib


def _check(rc: int, what: str):
    if rc != PA_OK:
        name = load_library().pa_status_string(rc).decode()
        raise PagedKVError(f"{what} failed: {name}")


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _cache_geometry(cache: torch.Tensor):
    """[num_blocks, Hkv, B, d] view (the block dim may be strided, e.g. a block-first pool)."""
    if cache.dim() != 4:
        raise ValueError("cache must be [num_blocks, num_kv_heads, block_size, head_dim]")
    nb, hkv, bs, d = cache.shape
    if cache.stride(3) != 1 or cache.stride(2) != d or cache.stride(1) != bs * d:
        raise ValueError("cache: the (head, slot, dim) dims of a block must be contiguous")
    return nb, hkv, bs, d, cache.stride(0)


def _kv_kind(cache, dtype, k_scale, v_scale):
    """(kv_dtype, k_scale, v_scale) of a cache tensor: E4M3 codes need both scales."""
    if cache.dtype in _E4M3:
        if k_scale is None or v_scale is None:
            raise ValueError("E4M3 caches need k_scale and v_scale")
        return PA_KV_E4M3, float(k_scale), float(v_scale)
    if cache.dtype != dtype:
        raise ValueError("q and caches must share a dtype (or the caches hold E4M3 codes)")
    return PA_KV_SAME, 1.0, 1.0


def forward_dims(q, k_cache, block_tables, ctx_lens, k_scale=None, v_scale=None) -> PaDims:
    nb, hkv, bs, d, bstride = _cache_geometry(k_cache)
    T, hq, dq = q.shape
    if dq != d:
        raise ValueError("q and cache head_dim differ")
    kind, ks, vs = _kv_kind(k_cache, q.dtype, k_scale, v_scale)
    return PaDims(_DTYPES[q.dtype], ctx_lens.shape[0], T, hq, hkv, d, bs, nb,
                  block_tables.shape[1], bstride, kind, ks, vs)


def _forward_args(q, k_cache, v_cache, block_tables, ctx_lens, q_lens, k_scale, v_scale) -> PaDims:
    """Checks the arguments of pa_forward and pa_forward_no_alloc (one set of rules for both:
    the library reads V with K's geometry and element size, and the index arrays as int32) and
    returns their dims.  Raises ValueError before anything reaches the device."""
    if q.dim() != 3 or not q.is_contiguous():
        raise ValueError("q must be contiguous [T, Hq, d]")
    if v_cache.shape != k_cache.shape or v_cache.stride() != k_cache.stride():
        raise ValueError("k_cache and v_cache must have the same shape and strides")
    if v_cache.dtype != k_cache.dtype:
        raise ValueError("k_cache and v_cache must share a dtype")
    for t in (block_tables, ctx_lens, q_lens):
        if t.dtype != torch.int32 or not t.is_contiguous():
            raise ValueError("block_tables, ctx_lens and q_lens must be contiguous int32")
    if block_tables.dim() != 2 or ctx_lens.dim() != 1 or q_lens.shape != ctx_lens.shape:
        raise ValueError("block_tables must be [S, max_blocks], ctx_lens and q_lens [S]")
    if block_tables.shape[0] != ctx_lens.shape[0]:
        raise ValueError("block_tables and ctx_lens disagree on the number of sequences")
    return forward_dims(q, k_cache, block_tables, ctx_lens, k_scale, v_scale)


def forward_workspace_size(q, k_cache, block_tables, ctx_lens) -> int:
    """Workspace bytes for pa_forward on these shapes: the required part, plus (E4M3 caches with
    multi-token turns) the widening scratch that lets every tensor-core sequence widen."""
    dims = forward_dims(q, k_cache, block_tables, ctx_lens, 1.0, 1.0)
    return _workspace_bytes(load_library(), dims)


def forward_widen_bytes(q, k_cache, block_tables, ctx_lens) -> int:
    """The widening scratch part of forward_workspace_size (0 unless the caches are E4M3)."""
    dims = forward_dims(q, k_cache, block_tables, ctx_lens, 1.0, 1.0)
    return int(load_library().pa_forward_widen_bytes(ctypes.byref(dims)))


def _workspace_bytes(lib, dims) -> int:
    base = int(lib.pa_forward_workspace_size(ctypes.byref(dims)))
    return base + int(lib.pa_forward_widen_bytes(ctypes.byref(dims))) if base else 0


def pa_forward(q, k_cache, v_cache, block_tables, ctx_lens, q_lens, scale=None, out=None,
               workspace=None, stream=None, k_scale=None, v_scale=None):
    """Generalized paged attention (see ``pa_forward`` in include/pagedkv.h).

    q: [T, Hq, d]; k_cache/v_cache: [num_blocks, Hkv, B, d] in q's dtype, or E4M3 codes (uint8 or
    float8_e4m3fn) with ``k_scale`` / ``v_scale``; block_tables: int32 [S, max_blocks];
    ctx_lens/q_lens: int32 [S].  Returns ``out`` ([T, Hq, d])."""
    dims = _forward_args(q, k_cache, v_cache, block_tables, ctx_lens, q_lens, k_scale, v_scale)
    lib = load_library()
    if scale is None:
        scale = 1.0 / float(dims.head_dim) ** 0.5
    if out is None:
        out = torch.empty_like(q)
    need = _workspace_bytes(lib, dims)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    rc = lib.pa_forward(ctypes.byref(dims), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                        _ptr(block_tables), _ptr(ctx_lens), _ptr(q_lens), ctypes.c_float(scale),
                        _ptr(out), _ptr(workspace), workspace.numel() * workspace.element_size(),
                        _stream(stream))
    _check(rc, "pa_forward")
    return out


def pa_forward_no_alloc(q, k_cache, v_cache, block_tables, ctx_lens, q_lens, scale=None, out=None,
                        stream=None, k_scale=None, v_scale=None):
    """pa_forward with the library's own fixed-size scratch (see ``pa_forward_no_alloc`` in
    include/pagedkv.h): for callers that cannot allocate device memory.  Raises if the batch
    needs more scratch than the library holds."""
    dims = _forward_args(q, k_cache, v_cache, block_tables, ctx_lens, q_lens, k_scale, v_scale)
    lib = load_library()
    if scale is None:
        scale = 1.0 / float(dims.head_dim) ** 0.5
    if out is None:
        out = torch.empty_like(q)
    rc = lib.pa_forward_no_alloc(ctypes.byref(dims), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                 _ptr(block_tables), _ptr(ctx_lens), _ptr(q_lens),
                                 ctypes.c_float(scale), _ptr(out), _stream(stream))
    _check(rc, "pa_forward_no_alloc")
    return out


def _append_args(q, k_new, v_new, slot_mapping, k_cache):
    """Checks the new-token arguments of pa_forward_append (raises ValueError)."""
    T, _, d = q.shape
    hkv = k_cache.shape[1]
    if k_new.shape != (T, hkv, d) or v_new.shape != k_new.shape:
        raise ValueError("k_new and v_new must be [T, Hkv, d] with q's T and d")
    if k_new.dtype != q.dtype or v_new.dtype != q.dtype:
        raise ValueError("k_new and v_new must have q's dtype")
    if not k_new.is_contiguous() or not v_new.is_contiguous():
        raise ValueError("k_new and v_new must be contiguous")
    if slot_mapping.dtype != torch.int64 or slot_mapping.shape != (T,) or not slot_mapping.is_contiguous():
        raise ValueError("slot_mapping must be contiguous int64 [T]")


def pa_forward_append(q, k_new, v_new, slot_mapping, k_cache, v_cache, block_tables, ctx_lens, q_lens,
                      scale=None, out=None, workspace=None, stream=None, k_scale=None, v_scale=None):
    """Writes the step's new tokens into their slots, then runs pa_forward (see
    ``pa_forward_append`` in include/pagedkv.h); same result as ``kv_append`` followed by
    ``pa_forward``.  k_new/v_new: [T, Hkv, d] in q's dtype, one row per query token;
    slot_mapping: int64 [T].  Returns ``out``."""
    dims = _forward_args(q, k_cache, v_cache, block_tables, ctx_lens, q_lens, k_scale, v_scale)
    _append_args(q, k_new, v_new, slot_mapping, k_cache)
    lib = load_library()
    if scale is None:
        scale = 1.0 / float(dims.head_dim) ** 0.5
    if out is None:
        out = torch.empty_like(q)
    need = _workspace_bytes(lib, dims)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    rc = lib.pa_forward_append(ctypes.byref(dims), _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(slot_mapping),
                               _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), _ptr(ctx_lens),
                               _ptr(q_lens), ctypes.c_float(scale), _ptr(out), _ptr(workspace),
                               workspace.numel() * workspace.element_size(), _stream(stream))
    _check(rc, "pa_forward_append")
    return out


def _event_handle(ev):
    """Raw cudaEvent_t of a torch.cuda.Event (recorded once on the current stream first, since
    torch creates the CUDA event at its first record)."""
    if ev is None:
        return None
    if not ev.cuda_event:
        ev.record()
    return ctypes.c_void_p(ev.cuda_event)


def set_timing_events(tc=None, cc=None):
    """Records (start, stop) torch.cuda.Event pairs around the attention kernels of later calls
    (see ``pa_set_timing_events`` in include/pagedkv.h): ``tc`` around the tcgen05 kernel, ``cc``
    around the decode kernel, each on the stream that kernel runs on.  None stops recording that
    pair."""
    lib = load_library()
    ts, te = (None, None) if tc is None else tc
    cs, ce = (None, None) if cc is None else cc
    rc = lib.pa_set_timing_events(_event_handle(ts), _event_handle(te), _event_handle(cs),
                                  _event_handle(ce))
    _check(rc, "pa_set_timing_events")


def kitty_record_bytes(promoted: int, head_dim: int = 128) -> int:
    """Bytes of one (page, KV head) record of the 2-bit page format (0 if unsupported)."""
    return int(load_library().pa_kitty_record_bytes(head_dim, promoted))


def kitty_dims(q_or_res, pages, promoted, num_q_heads=None, num_seqs=1, res_pages=None,
               max_pages_per_seq=1) -> KittyDims:
    """KittyDims from the page pool ([num_pages, Hkv, record] uint8) and a residual pool
    ([num_res, Hkv, 128, d])."""
    if pages.dim() != 3 or pages.dtype != torch.uint8 or not pages.is_contiguous():
        raise ValueError("pages must be contiguous uint8 [num_pages, Hkv, record_bytes]")
    if res_pages is None or res_pages.dim() != 4 or not res_pages.is_contiguous():
        raise ValueError("residual pages must be contiguous [num_res, Hkv, 128, d]")
    if res_pages.dtype not in (torch.bfloat16, torch.float16):
        raise ValueError("residual pages must be bf16 or f16")
    hkv = pages.shape[1]
    return KittyDims(_DTYPES[res_pages.dtype], int(num_seqs), int(num_q_heads or hkv), int(hkv),
                     int(res_pages.shape[3]), int(promoted), int(pages.shape[0]),
                     int(res_pages.shape[0]), int(max_pages_per_seq))


def kv_quantize_pages(res_k, res_v, pairs, pages, promoted, stream=None):
    """Quantises residual page s into record t of ``pages`` for every (s, t) row of ``pairs``
    (int64 [P, 2]), every KV head (see ``kv_quantize_pages`` in include/pagedkv.h)."""
    lib = load_library()
    if res_v.shape != res_k.shape or res_v.dtype != res_k.dtype:
        raise ValueError("res_k and res_v must match")
    if pairs.dtype != torch.int64 or not pairs.is_contiguous():
        raise ValueError("pairs must be contiguous int64 [P, 2]")
    dims = kitty_dims(None, pages, promoted, res_pages=res_k)
    rc = lib.kv_quantize_pages(ctypes.byref(dims), _ptr(res_k), _ptr(res_v), _ptr(pairs),
                               ctypes.c_int64(pairs.numel() // 2), _ptr(pages), _stream(stream))
    _check(rc, "kv_quantize_pages")
    return pages


def kitty_workspace_size(q, pages, res_k, block_tables, promoted) -> int:
    """Workspace bytes pa_forward_kitty needs for these shapes (0 if unsupported)."""
    dims = kitty_dims(q, pages, promoted, num_q_heads=q.shape[1], num_seqs=q.shape[0], res_pages=res_k,
                      max_pages_per_seq=block_tables.shape[1])
    return int(load_library().pa_kitty_workspace_size(ctypes.byref(dims)))


def pa_forward_kitty(q, pages, res_k, res_v, block_tables, ctx_lens, q_lens, promoted, scale=None,
                     out=None, workspace=None, stream=None):
    """Decode attention over 2-bit pages with promoted 4-bit key channels plus each sequence's
    residual page (see ``pa_forward_kitty`` in include/pagedkv.h).  q: [S, Hq, 128]; pages:
    uint8 [num_pages, Hkv, record]; res_k/res_v: [num_res, Hkv, 128, 128] in q's dtype;
    block_tables int32 [S, max_pages]; ctx_lens/q_lens int32 [S] (q_lens all 1)."""
    lib = load_library()
    for t in (block_tables, ctx_lens, q_lens):
        if t.dtype != torch.int32 or not t.is_contiguous():
            raise ValueError("block_tables, ctx_lens and q_lens must be contiguous int32")
    if not q.is_contiguous() or q.dim() != 3:
        raise ValueError("q must be contiguous [S, Hq, d]")
    if res_v.shape != res_k.shape or res_k.dtype != q.dtype or res_v.dtype != q.dtype:
        raise ValueError("residual pages must match each other and q's dtype")
    dims = kitty_dims(q, pages, promoted, num_q_heads=q.shape[1], num_seqs=q.shape[0],
                      res_pages=res_k, max_pages_per_seq=block_tables.shape[1])
    if scale is None:
        scale = 1.0 / float(dims.head_dim) ** 0.5
    if out is None:
        out = torch.empty_like(q)
    need = int(lib.pa_kitty_workspace_size(ctypes.byref(dims)))
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    rc = lib.pa_forward_kitty(ctypes.byref(dims), _ptr(q), _ptr(pages), _ptr(res_k), _ptr(res_v),
                              _ptr(block_tables), _ptr(ctx_lens), _ptr(q_lens),
                              ctypes.c_float(scale), _ptr(out), _ptr(workspace),
                              workspace.numel() * workspace.element_size(), _stream(stream))
    _check(rc, "pa_forward_kitty")
    return out


def kv_append(k_new, v_new, slot_mapping, k_cache, v_cache, stream=None, k_scale=None, v_scale=None):
    """Writes new tokens' K/V into their slots (see ``kv_append`` in include/pagedkv.h).

    Single layer: k_new [T, Hkv, d], caches [num_blocks, Hkv, B, d].  Several layers: k_new
    [L, T, Hkv, d], caches [L, num_blocks, Hkv, B, d] (layer and block dims may be strided).
    E4M3 caches (uint8 or float8_e4m3fn) quantise the new tokens with ``k_scale`` / ``v_scale``."""
    lib = load_library()
    if k_new.dim() == 3:
        k_new, v_new, k_cache, v_cache = (x.unsqueeze(0) for x in (k_new, v_new, k_cache, v_cache))
    L, T, hkv, d = k_new.shape
    if k_cache.shape[0] != L or v_cache.shape != k_cache.shape or v_new.shape != k_new.shape:
        raise ValueError("kv_append: inconsistent shapes")
    if k_cache.stride() != v_cache.stride() or k_new.stride() != v_new.stride():
        raise ValueError("kv_append: K and V must share strides")
    nb, hkv_c, bs, dc, bstride = _cache_geometry(k_cache[0])
    if (hkv_c, dc) != (hkv, d):
        raise ValueError("kv_append: cache and new tokens disagree on heads or head_dim")
    if k_new.stride(3) != 1 or k_new.stride(2) != d or k_new.stride(1) != hkv * d:
        raise ValueError("kv_append: each layer of k_new must be contiguous [T, Hkv, d]")
    if slot_mapping.dtype != torch.int64 or not slot_mapping.is_contiguous():
        raise ValueError("slot_mapping must be contiguous int64")
    if k_cache.dtype != v_cache.dtype:
        raise ValueError("kv_append: k_cache and v_cache must share a dtype")
    kind, ks, vs = _kv_kind(k_cache, k_new.dtype, k_scale, v_scale)
    dims = KvAppendDims(_DTYPES[k_new.dtype], T, hkv, d, bs, nb, bstride, L,
                        k_new.stride(0) if L > 1 else 0, k_cache.stride(0) if L > 1 else 0,
                        kind, ks, vs)
    rc = lib.kv_append(ctypes.byref(dims), _ptr(k_new), _ptr(v_new), _ptr(slot_mapping),
                       _ptr(k_cache), _ptr(v_cache), _stream(stream))
    _check(rc, "kv_append")


def block_copy(src, dst, pairs, stream=None, max_ctas=0):
    """Copies whole blocks of every plane (see ``block_copy`` in include/pagedkv.h).

    src/dst: [planes, num_blocks, ...] (each block's trailing dims contiguous; src or dst may be
    pinned host memory); pairs: int64 [P, 2] (source block, destination block) on the device.
    max_ctas > 0 bounds the copy's grid so that kernels on other streams keep the other SMs."""
    lib = load_library()
    if src.dim() < 2 or dst.dim() < 2 or src.shape[0] != dst.shape[0]:
        raise ValueError("block_copy: src and dst must be [planes, num_blocks, ...] with equal planes")
    if src.shape[2:] != dst.shape[2:] or src.dtype != dst.dtype:
        raise ValueError("block_copy: block shapes differ")
    es = src.element_size()
    block_elems = 1
    for x in src.shape[2:]:
        block_elems *= x
    for t in (src, dst):
        if not t[0, 0].is_contiguous():
            raise ValueError("block_copy: each block must be contiguous")
    if pairs.dtype != torch.int64 or not pairs.is_contiguous():
        raise ValueError("pairs must be contiguous int64 [P, 2]")
    dims = BlockCopyDims(block_elems * es, src.shape[0], src.stride(0) * es, dst.stride(0) * es,
                         src.stride(1) * es, dst.stride(1) * es, src.shape[1], dst.shape[1],
                         pairs.numel() // 2, int(max_ctas))
    rc = lib.block_copy(ctypes.byref(dims), _ptr(src), _ptr(dst), _ptr(pairs), _stream(stream))
    _check(rc, "block_copy")


def device_status(stream=None) -> int:
    """Synchronises the stream, returns and clears the device status bits (0 = no fault seen)."""
    lib = load_library()
    flags = ctypes.c_uint32(0)
    rc = lib.pa_get_device_status(ctypes.byref(flags), _stream(stream))
    if rc not in (0, 5):
        _check(rc, "pa_get_device_status")
    return int(flags.value)


def status_names(flags: int):
    return [n for b, n in STATUS_BITS.items() if flags & b]


def version() -> str:
    return load_library().pa_version().decode()
