"""The C ABI without a GPU: the library loads, exports every function include/pagedkv.h declares,
and rejects bad arguments on the host (before any CUDA call) with the documented status codes."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pagedkv.h")


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_generalized_gb300 import build, pagedkv

    build.build()
    return pagedkv.load_library()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\**\s*([a-z_][a-z0-9_]*)\s*\(",
                       text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = _declared_functions()
    for n in ("pa_forward", "pa_forward_workspace_size", "kv_append", "block_copy",
              "pa_get_device_status", "pa_status_string", "pa_version"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for n in _declared_functions():
        assert hasattr(lib, n), f"libpagedkv.so does not export {n}"


def test_binding_names_match_the_header():
    from paged_kv_cache_generalized_gb300 import pagedkv

    assert set(pagedkv.EXPORTED) <= set(_declared_functions())


def test_status_strings_and_version(lib):
    for code, name in enumerate(["PA_OK", "PA_ERR_INVALID_ARG", "PA_ERR_UNSUPPORTED",
                                 "PA_ERR_WORKSPACE", "PA_ERR_CUDA", "PA_ERR_DEVICE"]):
        assert lib.pa_status_string(code).decode() == name
    assert "sm_103a" in lib.pa_version().decode()


def _dims(**kw):
    from paged_kv_cache_generalized_gb300.pagedkv import PaDims

    base = dict(dtype=1, num_seqs=2, total_q=3, num_q_heads=8, num_kv_heads=2, head_dim=128,
                block_size=16, num_blocks=10, max_blocks_per_seq=4, kv_block_stride=0)
    base.update(kw)
    return PaDims(**base)


def test_workspace_size_is_host_only(lib):
    assert lib.pa_forward_workspace_size(ctypes.byref(_dims())) > 0
    assert lib.pa_forward_workspace_size(ctypes.byref(_dims(num_q_heads=7))) == 0
    big = lib.pa_forward_workspace_size(ctypes.byref(_dims(num_seqs=64, total_q=64, max_blocks_per_seq=257)))
    assert big >= 64 * 2 * 64 * 4 * 128 * 4          # split partials: heads x seqs x splits x rows x d


def test_widen_bytes_cover_every_tensor_core_candidate(lib):
    """E4M3 dims with multi-token turns: a 256-byte-aligned candidate prefix (S + 1 int32) and block
    table (S x max_blocks int32), K and V blocks of the query dtype for every sequence that may take
    the tensor-core kernel (q_len * g >= 16, so at most total_q // ceil(16 / g) sequences), then the
    chunk counters and partial rows."""
    def w(**kw):
        return lib.pa_forward_widen_bytes(ctypes.byref(_dims(**kw)))

    def up(x):
        return (x + 255) // 256 * 256

    e4 = dict(kv_dtype=1, k_scale=0.5, v_scale=0.25)
    chunks = 120 * 8 * 4 + 120 * 2 * 128 * 132 * 4       # chunk counters and partial rows
    # 8 sequences, 100 query tokens, GQA 4 (at least 4 tokens each): all 8 may take the kernel
    got = w(num_seqs=8, total_q=100, max_blocks_per_seq=40, **e4)
    assert got == up(9 * 4) + up(8 * 40 * 4) + 8 * 40 * 2 * (2 * 16 * 128 * 2) + chunks
    # 40 query tokens over 30 sequences: at most 10 of them have 4 tokens
    got = w(num_seqs=30, total_q=40, max_blocks_per_seq=7, **e4)
    assert got == up(31 * 4) + up(30 * 7 * 4) + 10 * 7 * 2 * (2 * 16 * 128 * 2) + chunks
    # MHA (g = 1): 16 tokens per candidate
    got = w(num_seqs=4, total_q=50, num_q_heads=2, max_blocks_per_seq=5, **e4)
    assert got == up(5 * 4) + up(4 * 5 * 4) + 3 * 5 * 2 * (2 * 16 * 128 * 2) + chunks
    assert w(num_seqs=4, total_q=4, **e4) == 0                  # decode only
    assert w(num_seqs=2, total_q=30) == 0                      # 16-bit caches need no widening
    assert w(num_seqs=2, total_q=30, head_dim=64, **e4) == 0   # unsupported E4M3 shape
    assert w(num_seqs=2, total_q=30, num_q_heads=7, **e4) == 0  # invalid dims


FAKE = ctypes.c_void_p(0x10000)   # 256-byte aligned, never dereferenced: validation fails first


@pytest.mark.parametrize("kw,code", [
    (dict(num_q_heads=6, num_kv_heads=4), 1),   # Hq % Hkv != 0
    (dict(head_dim=96), 2),                     # unsupported head_dim
    (dict(block_size=8), 2),                    # unsupported block size
    (dict(dtype=7), 1),                         # unknown dtype
    (dict(total_q=1), 1),                       # fewer rows than sequences
    (dict(kv_block_stride=100), 1),             # block stride smaller than a block
])
def test_forward_rejects_bad_dims(lib, kw, code):
    d = _dims(**kw)
    rc = lib.pa_forward(ctypes.byref(d), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.c_float(0.1),
                        ctypes.c_void_p(0x20000), FAKE, 1 << 30, None)
    assert rc == code


def test_forward_rejects_small_or_missing_workspace(lib):
    d = _dims()
    need = lib.pa_forward_workspace_size(ctypes.byref(d))
    args = [ctypes.byref(d), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.c_float(0.1),
            ctypes.c_void_p(0x20000)]
    assert lib.pa_forward(*args, FAKE, need - 1, None) == 3
    assert lib.pa_forward(*args, None, need, None) == 3
    assert lib.pa_forward(*args, ctypes.c_void_p(0x10010), need, None) == 3   # not 256-aligned


def test_forward_rejects_null_and_misaligned_pointers(lib):
    d = _dims()
    rc = lib.pa_forward(ctypes.byref(d), None, FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.c_float(0.1),
                        ctypes.c_void_p(0x20000), FAKE, 1 << 30, None)
    assert rc == 1
    rc = lib.pa_forward(ctypes.byref(d), ctypes.c_void_p(0x10008), FAKE, FAKE, FAKE, FAKE, FAKE,
                        ctypes.c_float(0.1), ctypes.c_void_p(0x20000), FAKE, 1 << 30, None)
    assert rc == 1
    # out aliasing q
    rc = lib.pa_forward(ctypes.byref(d), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.c_float(0.1),
                        FAKE, ctypes.c_void_p(0x40000), 1 << 30, None)
    assert rc == 1


def test_forward_append_rejects_bad_arguments(lib):
    """pa_forward_append runs pa_forward's checks and the append's own, all before device work."""
    d = _dims()
    W = ctypes.c_void_p(0x40000)
    out = ctypes.c_void_p(0x20000)

    def call(dims, q=FAKE, kn=FAKE, vn=FAKE, sm=FAKE, ws=W, wsb=1 << 30):
        return lib.pa_forward_append(ctypes.byref(dims), q, kn, vn, sm, FAKE, FAKE, FAKE, FAKE, FAKE,
                                     ctypes.c_float(0.1), out, ws, wsb, None)

    assert call(_dims(num_q_heads=6, num_kv_heads=4)) == 1          # pa_forward's dims check
    assert call(_dims(head_dim=96)) == 2
    assert call(d, kn=None) == 1                                     # no new K
    assert call(d, sm=None) == 1                                     # no slot mapping
    assert call(d, vn=ctypes.c_void_p(0x10008)) == 1                 # new V not 16-byte aligned
    assert call(d, sm=ctypes.c_void_p(0x10004)) == 1                 # slots not 8-byte aligned
    need = lib.pa_forward_workspace_size(ctypes.byref(d))
    assert call(d, wsb=need - 1) == 3                                # workspace checked first
    assert call(d, q=out) == 1                                       # out aliasing q
    e = _dims(kv_dtype=1, k_scale=0.0, v_scale=1.0)                  # E4M3 without a valid scale
    assert call(e) == 1


def test_timing_events_refuse_half_pairs(lib):
    """A start without a stop (or the reverse) is refused and changes nothing; all NULL clears."""
    assert lib.pa_set_timing_events(FAKE, None, None, None) == 1
    assert lib.pa_set_timing_events(None, None, None, FAKE) == 1
    assert lib.pa_set_timing_events(None, None, None, None) == 0


def test_append_and_copy_reject_bad_arguments(lib):
    from paged_kv_cache_generalized_gb300.pagedkv import BlockCopyDims, KvAppendDims

    a = KvAppendDims(dtype=1, num_tokens=4, num_kv_heads=2, head_dim=4, block_size=16,
                     num_blocks=8, kv_block_stride=0, num_layers=1, new_layer_stride=0,
                     cache_layer_stride=0)
    # a row of 4 bf16 (8 bytes) is not a whole number of 16-byte vectors
    assert lib.kv_append(ctypes.byref(a), FAKE, FAKE, FAKE, FAKE, FAKE, None) == 2
    a.head_dim = 64
    assert lib.kv_append(ctypes.byref(a), None, FAKE, FAKE, FAKE, FAKE, None) == 1
    a.num_tokens = 0                                   # empty append is a no-op
    assert lib.kv_append(ctypes.byref(a), None, None, None, None, None, None) == 0
    c = BlockCopyDims(block_bytes=100, num_planes=1, src_plane_stride=0, dst_plane_stride=0,
                      src_block_stride=0, dst_block_stride=0, src_num_blocks=4, dst_num_blocks=4,
                      num_pairs=1)
    assert lib.block_copy(ctypes.byref(c), FAKE, FAKE, FAKE, None) == 1    # not a multiple of 16
    c.block_bytes = 4096
    c.num_pairs = 0
    assert lib.block_copy(ctypes.byref(c), None, None, None, None) == 0   # no pairs: no-op
    c.num_pairs = 2
    assert lib.block_copy(ctypes.byref(c), ctypes.c_void_p(0x10004), FAKE, FAKE, None) == 1
    c.max_ctas = -1                                    # a negative grid bound is refused
    assert lib.block_copy(ctypes.byref(c), FAKE, FAKE, FAKE, None) == 1


@pytest.mark.parametrize("src_ps,dst_ps,src_bs,dst_bs,ok", [
    (0, 4 * 4096, 0, 0, False),             # two source planes on the same bytes
    (4 * 4096, 0, 0, 0, False),             # two destination planes on the same bytes
    (4096, 4 * 4096, 0, 0, False),          # plane 1 starts at plane 0's block 1
    (2048, 2048, 2 * 4096, 2 * 4096, False),  # side by side but narrower than a block
    (4 * 4096, 8 * 4096, 0, 0, True),       # layer-first: planes one after another
    (4096, 4096, 2 * 4096, 2 * 4096, True),  # block-first: planes side by side in each block
])
def test_block_copy_refuses_overlapping_planes(lib, src_ps, dst_ps, src_bs, dst_bs, ok):
    """With several planes, a plane stride that makes two planes share bytes would let one plane's
    copy overwrite another's blocks; the call refuses it on the host.  Without a GPU an accepted
    layout passes every host check and stops at the device lookup (PA_ERR_CUDA), so the two
    outcomes differ.  The fake pointers must never reach a launch, so the test does not run where
    a GPU is visible."""
    import torch

    from paged_kv_cache_generalized_gb300.pagedkv import BlockCopyDims

    if torch.cuda.is_available():
        pytest.skip("checks host-side refusals with fake pointers: only where no GPU is visible")
    c = BlockCopyDims(block_bytes=4096, num_planes=2, src_plane_stride=src_ps, dst_plane_stride=dst_ps,
                      src_block_stride=src_bs, dst_block_stride=dst_bs, src_num_blocks=4,
                      dst_num_blocks=4, num_pairs=1, max_ctas=0)
    rc = lib.block_copy(ctypes.byref(c), FAKE, FAKE, FAKE, None)
    assert rc == (4 if ok else 1)

def test_e4m3_caches_reject_bad_scales_and_unsupported_shapes(lib):
    from paged_kv_cache_generalized_gb300.pagedkv import KvAppendDims, PaDims

    d = PaDims(dtype=1, num_seqs=1, total_q=1, num_q_heads=8, num_kv_heads=8, head_dim=128,
               block_size=16, num_blocks=10, max_blocks_per_seq=4, kv_block_stride=0, kv_dtype=1,
               k_scale=0.5, v_scale=0.5)
    assert lib.pa_forward_workspace_size(ctypes.byref(d)) > 0
    for field, value, code in (("k_scale", 0.0, 1), ("v_scale", -1.0, 1), ("k_scale", float("nan"), 1),
                               ("v_scale", float("inf"), 1), ("kv_dtype", 2, 1), ("dtype", 0, 2),
                               ("head_dim", 64, 2)):
        bad = PaDims.from_buffer_copy(d)
        setattr(bad, field, value)
        assert lib.pa_forward_workspace_size(ctypes.byref(bad)) == 0, field
        rc = lib.pa_forward(ctypes.byref(bad), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.c_float(0.1),
                            ctypes.c_void_p(0x20000), FAKE, 1 << 30, None)
        assert rc == code, (field, rc)
    a = KvAppendDims(dtype=1, num_tokens=4, num_kv_heads=2, head_dim=64, block_size=16, num_blocks=8,
                     kv_block_stride=0, num_layers=1, new_layer_stride=0, cache_layer_stride=0,
                     kv_dtype=1, k_scale=0.0, v_scale=1.0)
    assert lib.kv_append(ctypes.byref(a), FAKE, FAKE, FAKE, FAKE, FAKE, None) == 1   # zero scale
    a.k_scale = 1.0
    a.head_dim = 8                                     # 8 codes per row: not a 16-byte vector
    assert lib.kv_append(ctypes.byref(a), FAKE, FAKE, FAKE, FAKE, FAKE, None) == 2


def _kdims(**kw):
    from paged_kv_cache_generalized_gb300.pagedkv import KittyDims

    base = dict(dtype=1, num_seqs=4, num_q_heads=8, num_kv_heads=2, head_dim=128, promoted=32,
                num_pages=20, num_res_pages=5, max_pages_per_seq=9)
    base.update(kw)
    return KittyDims(**base)


def test_kitty_record_and_workspace_sizes_are_host_only(lib):
    assert lib.pa_kitty_record_bytes(128, 32) == 11296
    assert lib.pa_kitty_record_bytes(128, 16) == 10784
    assert lib.pa_kitty_record_bytes(64, 16) == 0 and lib.pa_kitty_record_bytes(128, 8) == 0
    ws = lib.pa_kitty_workspace_size(ctypes.byref(_kdims()))
    # counters, arrival counts, and per row (4 x 8) at least two split records of 132 floats (the
    # quantised pages' and the residual page's)
    assert ws >= 4 * 8 * 2 * 132 * 4
    for bad in (dict(promoted=24), dict(head_dim=64), dict(num_q_heads=7), dict(dtype=0),
                dict(num_seqs=0), dict(num_seqs=4097), dict(max_pages_per_seq=0), dict(num_pages=-1)):
        assert lib.pa_kitty_workspace_size(ctypes.byref(_kdims(**bad))) == 0, bad


@pytest.mark.parametrize("kw,code", [(dict(promoted=24), 2), (dict(head_dim=64), 2), (dict(dtype=0), 2),
                                     (dict(num_q_heads=7), 1), (dict(num_seqs=0), 1)])
def test_kitty_calls_reject_bad_dims(lib, kw, code):
    d = _kdims(**kw)
    assert lib.pa_forward_kitty(ctypes.byref(d), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                                ctypes.c_float(0.1), FAKE, FAKE, 1 << 30, None) == code
    # the quantiser reads only the page geometry
    qcode = code if ("num_q_heads" not in kw and "num_seqs" not in kw) else None
    if qcode is not None:
        assert lib.kv_quantize_pages(ctypes.byref(d), FAKE, FAKE, FAKE, 1, FAKE, None) == qcode


def test_kitty_quantiser_ignores_decode_fields(lib):
    d = _kdims(num_seqs=0, num_q_heads=7, max_pages_per_seq=0)
    assert lib.kv_quantize_pages(ctypes.byref(d), FAKE, FAKE, FAKE, 0, FAKE, None) == 0   # no-op
    assert lib.kv_quantize_pages(ctypes.byref(_kdims(num_kv_heads=0)), FAKE, FAKE, FAKE, 0, FAKE, None) == 1


def test_kitty_calls_reject_bad_pointers_and_workspace(lib):
    d = _kdims()
    odd = ctypes.c_void_p(0x10008)
    out = ctypes.c_void_p(0x100000)                 # apart from q
    args = [FAKE] * 7
    assert lib.pa_forward_kitty(ctypes.byref(d), *args, ctypes.c_float(0.1), out, FAKE, 16, None) == 3
    assert lib.pa_forward_kitty(ctypes.byref(d), *args, ctypes.c_float(0.1), FAKE, FAKE, 1 << 30, None) == 1
    assert lib.pa_forward_kitty(ctypes.byref(d), odd, *args[1:], ctypes.c_float(0.1), out, FAKE,
                                1 << 30, None) == 1
    assert lib.pa_forward_kitty(ctypes.byref(d), *args, ctypes.c_float(float("nan")), out, FAKE,
                                1 << 30, None) == 1
    assert lib.kv_quantize_pages(ctypes.byref(d), FAKE, FAKE, FAKE, 0, FAKE, None) == 0   # no-op
    assert lib.kv_quantize_pages(ctypes.byref(d), FAKE, FAKE, FAKE, -1, FAKE, None) == 1
    assert lib.kv_quantize_pages(ctypes.byref(d), odd, FAKE, FAKE, 1, FAKE, None) == 1
