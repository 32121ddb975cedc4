"""Helpers for the GPU parity tests: moving generator arrays to the device and comparing against
the float64 oracle with the stated tolerances."""
import numpy as np
import torch

# Tolerances against the float64 oracle (max abs, mean abs).  bf16: 2e-2 / 2e-3 as stated for
# the attention outputs; fp32: 1e-4; f16 (not stated) is held to the bf16 bar.
TOL = {"f32": (1e-4, 1e-5), "bf16": (2e-2, 2e-3), "f16": (2e-2, 2e-3)}
TORCH_DTYPE = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}


def dev():
    return torch.device("cuda:0")


def to_dev(x, dtype=None, pin=False):
    t = torch.from_numpy(np.ascontiguousarray(x))
    if dtype in ("bf16", "f16"):
        t = t.view(torch.int16).view(TORCH_DTYPE[dtype])
    if pin:
        return t.pin_memory()
    return t.to(dev(), non_blocking=False)


def bits(t):
    """Raw bytes of a tensor as a numpy uint8 array (host copy)."""
    return t.detach().contiguous().cpu().view(torch.uint8).numpy()


def as_f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def batch_to_dev(b):
    return dict(q=to_dev(b.q, b.dtype), k=to_dev(b.k_cache, b.dtype), v=to_dev(b.v_cache, b.dtype),
                bt=to_dev(b.block_tables), ctx=to_dev(b.ctx_lens), ql=to_dev(b.q_lens))


def run_forward(b, d=None, **kw):
    import paged_kv_cache_generalized_gb300 as pkg

    d = d or batch_to_dev(b)
    out = pkg.pa_forward(d["q"], d["k"], d["v"], d["bt"], d["ctx"], d["ql"], b.scale, **kw)
    torch.cuda.synchronize()
    return out


def assert_close(got, ref, dtype, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64).reshape(got.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - ref)
    mx, mean = TOL[dtype]
    assert err.max() <= mx, f"{what}: max abs error {err.max():.3e} > {mx}"
    assert err.mean() <= mean, f"{what}: mean abs error {err.mean():.3e} > {mean}"
    return float(err.max()), float(err.mean())


def sample_rows(b, n, seed=0, include_last=True):
    """(seq, token, head) rows: a seeded sample plus every sequence's last token (the longest
    causal range) and first token."""
    rng = np.random.default_rng(seed)
    rows = set()
    for i in range(b.num_seqs):
        for j in {0, int(b.q_lens[i]) - 1} if include_last else {0}:
            rows.add((i, j, int(rng.integers(b.num_q_heads))))
    while len(rows) < n + 2 * b.num_seqs:
        i = int(rng.integers(b.num_seqs))
        rows.add((i, int(rng.integers(b.q_lens[i])), int(rng.integers(b.num_q_heads))))
    return np.array(sorted(rows), dtype=np.int64)


def gather_rows(out, b, rows):
    cu = b.cu_q
    idx_t = torch.tensor([cu[i] + j for i, j, _ in rows], device=out.device)
    idx_h = torch.tensor([h for _, _, h in rows], device=out.device)
    return as_f64(out[idx_t, idx_h])
