"""The Python binding's argument checks, on CPU tensors (no GPU, nothing reaches the library):
pa_forward and pa_forward_no_alloc apply the same rules, so a batch that one of them refuses the
other refuses too.  The library reads V with K's geometry and element size and the index arrays
as int32, so a mismatch must stop in the binding, before any pointer is passed on."""
import pytest
import torch

from paged_kv_cache_generalized_gb300 import pagedkv as pk


def _args(**over):
    a = dict(q=torch.zeros(3, 8, 128, dtype=torch.bfloat16),
             k_cache=torch.zeros(10, 2, 16, 128, dtype=torch.bfloat16),
             v_cache=torch.zeros(10, 2, 16, 128, dtype=torch.bfloat16),
             block_tables=torch.zeros(2, 4, dtype=torch.int32),
             ctx_lens=torch.tensor([5, 7], dtype=torch.int32),
             q_lens=torch.tensor([2, 1], dtype=torch.int32))
    a.update(over)
    return a


BAD = {
    "v dtype differs from k": dict(v_cache=torch.zeros(10, 2, 16, 128, dtype=torch.uint8)),
    "v shape differs from k": dict(v_cache=torch.zeros(10, 2, 16, 64, dtype=torch.bfloat16)),
    "int64 block tables": dict(block_tables=torch.zeros(2, 4, dtype=torch.int64)),
    "int64 ctx_lens": dict(ctx_lens=torch.tensor([5, 7], dtype=torch.int64)),
    "non-contiguous block tables": dict(block_tables=torch.zeros(4, 2, dtype=torch.int32).t()),
    "non-contiguous q": dict(q=torch.zeros(8, 3, 128, dtype=torch.bfloat16).transpose(0, 1)),
    "q_lens shorter than ctx_lens": dict(q_lens=torch.tensor([2], dtype=torch.int32)),
    "table rows differ from sequences": dict(block_tables=torch.zeros(3, 4, dtype=torch.int32)),
    "q dtype differs from caches": dict(q=torch.zeros(3, 8, 128, dtype=torch.float16)),
}


@pytest.mark.parametrize("fn", [pk.pa_forward, pk.pa_forward_no_alloc], ids=["pa_forward", "no_alloc"])
@pytest.mark.parametrize("case", sorted(BAD))
def test_forward_wrappers_refuse_the_same_bad_arguments(fn, case):
    with pytest.raises(ValueError):
        fn(**_args(**BAD[case]))


def test_good_arguments_pass_the_checks():
    a = _args()
    dims = pk._forward_args(a["q"], a["k_cache"], a["v_cache"], a["block_tables"], a["ctx_lens"],
                            a["q_lens"], None, None)
    assert (dims.num_seqs, dims.total_q, dims.num_q_heads, dims.num_kv_heads) == (2, 3, 8, 2)
    assert (dims.head_dim, dims.block_size, dims.num_blocks, dims.max_blocks_per_seq) == (128, 16, 10, 4)


BAD_APPEND = {
    "k_new rows differ from q": dict(k_new=torch.zeros(2, 2, 128, dtype=torch.bfloat16)),
    "k_new heads differ from caches": dict(k_new=torch.zeros(3, 4, 128, dtype=torch.bfloat16)),
    "v_new shape differs": dict(v_new=torch.zeros(3, 2, 64, dtype=torch.bfloat16)),
    "k_new dtype differs from q": dict(k_new=torch.zeros(3, 2, 128, dtype=torch.float16)),
    "non-contiguous v_new": dict(v_new=torch.zeros(3, 128, 2, dtype=torch.bfloat16).transpose(1, 2)),
    "int32 slot mapping": dict(slot_mapping=torch.zeros(3, dtype=torch.int32)),
    "slot mapping too short": dict(slot_mapping=torch.zeros(2, dtype=torch.int64)),
}


@pytest.mark.parametrize("case", sorted(BAD_APPEND))
def test_forward_append_refuses_bad_new_tokens(case):
    a = _args()
    a.update(k_new=torch.zeros(3, 2, 128, dtype=torch.bfloat16),
             v_new=torch.zeros(3, 2, 128, dtype=torch.bfloat16),
             slot_mapping=torch.zeros(3, dtype=torch.int64))
    a.update(BAD_APPEND[case])
    with pytest.raises(ValueError):
        pk.pa_forward_append(**a)


@pytest.mark.parametrize("case", sorted(BAD))
def test_forward_append_refuses_what_pa_forward_refuses(case):
    a = _args(**BAD[case])
    a.update(k_new=torch.zeros(3, 2, 128, dtype=torch.bfloat16),
             v_new=torch.zeros(3, 2, 128, dtype=torch.bfloat16),
             slot_mapping=torch.zeros(3, dtype=torch.int64))
    with pytest.raises(ValueError):
        pk.pa_forward_append(**a)
