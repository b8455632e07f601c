"""Refusals of the merge and sampling entry points, on the CPU: every check
below fails before anything is launched, so host tensors suffice."""
import pytest
import torch

import paged_kv_attention_13_gb300 as fi


def _status(fn, *a, **k):
    with pytest.raises(fi.FiError) as e:
        fn(*a, **k)
    return e.value.status_name


def _states(rows=4, heads=2, d=8, dtype=torch.float32):
    return torch.zeros((rows, heads, d), dtype=dtype), torch.zeros((rows, heads))


def test_merge_state_refusals():
    va, sa = _states()
    vb, sb = _states()
    # v shapes that differ
    assert _status(fi.fi_merge_state, va, sa, torch.zeros((4, 2, 16)), sb) == "FI_ERR_INVALID_ARG"
    # a strided last dim
    strided = torch.zeros((4, 2, 16))[:, :, ::2]
    assert _status(fi.fi_merge_state, strided, sa, vb, sb) == "FI_ERR_STRIDED_LAST_DIM"
    # LSEs that are not fp32
    assert _status(fi.fi_merge_state, va, sa.half(), vb, sb) == "FI_ERR_INVALID_ARG"
    # v dtypes that differ
    assert _status(fi.fi_merge_state, va, sa, vb.half(), sb) == "FI_ERR_INVALID_ARG"
    # an output that is not packed
    out = torch.zeros((4, 4, 8))[:, ::2, :]
    assert _status(fi.fi_merge_state, va, sa, vb, sb, v_out=out) == "FI_ERR_NONCONTIGUOUS_OUTPUT"


def test_merge_states_refusals():
    v, s = _states(rows=6)
    indptr = torch.tensor([0, 2, 6], dtype=torch.int32)
    out, s_out = _states(rows=2)
    assert _status(fi.fi_merge_states, v, s, indptr, -1, v_out=out,
                   s_out=s_out) == "FI_ERR_INVALID_ARG"
    assert _status(fi.fi_merge_states, v.half(), s, indptr, 2) == "FI_ERR_INVALID_ARG"
    assert _status(fi.fi_merge_states, v, s.half(), indptr, 2) == "FI_ERR_INVALID_ARG"


def test_chain_speculative_sampling_refusals():
    B, n, V = 3, 4, 64
    dp = torch.zeros((B, n, V))
    ids = torch.zeros((B, n), dtype=torch.int32)
    tp = torch.zeros((B, n + 1, V))
    ua = torch.zeros((B, n))
    us = torch.zeros((B,))
    f = fi.fi_chain_speculative_sampling
    # target probabilities that are not fp32
    assert _status(f, dp, ids, tp.half(), ua, us) == "FI_ERR_INVALID_ARG"
    # an output of the wrong shape
    assert _status(f, dp, ids, tp, ua, us,
                   output_token_ids=torch.zeros((B, n), dtype=torch.int32)) == "FI_ERR_INVALID_ARG"
    # uniforms for the wrong batch
    assert _status(f, dp, ids, tp, ua, torch.zeros((B + 1,))) == "FI_ERR_INVALID_ARG"
