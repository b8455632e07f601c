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


def test_noalloc_decode_refusals():
    """The no-allocation decode checks its shapes on the host before it looks
    up its scratch or launches anything, so host tensors suffice."""
    B, Hq, Hk, d, P, pages = 3, 8, 2, 128, 16, 10
    q = torch.zeros((B, Hq, d), dtype=torch.bfloat16)
    k = torch.zeros((pages, P, Hk, d), dtype=torch.bfloat16)
    v = torch.zeros_like(k)
    idx = torch.zeros((pages,), dtype=torch.int32)
    indptr = torch.zeros((B + 1,), dtype=torch.int32)
    last = torch.ones((B,), dtype=torch.int32)
    f = fi.fi_batch_decode_paged_noalloc
    # a V cache with fewer pages than K: the K map's extent would let V's
    # copies read past V's allocation
    assert _status(f, q, k, v[: pages - 1], idx, indptr, last, 0.1) == "FI_ERR_INVALID_ARG"
    # an lse with fewer rows than the batch
    assert _status(f, q, k, v, idx, indptr, last, 0.1,
                   lse=torch.zeros((B - 1, Hq))) == "FI_ERR_INVALID_ARG"
    # an out with fewer rows than the batch
    assert _status(f, q, k, v, idx, indptr, last, 0.1,
                   out=torch.zeros((B - 1, Hq, d), dtype=torch.bfloat16)) == "FI_ERR_INVALID_ARG"
    # kv_chunks outside [1, 64]
    assert _status(f, q, k, v, idx, indptr, last, 0.1, kv_chunks=0) == "FI_ERR_INVALID_ARG"
    # a group the kernel is not built for
    assert _status(f, torch.zeros((B, 3 * Hk, d), dtype=torch.bfloat16), k, v, idx, indptr,
                   last, 0.1) == "FI_ERR_UNSUPPORTED"


def test_log_levels_print_refusals_and_plans():
    """FI_LOG=1 prints each refusal on stderr, 2 also each committed plan;
    unset prints nothing (host-only plans, no GPU)."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    code = (
        "import paged_kv_attention_13_gb300 as fi\n"
        "p = fi.Plan(None)\n"
        "p.plan([0, 4], [0, 2], [5], 16, 8, 2, 128, causal=True)\n"
        "try:\n"
        "    p.plan([0, 4], [0, 2], [5], 16, 8, 3, 128)\n"
        "except fi.FiError:\n"
        "    pass\n")

    def run(level):
        env = dict(os.environ)
        env.pop("FI_LOG", None)
        if level is not None:
            env["FI_LOG"] = str(level)
        r = subprocess.run([sys.executable, "-c", code], cwd=root, env=env, capture_output=True,
                           text=True, timeout=300)
        assert r.returncode == 0, r.stderr
        return [ln for ln in r.stderr.splitlines() if ln.startswith("[fi]")]

    assert run(None) == []
    one = run(1)
    assert len(one) == 1 and "refused" in one[0] and "num_kv_heads=3" in one[0], one
    two = run(2)
    plans = [ln for ln in two if ln.startswith("[fi] plan:")]
    assert len(plans) == 1 and "kernel=" in plans[0] and "items=" in plans[0] \
        and "grid=" in plans[0], two
    assert any("refused" in ln for ln in two)
