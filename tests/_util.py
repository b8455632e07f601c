"""Shared test helpers: run the CUDA path through the C ABI, run the oracle on
the same seeded inputs, compare within the stated tolerances.

Tolerances (fixed for floating outputs): max |o - o_ref| <= 2e-2 on the
bf16/fp16 output and max |lse - lse_ref| <= 1e-3 on the fp32 natural-log LSE.
Integer plan metadata is compared exactly.
"""
import numpy as np
import torch

import workloads
from oracle.reference import attention_rows

O_TOL = 2e-2
LSE_TOL = 1e-3

TD = {"bf16": torch.bfloat16, "f16": torch.float16}


def to_dev(pb, dev="cuda"):
    return (pb.q.to(dev), pb.k_cache.to(dev), pb.v_cache.to(dev), pb.kv_indices.to(dev))


def workspace(nbytes=256 << 20, dev="cuda"):
    return torch.empty(nbytes, dtype=torch.uint8, device=dev)


def run_gpu(pb, causal, window_left, mode="prefill", force_kv_chunks=0, ws=None, plan=None,
            q_len_per_req=None):
    """Plan + run one batch on the GPU; returns (out, lse, plan)."""
    import paged_kv_attention_13_gb300 as fi
    if ws is None:
        ws = workspace()
    if plan is None:
        plan = fi.Plan(ws)
    q, k, v, idx = to_dev(pb)
    if mode == "prefill":
        plan.plan(pb.qo_indptr, pb.kv_indptr, pb.last_page_len, pb.page_size, pb.num_qo_heads,
                  pb.num_kv_heads, pb.head_dim, causal=causal, window_left=window_left,
                  dtype=TD[pb.dtype], force_kv_chunks=force_kv_chunks)
        out, lse = fi.fi_batch_prefill_paged(plan, q, k, v, idx, pb.sm_scale)
    else:
        qlpr = q_len_per_req or (1 if mode == "decode" else pb.extra.get("q_len_per_req", 4))
        plan.plan(None, pb.kv_indptr, pb.last_page_len, pb.page_size, pb.num_qo_heads,
                  pb.num_kv_heads, pb.head_dim, causal=causal, window_left=window_left,
                  dtype=TD[pb.dtype], q_len_per_req=qlpr, force_kv_chunks=force_kv_chunks)
        out, lse = fi.fi_batch_decode_paged(plan, q, k, v, idx, pb.sm_scale)
    torch.cuda.synchronize()
    assert plan.device_error() == 0, "a kernel gave up an expired bounded wait"
    return out, lse, plan


def oracle_rows(pb, causal, window_left, toks, heads):
    return attention_rows(*pb.oracle_args(), causal, window_left, pb.sm_scale, toks, heads,
                          dtype=pb.dtype)


def all_rows(pb):
    T = int(pb.qo_indptr[-1])
    H = pb.num_qo_heads
    return (np.repeat(np.arange(T, dtype=np.int64), H), np.tile(np.arange(H, dtype=np.int32), T))


def compare(pb, out, lse, causal, window_left, toks=None, heads=None):
    """Max errors of (out, lse) against the oracle on the given rows (default all)."""
    if toks is None:
        toks, heads = all_rows(pb)
    if len(toks) == 0:
        return 0.0, 0.0
    o_ref, l_ref = oracle_rows(pb, causal, window_left, toks, heads)
    o = out.float().cpu().numpy()[toks, heads]
    l = lse.cpu().numpy()[toks, heads]
    # rows with no valid key: o = 0 and lse = -inf on both sides
    empty = np.isneginf(l_ref)
    assert np.array_equal(np.isneginf(l), empty), "rows with no valid key disagree"
    assert np.all(np.isfinite(o)), "non-finite output"
    err_o = float(np.abs(o - o_ref).max())
    err_l = float(np.abs(l[~empty] - l_ref[~empty]).max()) if (~empty).any() else 0.0
    return err_o, err_l


def assert_close(pb, out, lse, causal, window_left, toks=None, heads=None, what=""):
    err_o, err_l = compare(pb, out, lse, causal, window_left, toks, heads)
    assert err_o <= O_TOL and err_l <= LSE_TOL, "%s: max|o err|=%.3g max|lse err|=%.3g" % (
        what, err_o, err_l)
    return err_o, err_l


def sample(pb, n, seed):
    return workloads.sample_rows(pb, n, seed)
