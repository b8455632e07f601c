"""plan() and run() on different streams.

The library keeps their order itself: a run() on another stream than the
plan's upload waits for that upload, and a re-plan waits for the plan's
latest run() before it overwrites the workspace. Captured graphs are the
caller's to order ("Support speculative-decode verify on ROCm, and stop auto
routing short-query prefill to AITER" (#362), "Architecture / design notes":
a captured run must not see its buffers change under it).

Each case queues a long device copy in front of one side, so that without
the library's ordering the other side would run first. The device buffers
are sized for both batches of a case (page tables padded with page 0), so a
run that read the other batch's plan would give wrong numbers, never an
access outside its buffers.
"""
import pytest
import torch

import workloads
from tests._util import TD, assert_close, workspace

pytestmark = pytest.mark.gpu


def _busy(stream, mib=512, reps=6):
    """Queue a few hundred microseconds of copies on `stream`."""
    a = torch.empty(mib << 20, dtype=torch.uint8, device="cuda")
    b = torch.empty_like(a)
    with torch.cuda.stream(stream):
        for _ in range(reps):
            b.copy_(a)
    return a, b


def _device(pb, pages, n_idx):
    k = torch.zeros((pages,) + tuple(pb.k_cache.shape[1:]), dtype=pb.k_cache.dtype, device="cuda")
    v = torch.zeros_like(k)
    k[: pb.k_cache.shape[0]].copy_(pb.k_cache)
    v[: pb.v_cache.shape[0]].copy_(pb.v_cache)
    idx = torch.zeros((n_idx,), dtype=torch.int32, device="cuda")
    idx[: pb.kv_indices.shape[0]].copy_(pb.kv_indices)
    return pb.q.cuda(), k, v, idx


def _pair():
    pb0 = workloads.batch_decode(variant=5, batch=16, kv_lo=64, kv_hi=2500)
    pb1 = workloads.batch_decode(variant=6, batch=16, kv_lo=1500, kv_hi=6000)
    pages = max(pb0.k_cache.shape[0], pb1.k_cache.shape[0])
    n_idx = 2 * max(pb0.kv_indices.shape[0], pb1.kv_indices.shape[0])
    return (pb0, _device(pb0, pages, n_idx)), (pb1, _device(pb1, pages, n_idx))


def _plan(plan, pb, stream):
    plan.plan(None, pb.kv_indptr, pb.last_page_len, pb.page_size, pb.num_qo_heads,
              pb.num_kv_heads, pb.head_dim, dtype=TD[pb.dtype], q_len_per_req=1,
              force_kv_chunks=3, stream=stream)


def test_run_on_another_stream_waits_for_the_upload():
    import paged_kv_attention_13_gb300 as fi
    (pb0, d0), (pb1, d1) = _pair()
    A, B = torch.cuda.Stream(), torch.cuda.Stream()
    plan = fi.Plan(workspace())
    _plan(plan, pb0, A)  # the workspace holds a valid plan of another batch
    o, l = fi.fi_batch_decode_paged(plan, *d0, pb0.sm_scale, stream=A)
    torch.cuda.synchronize()
    assert_close(pb0, o, l, False, -1, what="first plan")
    keep = _busy(A)
    _plan(plan, pb1, A)  # its upload sits behind the copies on A
    out, lse = fi.fi_batch_decode_paged(plan, *d1, pb1.sm_scale, stream=B)
    torch.cuda.synchronize()
    del keep
    assert plan.device_error() == 0
    assert_close(pb1, out, lse, False, -1, what="run on B after a plan on A")


def test_replan_waits_for_a_queued_run_on_another_stream():
    import paged_kv_attention_13_gb300 as fi
    (pb0, d0), (pb1, d1) = _pair()
    A, B = torch.cuda.Stream(), torch.cuda.Stream()
    plan = fi.Plan(workspace())
    _plan(plan, pb0, A)
    torch.cuda.synchronize()
    keep = _busy(B)
    out0, lse0 = fi.fi_batch_decode_paged(plan, *d0, pb0.sm_scale, stream=B)  # queued on B
    _plan(plan, pb1, A)  # must not overwrite the workspace before that run
    out1, lse1 = fi.fi_batch_decode_paged(plan, *d1, pb1.sm_scale, stream=A)
    torch.cuda.synchronize()
    del keep
    assert plan.device_error() == 0
    assert_close(pb0, out0, lse0, False, -1, what="queued run on B")
    assert_close(pb1, out1, lse1, False, -1, what="run on A after the re-plan")


def test_runs_of_one_plan_on_two_streams_are_serialised():
    """Two runs of one split-KV plan on two streams share its partial states:
    the second waits for the first."""
    import paged_kv_attention_13_gb300 as fi
    (pb0, d0), _ = _pair()
    A, B = torch.cuda.Stream(), torch.cuda.Stream()
    plan = fi.Plan(workspace())
    _plan(plan, pb0, A)
    keep = _busy(A)
    out_a, lse_a = fi.fi_batch_decode_paged(plan, *d0, pb0.sm_scale, stream=A)
    out_b, lse_b = fi.fi_batch_decode_paged(plan, *d0, pb0.sm_scale, stream=B)
    torch.cuda.synchronize()
    del keep
    assert plan.device_error() == 0
    assert_close(pb0, out_a, lse_a, False, -1, what="run on A")
    assert_close(pb0, out_b, lse_b, False, -1, what="run on B")
