"""The failure path of the bounded waits, made to run on purpose.

Every wait of the TMA kernels on an mbarrier gives up after a limit (2 s by
default). Here the limit is set to 1 ns for one plan, so any wait that does
not succeed at once expires: the kernel must raise its abort flag, stop
issuing work, drain its own copies and tensor-core work (those waits keep the
2 s limit), free its tensor memory, return, and report the expiry in the
workspace. The context must stay usable: a normal run afterwards matches the
oracle ("Refuse attention inputs the ROCm kernels would compute wrongly"
(#399), "Architecture / design notes": fail loudly, never crash). Nothing
here traps, faults or waits without a bound.
"""
import pytest
import torch

import workloads
from tests._util import TD, assert_close, sample, workspace

pytestmark = pytest.mark.gpu


def _prefill(fi, plan, pb, d):
    plan.plan(pb.qo_indptr, pb.kv_indptr, pb.last_page_len, pb.page_size, pb.num_qo_heads,
              pb.num_kv_heads, pb.head_dim, causal=True, dtype=TD[pb.dtype])
    assert plan.info()["kernel_name"] == "prefill_m128"
    return fi.fi_batch_prefill_paged(plan, *d, pb.sm_scale)


def _decode(fi, plan, pb, d):
    plan.plan(None, pb.kv_indptr, pb.last_page_len, pb.page_size, pb.num_qo_heads,
              pb.num_kv_heads, pb.head_dim, dtype=TD[pb.dtype], q_len_per_req=1)
    assert plan.info()["kernel_name"] == "decode"
    return fi.fi_batch_decode_paged(plan, *d, pb.sm_scale)


def _dev(pb):
    return pb.q.cuda(), pb.k_cache.cuda(), pb.v_cache.cuda(), pb.kv_indices.cuda()


@pytest.mark.parametrize("kind", ["prefill_tcgen05", "decode_short_query"])
def test_expired_waits_abort_and_the_context_stays_usable(kind):
    import paged_kv_attention_13_gb300 as fi
    if kind == "prefill_tcgen05":
        pb = workloads.batch_prefill(page_size=16, batch=4)
        run = _prefill
    else:
        pb = workloads.batch_decode(batch=64)
        run = _decode
    d = _dev(pb)
    plan = fi.Plan(workspace(512 << 20))
    # a normal run first (configures the kernel, warms the context)
    out, lse = run(fi, plan, pb, d)
    torch.cuda.synchronize()
    assert plan.device_error() == 0
    # 1 ns: every wait that is not satisfied at once expires
    plan.set_wait_limit(1)
    for _ in range(2):
        out, lse = run(fi, plan, pb, d)  # the call returns
        torch.cuda.synchronize()         # and the launch ends
        assert plan.device_error(clear=True) == 1, "no wait expired under a 1 ns limit"
    # back to the default limit: the same context computes correctly
    plan.set_wait_limit(0)
    out, lse = run(fi, plan, pb, d)
    torch.cuda.synchronize()
    assert plan.device_error() == 0
    toks, heads = sample(pb, 1500, seed=11)
    assert_close(pb, out, lse, True, -1, toks, heads, what=kind + " after an aborted launch")
