"""The decode entry point that allocates nothing.

Some callers cannot allocate device memory at the moment they run attention:
a serving loop that reserved all GPU memory for its own pool up front, code
running inside another framework's allocator, or a host path where a
cudaMalloc/cudaFree would synchronise the device. For them
fi_batch_decode_paged_noalloc keeps its split-KV scratch in a fixed device
array inside libfi. This file checks it against the regular planned decode
(fi_plan + fi_batch_decode_paged) on two calls in a row that share that
array. It is collected last so a failure here never hides another test.
"""
import numpy as np
import pytest
import torch

import workloads
from tests._util import LSE_TOL, O_TOL, workspace

pytestmark = pytest.mark.gpu


def _planned(pb, chunks):
    import paged_kv_attention_13_gb300 as fi
    plan = fi.Plan(workspace())
    plan.plan(None, pb.kv_indptr, pb.last_page_len, pb.page_size, pb.num_qo_heads,
              pb.num_kv_heads, pb.head_dim, dtype=workloads.TORCH_DTYPE[pb.dtype], q_len_per_req=1,
              force_kv_chunks=chunks)
    out, lse = fi.fi_batch_decode_paged(plan, pb.q.cuda(), pb.k_cache.cuda(), pb.v_cache.cuda(),
                                        pb.kv_indices.cuda(), pb.sm_scale)
    torch.cuda.synchronize()
    return out, lse


def _noalloc(pb, chunks):
    import paged_kv_attention_13_gb300 as fi
    out, lse = fi.fi_batch_decode_paged_noalloc(
        pb.q.cuda(), pb.k_cache.cuda(), pb.v_cache.cuda(), pb.kv_indices.cuda(),
        pb.kv_indptr.cuda(), pb.last_page_len.cuda(), pb.sm_scale, kv_chunks=chunks)
    torch.cuda.synchronize()
    return out, lse


def test_noalloc_decode_matches_planned_decode_twice_in_a_row():
    # two different batches through the shared scratch, back to back
    cases = [(workloads.batch_decode(batch=24, kv_lo=64, kv_hi=3000), 4),
             (workloads.batch_decode(variant=1, batch=9, kv_lo=1, kv_hi=5000, num_qo_heads=16,
                                     num_kv_heads=8), 7)]
    for pb, chunks in cases:
        ref_o, ref_l = _planned(pb, chunks)
        got_o, got_l = _noalloc(pb, chunks)
        assert (got_o.float() - ref_o.float()).abs().max().item() <= O_TOL
        fin = torch.isfinite(ref_l)
        assert torch.equal(torch.isfinite(got_l), fin)
        assert (got_l[fin] - ref_l[fin]).abs().max().item() <= LSE_TOL


def test_noalloc_refuses_more_than_its_scratch():
    import paged_kv_attention_13_gb300 as fi
    pb = workloads.batch_decode(batch=512, kv_lo=16, kv_hi=32)
    with pytest.raises(fi.FiError) as e:
        _noalloc(pb, 64)
    assert e.value.status_name == "FI_ERR_CAPACITY" and "scratch" in str(e.value)
