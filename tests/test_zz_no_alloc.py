"""The decode entry point that allocates nothing.

Some callers cannot allocate device memory at the moment they run attention:
a serving loop that reserved all GPU memory for its own pool up front, code
running inside another framework's allocator, or a host path where a
cudaMalloc/cudaFree would synchronise the device. For them
fi_batch_decode_paged_noalloc keeps its split-KV scratch in a fixed device
array inside libfi. This file checks it against the oracle and against the
regular planned decode (fi_plan + fi_batch_decode_paged), on calls in a row
that share that array, and reads its error flag after each call. It is
collected last so a failure here never hides another test.
"""
import pytest
import torch

import workloads
from tests._util import LSE_TOL, O_TOL, assert_close, workspace

pytestmark = pytest.mark.gpu


def _planned(pb, chunks, window_left):
    import paged_kv_attention_13_gb300 as fi
    plan = fi.Plan(workspace())
    plan.plan(None, pb.kv_indptr, pb.last_page_len, pb.page_size, pb.num_qo_heads,
              pb.num_kv_heads, pb.head_dim, window_left=window_left,
              dtype=workloads.TORCH_DTYPE[pb.dtype], q_len_per_req=1, force_kv_chunks=chunks)
    out, lse = fi.fi_batch_decode_paged(plan, pb.q.cuda(), pb.k_cache.cuda(), pb.v_cache.cuda(),
                                        pb.kv_indices.cuda(), pb.sm_scale)
    torch.cuda.synchronize()
    assert plan.device_error() == 0
    return out, lse


def _noalloc(pb, chunks, window_left=-1, with_lse=True):
    import paged_kv_attention_13_gb300 as fi
    out, lse = fi.fi_batch_decode_paged_noalloc(
        pb.q.cuda(), pb.k_cache.cuda(), pb.v_cache.cuda(), pb.kv_indices.cuda(),
        pb.kv_indptr.cuda(), pb.last_page_len.cuda(), pb.sm_scale, window_left=window_left,
        kv_chunks=chunks, return_lse=with_lse)
    torch.cuda.synchronize()
    assert fi.fi_noalloc_device_error() == 0, "a bounded wait of the no-allocation decode expired"
    return out, lse


def _cases():
    # (batch, chunks, window_left, with lse, what it covers)
    zero = workloads.make_paged_batch([1] * 6, [700, 0, 1, 4999, 128, 2500], 16, 8, 128, 16,
                                      "f16", 9001)
    return [
        (workloads.batch_decode(batch=24, kv_lo=64, kv_hi=3000), 4, -1, True,
         "bf16, GQA 4, page 16"),
        (zero, 7, 127, True,
         "fp16, GQA 2, window 127 (most chunks outside the window), a request with no page"),
        (workloads.batch_decode(variant=1, batch=10, kv_lo=1, kv_hi=2000, num_qo_heads=8,
                                num_kv_heads=8, head_dim=64, page_size=4), 1, -1, False,
         "GQA 1 on page 4 (the CUDA-core consumer), head_dim 64, one chunk, no lse"),
        (workloads.batch_decode(variant=2, batch=9, kv_lo=300, kv_hi=5000, head_dim=64,
                                dtype="f16"), 64, 40, True,
         "fp16, head_dim 64, 64 chunks, window 40"),
    ]


def test_noalloc_decode_matches_the_oracle_and_the_planned_decode_in_a_row():
    # the cases run back to back through the one shared scratch array
    for pb, chunks, wl, with_lse, what in _cases():
        got_o, got_l = _noalloc(pb, chunks, wl, with_lse)
        if with_lse:
            assert_close(pb, got_o, got_l, False, wl, what="no-allocation decode: " + what)
        else:
            assert got_l is None
            ref_o, ref_l = _planned(pb, 0, wl)  # lse of the planned run for the comparison
            assert_close(pb, got_o, ref_l, False, wl, what="no-allocation decode: " + what)
        ref_o, ref_l = _planned(pb, chunks, wl)
        assert (got_o.float() - ref_o.float()).abs().max().item() <= O_TOL, what
        if with_lse:
            fin = torch.isfinite(ref_l)
            assert torch.equal(torch.isfinite(got_l), fin), what
            assert (got_l[fin] - ref_l[fin]).abs().max().item() <= LSE_TOL, what


def test_noalloc_decode_twice_in_a_row_gives_the_same_result():
    pb, chunks, wl, _, _ = _cases()[0]
    a_o, a_l = _noalloc(pb, chunks, wl)
    b_o, b_l = _noalloc(pb, chunks, wl)
    assert torch.equal(a_o, b_o) and torch.equal(a_l, b_l)


def test_noalloc_refuses_more_than_its_scratch():
    import paged_kv_attention_13_gb300 as fi
    pb = workloads.batch_decode(batch=512, kv_lo=16, kv_hi=32)
    with pytest.raises(fi.FiError) as e:
        _noalloc(pb, 64)
    assert e.value.status_name == "FI_ERR_CAPACITY" and "scratch" in str(e.value)
