"""K/V cache layouts other than separate NHD tensors, through every kernel.

The kernels take the cache as [pages, page_size, kv_heads, head_dim] element
strides, so the other layouts are views with no copy:
  hnd        a [pages, kv_heads, page_size, head_dim] tensor, permuted;
  fused      one [pages, 2, page_size, kv_heads, head_dim] tensor, K at
             index 0 and V at index 1 of dim 1;
  fused_hnd  one [pages, 2, kv_heads, page_size, head_dim] tensor, permuted.
Each case runs a kernel path (TMA decode, mma.sync verify and short prefill,
tcgen05 prefill) on a layout and is checked against the oracle, which reads
the plain NHD copy of the same values.
"""
import pytest
import torch

import workloads
from tests._util import TD, assert_close, sample, workspace

pytestmark = pytest.mark.gpu

LAYOUTS = ["nhd", "hnd", "fused", "fused_hnd"]


def cache_views(pb, layout):
    """Device (k, v) views of the batch's cache in the given layout."""
    k, v = pb.k_cache, pb.v_cache
    if layout == "nhd":
        return k.cuda(), v.cuda()
    if layout == "hnd":
        return (k.permute(0, 2, 1, 3).contiguous().cuda().permute(0, 2, 1, 3),
                v.permute(0, 2, 1, 3).contiguous().cuda().permute(0, 2, 1, 3))
    if layout == "fused":
        kv = torch.stack([k, v], 1).cuda()
        return kv[:, 0], kv[:, 1]
    if layout == "fused_hnd":
        kv = torch.stack([k.permute(0, 2, 1, 3), v.permute(0, 2, 1, 3)], 1).contiguous().cuda()
        return kv[:, 0].permute(0, 2, 1, 3), kv[:, 1].permute(0, 2, 1, 3)
    raise ValueError(layout)


def run(pb, layout, mode, causal, window_left, q_len_per_req=1):
    import paged_kv_attention_13_gb300 as fi
    k, v = cache_views(pb, layout)
    if layout != "nhd" and pb.page_size > 1:  # with one slot per page HND is NHD
        assert not (k.is_contiguous() and v.is_contiguous())
    plan = fi.Plan(workspace())
    if mode == "prefill":
        plan.plan(pb.qo_indptr, pb.kv_indptr, pb.last_page_len, pb.page_size, pb.num_qo_heads,
                  pb.num_kv_heads, pb.head_dim, causal=causal, window_left=window_left,
                  dtype=TD[pb.dtype])
        f = fi.fi_batch_prefill_paged
    else:
        plan.plan(None, pb.kv_indptr, pb.last_page_len, pb.page_size, pb.num_qo_heads,
                  pb.num_kv_heads, pb.head_dim, causal=causal, window_left=window_left,
                  dtype=TD[pb.dtype], q_len_per_req=q_len_per_req)
        f = fi.fi_batch_decode_paged
    out, lse = f(plan, pb.q.cuda(), k, v, pb.kv_indices.cuda(), pb.sm_scale)
    torch.cuda.synchronize()
    assert plan.device_error() == 0
    return out, lse, plan.info()["kernel_name"]


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("page_size", [16, 1, 64])
def test_decode_layouts(layout, page_size):
    pb = workloads.make_paged_batch([1] * 9, [1, 17, 300, 64, 1000, 5, 129, 700, 33], 16, 4, 128,
                                    page_size, "bf16", 101 + page_size)
    out, lse, kern = run(pb, layout, "decode", False, -1)
    assert kern == "decode"
    assert_close(pb, out, lse, False, -1, what="decode %s P=%d" % (layout, page_size))


@pytest.mark.parametrize("layout", LAYOUTS)
def test_decode_head_dim_64_window(layout):
    pb = workloads.make_paged_batch([1] * 6, [40, 900, 2, 257, 64, 1300], 8, 8, 64, 16, "f16", 77)
    out, lse, kern = run(pb, layout, "decode", True, 100)
    assert kern == "decode"
    assert_close(pb, out, lse, True, 100, what="decode d64 %s" % layout)


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("page_size,kernel", [(16, "decode"), (2, "prefill_m16")])
def test_verify_layouts(layout, page_size, kernel):
    """Verify runs on the short-query TMA kernel where its boxes span whole
    swizzle atoms, else on the cp.async mma kernel."""
    pb = workloads.make_paged_batch([4] * 5, [4, 60, 333, 1024, 9], 32, 8, 128, page_size, "bf16",
                                    55 + page_size)
    out, lse, kern = run(pb, layout, "verify", True, -1, q_len_per_req=4)
    assert kern == kernel
    assert_close(pb, out, lse, True, -1, what="verify %s P=%d" % (layout, page_size))


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("page_size,kernel", [(16, "prefill_m128"), (2, "prefill_m64")])
def test_short_prefill_layouts(layout, page_size, kernel):
    """14..62 packed rows: the tcgen05 kernel (one half-used Q tile) where its
    boxes fit, the cp.async mma kernel for page sizes under 8."""
    pb = workloads.make_paged_batch([20, 7, 31], [20, 300, 64], 8, 4, 64, page_size, "bf16",
                                    56 + page_size)
    out, lse, kern = run(pb, layout, "prefill", True, 31)
    assert kern == kernel
    assert_close(pb, out, lse, True, 31, what="short prefill %s P=%d" % (layout, page_size))


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("page_size", [16, 128])
def test_tensor_core_prefill_layouts(layout, page_size):
    pb = workloads.make_paged_batch([300, 70, 129], [300, 700, 200], 16, 4, 128, page_size,
                                    "bf16", 57 + page_size)
    out, lse, kern = run(pb, layout, "prefill", True, -1)
    assert kern == "prefill_m128"
    toks, heads = sample(pb, 3000, 5)
    assert_close(pb, out, lse, True, -1, toks, heads, what="tc prefill %s P=%d" % (layout,
                                                                                   page_size))
