"""Ragged prefill over contiguous K/V against the oracle.

The batch is generated as a page-size-1 cache with an unpermuted page table,
so the cache rows are the contiguous K/V in request order: the ragged tensors
are that cache with the page dim dropped, and the oracle reads the paged
view of the same values. Every kernel path is covered: the short-query
kernel (requests of at most 16 packed rows) and the tcgen05 kernel (above 32
packed rows, head_dim 64 and 128).
"""
import pytest
import torch

import workloads
from tests._util import TD, assert_close, sample, workspace

pytestmark = pytest.mark.gpu


def ragged_batch(q_lens, kv_lens, hq, hk, d, dtype, seed):
    return workloads.make_paged_batch(q_lens, kv_lens, hq, hk, d, 1, dtype, seed,
                                      permute_pages=False)


def run_ragged(pb, causal, wl, force=0, kv_view=None):
    import paged_kv_attention_13_gb300 as fi
    rows = pb.k_cache.shape[0]
    k = pb.k_cache.reshape(rows, pb.num_kv_heads, pb.head_dim).cuda()
    v = pb.v_cache.reshape(rows, pb.num_kv_heads, pb.head_dim).cuda()
    if kv_view is not None:
        k, v = kv_view(k), kv_view(v)
    plan = fi.Plan(workspace())
    plan.plan_ragged(pb.qo_indptr, pb.kv_indptr, pb.num_qo_heads, pb.num_kv_heads, pb.head_dim,
                     causal=causal, window_left=wl, dtype=TD[pb.dtype], force_kv_chunks=force)
    out, lse = fi.fi_batch_prefill_ragged(plan, pb.q.cuda(), k, v, pb.sm_scale)
    torch.cuda.synchronize()
    assert plan.device_error() == 0
    return out, lse, plan.info()["kernel_name"]


@pytest.mark.parametrize("causal,wl", [(True, -1), (False, -1), (True, 63), (False, 100), (True, 0)])
@pytest.mark.parametrize("force", [0, 6])
def test_ragged_tensor_core_prefill(causal, wl, force):
    pb = ragged_batch([300, 77, 0, 129, 1], [300, 900, 40, 129, 2000], 16, 4, 128, "bf16", 11)
    out, lse, kern = run_ragged(pb, causal, wl, force)
    assert kern == "prefill_m128"
    toks, heads = sample(pb, 3000, 3)
    assert_close(pb, out, lse, causal, wl, toks, heads, what="ragged tc %s %d %d" % (causal, wl, force))


@pytest.mark.parametrize("causal,wl", [(True, -1), (False, 31)])
def test_ragged_mid_prefill(causal, wl):
    """Requests of 17..64 packed rows, head_dim 64, fp16: above the
    short-query kernel's 32 rows they take the tcgen05 kernel (one half-used
    Q tile per item)."""
    pb = ragged_batch([20, 9, 32], [20, 333, 64], 8, 4, 64, "f16", 12)
    out, lse, kern = run_ragged(pb, causal, wl)
    assert kern == "prefill_m128"
    assert_close(pb, out, lse, causal, wl, what="ragged mid")


@pytest.mark.parametrize("causal,wl", [(True, -1), (False, -1), (True, 9)])
@pytest.mark.parametrize("force", [0, 3])
def test_ragged_short_prefill(causal, wl, force):
    """Requests of at most 16 packed rows run on the short-query kernel."""
    pb = ragged_batch([4, 1, 3, 2, 4], [4, 500, 70, 2, 1300], 32, 8, 128, "bf16", 13)
    out, lse, kern = run_ragged(pb, causal, wl, force)
    assert kern == "decode"
    assert_close(pb, out, lse, causal, wl, what="ragged short")


def test_ragged_strided_rows():
    """K/V as views with a row stride wider than Hk * d (a slice of a wider
    tensor): strides are read as given."""
    pb = ragged_batch([100, 60], [180, 60], 16, 2, 128, "bf16", 14)

    def wide(t):
        w = torch.zeros((t.shape[0], t.shape[1] + 1, t.shape[2]), dtype=t.dtype, device=t.device)
        w[:, 1:] = t
        return w[:, 1:]

    out, lse, kern = run_ragged(pb, True, -1, kv_view=wide)
    assert_close(pb, out, lse, True, -1, what="ragged strided")
