"""Paged prefill with a custom (tree) mask against the oracle.

Tree drafts: every request's draft nodes see the prefix and their own
ancestors. Covered: the short-query kernel (at most 16 packed rows), the
mma.sync M = 16 kernel (page size 2), the tcgen05 kernel (more than 32
packed rows) and the mma.sync M = 64 kernel (the same at page size 2),
masks ANDed with causal / window, split-KV, and an all-ones mask equal to
no mask.
"""
import numpy as np
import pytest
import torch

import workloads
from oracle.reference import attention_rows
from tests._util import O_TOL, LSE_TOL, TD, all_rows, sample, workspace

pytestmark = pytest.mark.gpu


def run_masked(pb, causal, wl, force=0, masks=None):
    import paged_kv_attention_13_gb300 as fi
    if masks is None:
        mask, mi = pb.extra["mask"], pb.extra["mask_indptr"]
    else:
        packed, mi = workloads.pack_masks(masks)
        mask, mi = torch.from_numpy(packed), torch.from_numpy(mi)
    plan = fi.Plan(workspace())
    plan.plan_masked(pb.qo_indptr, pb.kv_indptr, pb.last_page_len, pb.page_size,
                     pb.num_qo_heads, pb.num_kv_heads, pb.head_dim, mi, causal=causal,
                     window_left=wl, dtype=TD[pb.dtype], force_kv_chunks=force)
    out, lse = fi.fi_batch_prefill_paged_masked(plan, pb.q.cuda(), pb.k_cache.cuda(),
                                                pb.v_cache.cuda(), pb.kv_indices.cuda(),
                                                mask.cuda(), pb.sm_scale)
    torch.cuda.synchronize()
    assert plan.device_error() == 0
    return out, lse, plan.info()["kernel_name"], mask.numpy(), mi.numpy()


def check(pb, out, lse, causal, wl, mask, mi, toks=None, heads=None, what=""):
    if toks is None:
        toks, heads = all_rows(pb)
    o_ref, l_ref = attention_rows(*pb.oracle_args(), causal, wl, pb.sm_scale, toks, heads,
                                  dtype=pb.dtype, custom_mask=mask, mask_indptr=mi)
    o = out.float().cpu().numpy()[toks, heads]
    l = lse.cpu().numpy()[toks, heads]
    empty = np.isneginf(l_ref)
    assert np.array_equal(np.isneginf(l), empty), what + ": rows with no valid key disagree"
    err_o = float(np.abs(o - o_ref).max())
    err_l = float(np.abs(l[~empty] - l_ref[~empty]).max()) if (~empty).any() else 0.0
    assert err_o <= O_TOL and err_l <= LSE_TOL, "%s: o %.3g lse %.3g" % (what, err_o, err_l)


@pytest.mark.parametrize("causal,wl", [(True, -1), (False, -1), (True, 100)])
@pytest.mark.parametrize("force", [0, 4])
def test_tree_verify_short_kernel(causal, wl, force):
    pb = workloads.tree_verify(batch=6, n_draft=4, kv_lo=40, kv_hi=900)
    out, lse, kern, mask, mi = run_masked(pb, causal, wl, force)
    assert kern == "decode"
    check(pb, out, lse, causal, wl, mask, mi, what="tree short %s %d %d" % (causal, wl, force))


def test_tree_verify_m16_kernel():
    pb = workloads.tree_verify(batch=5, n_draft=4, kv_lo=30, kv_hi=600, page_size=2)
    out, lse, kern, mask, mi = run_masked(pb, True, -1)
    assert kern == "prefill_m16"
    check(pb, out, lse, True, -1, mask, mi, what="tree m16")


@pytest.mark.parametrize("force", [0, 3])
@pytest.mark.parametrize("page_size,kernel", [(16, "prefill_m128"), (2, "prefill_m64")])
def test_tree_verify_wide_trees(force, page_size, kernel):
    """40 draft nodes x GQA 4 = 160 packed rows: the tcgen05 kernel with the
    mask ANDed per element, or the mma.sync M = 64 kernel at page size 2."""
    pb = workloads.tree_verify(batch=4, n_draft=40, kv_lo=60, kv_hi=700, page_size=page_size)
    out, lse, kern, mask, mi = run_masked(pb, True, -1, force)
    assert kern == kernel
    toks, heads = sample(pb, 2000, 9)
    check(pb, out, lse, True, -1, mask, mi, toks, heads, what="tree %s" % kernel)


@pytest.mark.parametrize("causal,wl", [(False, -1), (True, 50), (False, 70)])
def test_random_masks_on_tcgen05(causal, wl):
    """Random bit masks over requests of 40..300 packed rows on the tcgen05
    kernel, every row; includes rows whose mask keeps no key."""
    rng = np.random.default_rng(777 + wl)
    ql = rng.integers(10, 76, size=5)
    kl = ql + rng.integers(0, 400, size=5)
    pb = workloads.make_paged_batch(ql, kl, 8, 2, 128, 16, "bf16", 778 + wl)
    masks = [rng.random((int(a), int(b))) < 0.6 for a, b in zip(ql, kl)]
    masks[0][3, :] = False  # a row with no kept key
    pb.extra["masks"] = masks
    packed, mi = workloads.pack_masks(masks)
    pb.extra["mask"], pb.extra["mask_indptr"] = torch.from_numpy(packed), torch.from_numpy(mi)
    out, lse, kern, mask, mi = run_masked(pb, causal, wl, 0)
    assert kern == "prefill_m128"
    check(pb, out, lse, causal, wl, mask, mi, what="random masks tcgen05")


def test_random_masks_with_empty_rows():
    """Arbitrary (non-tree) masks, some rows masked out entirely."""
    rng = np.random.default_rng(4)
    q_lens, kv_lens = [3, 4, 2], [50, 9, 300]
    masks = [rng.random((q, k)) < 0.3 for q, k in zip(q_lens, kv_lens)]
    masks[0][1, :] = False
    pb = workloads.make_paged_batch(q_lens, kv_lens, 16, 4, 128, 16, "bf16", 77)
    out, lse, kern, mask, mi = run_masked(pb, False, -1, masks=masks)
    check(pb, out, lse, False, -1, mask, mi, what="random masks")


def test_all_ones_mask_equals_no_mask():
    from tests._util import run_gpu
    pb = workloads.tree_verify(batch=4, n_draft=4, kv_lo=40, kv_hi=500)
    ones = [np.ones_like(m) for m in pb.extra["masks"]]
    out, lse, _, _, _ = run_masked(pb, True, -1, masks=ones)
    out0, lse0, _ = run_gpu(pb, True, -1, mode="prefill")
    assert torch.equal(out, out0) and torch.equal(lse, lse0)


@pytest.mark.parametrize("force", [0, 3])
def test_tree_verify_two_row_tiles(force):
    """8 draft nodes at GQA 4 (32 packed rows): two 16-row tiles of the
    short-query kernel per request."""
    pb = workloads.tree_verify(batch=6, n_draft=8, kv_lo=40, kv_hi=900)
    out, lse, kern, mask, mi = run_masked(pb, True, -1, force)
    assert kern == "decode"
    check(pb, out, lse, True, -1, mask, mi, what="tree 2 tiles force=%d" % force)
