"""CUDA path vs the CPU oracle, element by element, through the C ABI.

Small cases are compared on every row (several tiles, ragged tails, empty
requests); the full-size workloads on seeded samples of rows, in the launch
configuration the benchmark times.
"""
import numpy as np
import pytest
import torch

import workloads
from tests._util import (LSE_TOL, O_TOL, all_rows, assert_close, compare, run_gpu, sample,
                         workspace)

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("case", workloads.PR1_CASES, ids=lambda c: "causal%d_wl%d" % (c["causal"], c["window_left"]))
def test_pr1_reference_every_row(case):
    pb = workloads.pr1_reference()
    out, lse, _ = run_gpu(pb, case["causal"], case["window_left"])
    assert_close(pb, out, lse, case["causal"], case["window_left"], what=str(case))


def test_pr1_window_changes_the_gpu_answer():
    """Anti-vacuity: the windowed and unwindowed results differ by > 0.1."""
    pb = workloads.pr1_reference()
    for causal in (True, False):
        o1, _, _ = run_gpu(pb, causal, -1)
        o2, _, _ = run_gpu(pb, causal, 31)
        assert (o1.float() - o2.float()).abs().max().item() > 0.1


def _random_batch(seed, decode=False):
    rng = np.random.default_rng(seed)
    B = int(rng.integers(1, 6))
    g = int(rng.choice([1, 2, 3, 4, 8]))
    Hk = int(rng.integers(1, 3))
    d = int(rng.choice([64, 128]))
    P = int(rng.choice([1, 3, 16, 64]))
    dtype = str(rng.choice(["bf16", "f16"]))
    causal = bool(rng.integers(0, 2)) or decode
    wl = int(rng.choice([-1, -1, 0, 5, 40, 300]))
    ql, kl = [], []
    for _ in range(B):
        lk = int(rng.integers(0, 400))
        if decode:
            lq = 1
            lk = max(lk, 1)
        else:
            lq = int(rng.integers(0, 90))
            if causal:
                lq = min(lq, lk)
        ql.append(lq)
        kl.append(lk)
    pb = workloads.make_paged_batch(ql, kl, g * Hk, Hk, d, P, dtype, 5000 + seed,
                                    extra_pool_pages=3)
    return pb, causal, wl


@pytest.mark.parametrize("seed", range(24))
@pytest.mark.parametrize("force", [0, 3])
def test_random_ragged_prefill_every_row(seed, force):
    pb, causal, wl = _random_batch(seed)
    out, lse, plan = run_gpu(pb, causal, wl, force_kv_chunks=force)
    assert_close(pb, out, lse, causal, wl, what="seed %d %s" % (seed, plan.info()))


@pytest.mark.parametrize("seed", range(16))
@pytest.mark.parametrize("force", [0, 4])
def test_random_decode_every_row(seed, force):
    pb, causal, wl = _random_batch(100 + seed, decode=True)
    out, lse, plan = run_gpu(pb, causal, wl, mode="decode", force_kv_chunks=force)
    assert_close(pb, out, lse, causal, wl, what="seed %d %s" % (seed, plan.info()))


def test_decode_full_size_sampled():
    """Batch 64, kv in [512, 8192], 32/8 heads, d 128, bf16, page 16 (the
    benchmarked decode launch), sampled rows."""
    pb = workloads.batch_decode()
    out, lse, plan = run_gpu(pb, False, -1, mode="decode")
    info = plan.info()
    assert info["kernel_name"] == "decode"
    toks, heads = all_rows(pb)  # 64 x 32 rows: cheap enough for every row
    assert_close(pb, out, lse, False, -1, toks, heads, what="decode full")


@pytest.mark.parametrize("batch", [4, 32])
def test_verify_matches_oracle_and_causal_prefill(batch):
    pb = workloads.speculative_verify(batch=batch)
    out, lse, plan = run_gpu(pb, True, -1, mode="verify", q_len_per_req=4)
    toks, heads = all_rows(pb) if batch == 4 else sample(pb, 400, 7)
    assert_close(pb, out, lse, True, -1, toks, heads, what="verify B=%d" % batch)
    # verify == causal paged prefill over qo_indptr = 4 i
    out2, lse2, _ = run_gpu(pb, True, -1, mode="prefill")
    assert torch.equal(out, out2)
    assert torch.equal(lse, lse2)


@pytest.mark.parametrize("page_size", [16, 1024])
@pytest.mark.parametrize("case", workloads.PREFILL_CASES, ids=lambda c: "causal%d_wl%d" % (c["causal"], c["window_left"]))
def test_batch_prefill_full_size_sampled(page_size, case):
    pb = workloads.batch_prefill(page_size=page_size)
    out, lse, _ = run_gpu(pb, case["causal"], case["window_left"])
    toks, heads = sample(pb, 160, 11 + page_size)
    assert_close(pb, out, lse, case["causal"], case["window_left"], toks, heads,
                 what="prefill P=%d %s" % (page_size, case))


@pytest.mark.parametrize("chunks", workloads.LONG_CONTEXT_CHUNKS)
@pytest.mark.parametrize("case", workloads.LONG_CONTEXT_CASES, ids=lambda c: "causal%d_wl%d" % (c["causal"], c["window_left"]))
def test_long_context_split_kv_sampled(chunks, case):
    pb = workloads.long_context()
    out, lse, plan = run_gpu(pb, case["causal"], case["window_left"], force_kv_chunks=chunks)
    info = plan.info()
    assert info["max_chunks"] == chunks and info["num_merge_rows"] == int(pb.qo_indptr[-1])
    toks, heads = sample(pb, 96, 13 + chunks)
    assert_close(pb, out, lse, case["causal"], case["window_left"], toks, heads,
                 what="long ctx chunks=%d %s" % (chunks, case))
    # split + merge == the planner's own split (or none): same rows within tolerance
    out2, lse2, _ = run_gpu(pb, case["causal"], case["window_left"])
    assert (out.float() - out2.float()).abs().max().item() <= O_TOL
    assert (lse - lse2).abs().max().item() <= LSE_TOL


def test_page_sizes_agree():
    """Page 1, 16 and 1024 give the same answer (same keys, different pages)."""
    res = []
    for P in (1, 16, 1024):
        pb = workloads.make_paged_batch([37, 5], [300, 5], 8, 2, 128, P, "bf16", 42,
                                        permute_pages=(P != 1024))
        res.append(run_gpu(pb, True, 50)[:2])
        assert_close(pb, *res[-1], True, 50, what="P=%d" % P)


def test_rows_past_planned_total_are_untouched():
    pb = workloads.make_paged_batch([20, 9], [40, 30], 8, 2, 128, 16, "bf16", 3)
    import paged_kv_attention_13_gb300 as fi
    ws = workspace()
    plan = fi.Plan(ws)
    plan.plan(pb.qo_indptr, pb.kv_indptr, pb.last_page_len, 16, 8, 2, 128, causal=True)
    T = int(pb.qo_indptr[-1])
    q = torch.zeros((T + 7, 8, 128), dtype=torch.bfloat16, device="cuda")
    q[:T] = pb.q.cuda()
    out = torch.full((T + 7, 8, 128), 7.0, dtype=torch.bfloat16, device="cuda")
    lse = torch.full((T + 7, 8), 7.0, dtype=torch.float32, device="cuda")
    fi.fi_batch_prefill_paged(plan, q, pb.k_cache.cuda(), pb.v_cache.cuda(), pb.kv_indices.cuda(),
                              pb.sm_scale, out=out, lse=lse)
    torch.cuda.synchronize()
    assert torch.all(out[T:] == 7.0) and torch.all(lse[T:] == 7.0)
    assert_close(pb, out[:T], lse[:T], True, -1)


def test_strided_token_and_head_strides_are_honoured():
    """q taken as a head slice of a wider tensor, caches as views with padded
    pages: strides other than the last dim are read as given."""
    pb = workloads.make_paged_batch([33, 4], [100, 50], 8, 2, 128, 16, "bf16", 4)
    import paged_kv_attention_13_gb300 as fi
    T = int(pb.qo_indptr[-1])
    qbig = torch.zeros((T, 12, 128), dtype=torch.bfloat16, device="cuda")
    qbig[:, 2:10] = pb.q.cuda()
    q = qbig[:, 2:10]
    n = pb.k_cache.shape[0]
    kbig = torch.zeros((n, 16, 3, 128), dtype=torch.bfloat16, device="cuda")
    vbig = torch.zeros((n, 16, 3, 128), dtype=torch.bfloat16, device="cuda")
    kbig[:, :, :2] = pb.k_cache.cuda()
    vbig[:, :, :2] = pb.v_cache.cuda()
    plan = fi.Plan(workspace())
    plan.plan(pb.qo_indptr, pb.kv_indptr, pb.last_page_len, 16, 8, 2, 128, causal=True)
    out, lse = fi.fi_batch_prefill_paged(plan, q, kbig[:, :, :2], vbig[:, :, :2],
                                         pb.kv_indices.cuda(), pb.sm_scale)
    torch.cuda.synchronize()
    assert_close(pb, out, lse, True, -1)


def test_device_metadata_equals_host_plan():
    pb = workloads.batch_decode(batch=16, kv_lo=100, kv_hi=5000)
    import paged_kv_attention_13_gb300 as fi
    plan = fi.Plan(workspace())
    plan.plan(None, pb.kv_indptr, pb.last_page_len, 16, 32, 8, 128, q_len_per_req=1,
              force_kv_chunks=5)
    host = plan.info(with_arrays=True)
    items, merge = plan.read_device()
    assert np.array_equal(items, host["items"])
    assert np.array_equal(merge, host["merge_indptr"])
