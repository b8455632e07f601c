"""merge_state / merge_states against the oracle's merge, the device row bound,
and CUDA-graph capture of a planned run replayed after re-plans."""
import numpy as np
import pytest
import torch

import workloads
from oracle.reference import merge_states as oracle_merge
from tests._util import LSE_TOL, O_TOL, assert_close, run_gpu, workspace

pytestmark = pytest.mark.gpu


def _states(rows, heads, d, seed, dtype=torch.float32, neg_inf_frac=0.1):
    g = torch.Generator().manual_seed(seed)
    v = torch.randn((rows, heads, d), generator=g).to(dtype)
    s = torch.randn((rows, heads), generator=g) * 3
    s[torch.rand((rows, heads), generator=g) < neg_inf_frac] = -float("inf")
    return v, s


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16])
def test_merge_state_matches_oracle(dtype):
    import paged_kv_attention_13_gb300 as fi
    va, sa = _states(37, 5, 128, 1, dtype)
    vb, sb = _states(37, 5, 128, 2, dtype)
    vo, so = fi.fi_merge_state(va.cuda(), sa.cuda(), vb.cuda(), sb.cuda())
    torch.cuda.synchronize()
    v = torch.stack([va, vb], 2).double().reshape(37 * 5, 2, 128).numpy()
    s = torch.stack([sa, sb], 2).double().reshape(37 * 5, 2).numpy()
    v_ref, s_ref = oracle_merge(v, s)
    got_v = vo.float().cpu().reshape(37 * 5, 128).numpy()
    got_s = so.cpu().reshape(-1).numpy()
    tol = 1e-5 if dtype == torch.float32 else O_TOL
    assert np.abs(got_v - v_ref).max() <= tol
    fin = np.isfinite(s_ref)
    assert np.array_equal(np.isfinite(got_s), fin)
    assert np.abs(got_s[fin] - s_ref[fin]).max() <= LSE_TOL


def test_merge_state_in_place_and_row_bound():
    import paged_kv_attention_13_gb300 as fi
    va, sa = _states(16, 4, 64, 3)
    vb, sb = _states(16, 4, 64, 4)
    va_d, sa_d = va.cuda(), sa.cuda()
    bound = torch.tensor([9], dtype=torch.int32, device="cuda")
    fi.fi_merge_state(va_d, sa_d, vb.cuda(), sb.cuda(), v_out=va_d, s_out=sa_d, num_rows_dev=bound)
    torch.cuda.synchronize()
    # rows past the device bound are untouched
    assert torch.equal(va_d[9:].cpu(), va[9:]) and torch.equal(sa_d[9:].cpu(), sa[9:])
    v = torch.stack([va[:9], vb[:9]], 2).double().reshape(36, 2, 64).numpy()
    s = torch.stack([sa[:9], sb[:9]], 2).double().reshape(36, 2).numpy()
    v_ref, _ = oracle_merge(v, s)
    assert np.abs(va_d[:9].cpu().reshape(36, 64).numpy() - v_ref).max() <= 1e-5


def test_merge_states_variable_length():
    import paged_kv_attention_13_gb300 as fi
    counts = [3, 0, 1, 7, 2, 32]
    n = sum(counts)
    v, s = _states(n, 6, 128, 5, neg_inf_frac=0.3)
    indptr = torch.tensor(np.concatenate([[0], np.cumsum(counts)]), dtype=torch.int32)
    vo, so = fi.fi_merge_states(v.cuda(), s.cuda(), indptr.cuda(), len(counts),
                                out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    for r, c in enumerate(counts):
        a, b = int(indptr[r]), int(indptr[r + 1])
        vv = v[a:b].double().permute(1, 0, 2).numpy()       # [H, c, d]
        ss = s[a:b].double().permute(1, 0).numpy()          # [H, c]
        if c == 0:
            v_ref, s_ref = np.zeros((6, 128)), np.full(6, -np.inf)
        else:
            v_ref, s_ref = oracle_merge(vv, ss)
        assert np.abs(vo[r].float().cpu().numpy() - v_ref).max() <= O_TOL
        got = so[r].cpu().numpy()
        fin = np.isfinite(s_ref)
        assert np.array_equal(np.isfinite(got), fin)
        if fin.any():
            assert np.abs(got[fin] - s_ref[fin]).max() <= LSE_TOL


def test_graph_captured_decode_replays_after_replan():
    """Plan once, capture run() in a CUDA graph, re-plan other lengths within
    the capacity, replay: the replay follows the new plan."""
    import paged_kv_attention_13_gb300 as fi
    B, cap_pages = 16, 16 * 300
    ws = workspace()
    plan = fi.Plan(ws, enable_graph_capture=True, max_batch=B, max_total_rows=B)
    pbs = [workloads.batch_decode(variant=v, batch=B, kv_lo=64, kv_hi=4000) for v in range(3)]
    npages = max(pb.k_cache.shape[0] for pb in pbs)
    k = torch.zeros((npages, 16, 8, 128), dtype=torch.bfloat16, device="cuda")
    vv = torch.zeros_like(k)
    q = torch.zeros((B, 32, 128), dtype=torch.bfloat16, device="cuda")
    idx = torch.zeros((cap_pages,), dtype=torch.int32, device="cuda")
    out = torch.zeros((B, 32, 128), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((B, 32), dtype=torch.float32, device="cuda")

    def stage(pb):
        k[: pb.k_cache.shape[0]].copy_(pb.k_cache)
        vv[: pb.v_cache.shape[0]].copy_(pb.v_cache)
        q.copy_(pb.q)
        idx[: pb.kv_indices.shape[0]].copy_(pb.kv_indices)
        plan.plan(None, pb.kv_indptr, pb.last_page_len, 16, 32, 8, 128, q_len_per_req=1)

    stage(pbs[0])
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _ in range(2):  # warm up before capture
            fi.fi_batch_decode_paged(plan, q, k, vv, idx, pbs[0].sm_scale, out=out, lse=lse, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        fi.fi_batch_decode_paged(plan, q, k, vv, idx, pbs[0].sm_scale, out=out, lse=lse)
    for pb in pbs[1:] + pbs[:1]:
        stage(pb)
        out.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert_close(pb, out, lse, False, -1, what="graph replay")
        # the replayed graph read this plan's metadata
        items, merge = plan.read_device()
        assert np.array_equal(items, plan.info(with_arrays=True)["items"])


def test_graph_mode_refuses_frozen_shape_change_and_keeps_plan():
    import paged_kv_attention_13_gb300 as fi
    plan = fi.Plan(workspace(), enable_graph_capture=True, max_batch=8, max_total_rows=32)
    pb = workloads.speculative_verify(batch=8, kv_lo=64, kv_hi=500)
    plan.plan(None, pb.kv_indptr, pb.last_page_len, 16, 32, 8, 128, causal=True, q_len_per_req=4)
    before = plan.info(with_arrays=True)
    with pytest.raises(fi.FiError) as e:
        plan.plan(None, pb.kv_indptr, pb.last_page_len, 16, 32, 8, 128, causal=True,
                  q_len_per_req=2)
    assert e.value.status_name == "FI_ERR_CAPACITY"
    after = plan.info(with_arrays=True)
    assert np.array_equal(before["items"], after["items"])
    out, lse, _ = run_gpu(pb, True, -1, mode="verify", plan=plan, q_len_per_req=4)
    assert_close(pb, out, lse, True, -1)
