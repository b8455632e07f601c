"""The opt-in page-table check (fi_check_kv_indices, FI_CHECK_INDICES).

A page index outside the cache turns into a memory fault in the kernels that
gather pages ("Support speculative-decode verify on ROCm, and stop auto
routing short-query prefill to AITER" (#362), "Review notes"). The check
counts such entries on the device and never traps. It is tested by itself on
tables with bad entries; no attention kernel is ever launched on such a table.
With FI_CHECK_INDICES=1 every paged run() checks first: a normal run on a
valid table must still match the oracle.
"""
import os
import subprocess
import sys

import pytest
import torch

import workloads
from tests._util import TD, workspace

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_check_kernel_counts_bad_entries_and_passes_a_valid_table():
    import paged_kv_attention_13_gb300 as fi
    pb = workloads.batch_decode(batch=12, kv_lo=100, kv_hi=3000)
    plan = fi.Plan(workspace())
    plan.plan(None, pb.kv_indptr, pb.last_page_len, pb.page_size, pb.num_qo_heads,
              pb.num_kv_heads, pb.head_dim, dtype=TD[pb.dtype], q_len_per_req=1)
    npages = int(pb.k_cache.shape[0])
    good = pb.kv_indices.cuda()
    plan.check_kv_indices(good, npages)
    assert plan.device_error() == 0
    for pos, val in ((0, npages), (len(good) // 2, -1), (len(good) - 1, 1 << 30)):
        bad = good.clone()
        bad[pos] = val
        plan.check_kv_indices(bad, npages)
        assert plan.device_error() == 2, (pos, val)
    # one page fewer in the cache than the table uses: the largest entry fails
    plan.check_kv_indices(good, int(good.max().item()))
    assert plan.device_error(clear=True) == 2
    # entries past kv_indptr[batch] are not the plan's: not checked
    longer = torch.cat([good, torch.full((7,), -5, dtype=torch.int32, device="cuda")])
    plan.check_kv_indices(longer, npages)
    assert plan.device_error() == 0


def test_runs_with_the_check_enabled_match_the_oracle():
    code = r"""
import torch, workloads
import paged_kv_attention_13_gb300 as fi
from tests._util import TD, assert_close, sample, workspace, run_gpu
torch.cuda.set_device(0)
pb = workloads.batch_decode(batch=24, kv_lo=64, kv_hi=4000)
out, lse, plan = run_gpu(pb, False, -1, mode="decode", force_kv_chunks=3)
assert plan.device_error() == 0
assert_close(pb, out, lse, False, -1, what="decode with the index check")
pb = workloads.batch_prefill(page_size=16, batch=3)
out, lse, plan = run_gpu(pb, True, -1)
assert plan.info()["kernel_name"] == "prefill_m128"
assert plan.device_error() == 0
toks, heads = sample(pb, 800, seed=5)
assert_close(pb, out, lse, True, -1, toks, heads, what="prefill with the index check")
pb = workloads.pr1_reference()
out, lse, plan = run_gpu(pb, True, 31)
assert plan.device_error() == 0
assert_close(pb, out, lse, True, 31, what="mma.sync prefill with the index check")
print("index-check runs ok")
"""
    env = dict(os.environ)
    env["FI_CHECK_INDICES"] = "1"
    env["FI_LOG"] = "3"
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert "index-check runs ok" in r.stdout
    # the run log shows that every run went through the check
    runs = [ln for ln in r.stderr.splitlines() if ln.startswith("[fi] batch_")]
    assert runs and all("index-check" in ln for ln in runs), r.stderr[-2000:]
