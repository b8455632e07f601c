"""Shapes that now take the tcgen05 prefill kernel instead of the mma.sync one,
checked against the CPU oracle.

- head_dim 64 (the kernel is built for 64 and 128);
- page sizes that do not divide 128, or that are not multiples of 128 above
  it: K/V boxes of gcd(page size, 128) slots, each inside one page;
- requests of 33..64 packed rows (one half-used 128-row Q tile).

The paged prefill of "Route non-causal windowed prefill to AITER's masked
kernel" (#339), "Test plan", runs both small and large pages; "Support
speculative-decode verify on ROCm, and stop auto routing short-query prefill
to AITER" (#362), "Architecture / design notes", gives the tile rule over
every query length and head dim.
"""
import numpy as np
import pytest

import workloads
from tests._util import assert_close, run_gpu, sample

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("causal,wl", [(True, -1), (False, -1), (True, 127), (False, 127)],
                         ids=lambda v: str(v))
def test_hd64_fp16_batch_prefill_full_size(causal, wl):
    # the batch-16 prefill lengths (qo_len U[512, 2048], prefix U[0, 4096]),
    # 4 q / 2 kv heads, head_dim 64, fp16, page 16
    pb = workloads.batch_prefill_hd64()
    out, lse, plan = run_gpu(pb, causal, wl)
    assert plan.info()["kernel_name"] == "prefill_m128", plan.info()
    toks, heads = sample(pb, 2500, seed=64 + (1 if causal else 0) + (2 if wl >= 0 else 0))
    assert_close(pb, out, lse, causal, wl, toks, heads, what="hd64 fp16 prefill")


@pytest.mark.parametrize("page_size", [8, 24, 48, 96, 200])
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_page_sizes_off_128_every_row(page_size, dtype):
    rng = np.random.default_rng(4800 + page_size)
    ql = rng.integers(20, 90, size=6)
    kl = ql + rng.integers(0, 700, size=6)
    pb = workloads.make_paged_batch(ql, kl, 8, 2, 128, page_size, dtype, 4900 + page_size)
    for causal, wl, force in ((True, -1, 0), (False, 60, 0), (True, 200, 3)):
        out, lse, plan = run_gpu(pb, causal, wl, force_kv_chunks=force)
        assert plan.info()["kernel_name"] == "prefill_m128", plan.info()
        assert_close(pb, out, lse, causal, wl,
                     what="page %d %s causal=%s wl=%d" % (page_size, dtype, causal, wl))


def test_page_48_batch_prefill_sampled():
    pb = workloads.batch_prefill(page_size=48, batch=6)
    out, lse, plan = run_gpu(pb, True, -1)
    assert plan.info()["kernel_name"] == "prefill_m128", plan.info()
    toks, heads = sample(pb, 1500, seed=48)
    assert_close(pb, out, lse, True, -1, toks, heads, what="page 48 prefill")


@pytest.mark.parametrize("head_dim", [64, 128])
def test_33_to_64_packed_rows_on_tcgen05(head_dim):
    # 9..16 query rows x GQA 4 = 36..64 packed rows per request
    rng = np.random.default_rng(3364 + head_dim)
    ql = rng.integers(9, 17, size=10)
    kl = ql + rng.integers(0, 900, size=10)
    pb = workloads.make_paged_batch(ql, kl, 8, 2, head_dim, 16, "bf16", 3365 + head_dim)
    for causal, wl in ((True, -1), (False, 100)):
        out, lse, plan = run_gpu(pb, causal, wl)
        assert plan.info()["kernel_name"] == "prefill_m128", plan.info()
        assert_close(pb, out, lse, causal, wl, what="33-64 rows d%d" % head_dim)


@pytest.mark.parametrize("seed", range(4))
def test_hd64_random_batches(seed):
    rng = np.random.default_rng(6400 + seed)
    B = int(rng.integers(1, 9))
    ql = rng.integers(1, 200, size=B)
    causal = bool(seed & 1)
    kl = ql + rng.integers(0, 500, size=B) if causal else rng.integers(0, 600, size=B)
    g = int(rng.choice([1, 2, 4, 8]))
    pb = workloads.make_paged_batch(ql, kl, 2 * g, 2, 64, int(rng.choice([16, 32, 64])),
                                    "f16" if seed & 2 else "bf16", 6500 + seed)
    wl = int(rng.choice([-1, 0, 30, 200]))
    out, lse, plan = run_gpu(pb, causal, wl, force_kv_chunks=int(rng.choice([0, 2])))
    assert_close(pb, out, lse, causal, wl, what="hd64 random %d %s" % (seed, plan.info()))
