"""The tcgen05 prefill kernel's split items against the CPU oracle.

An item of one 128-row Q tile with two or more key tiles runs on both
softmax warpgroups, even key tiles on one and odd tiles on the other, and
the two states are combined by their maxima before the output is written.
These cases cover odd and even tile counts, causal and windowed masks,
direct and split-KV (partial) outputs, and CTAs that mix split items with
two-tile items over many items in a row.
"""
import numpy as np
import pytest

import workloads
from tests._util import assert_close, run_gpu, sample

pytestmark = pytest.mark.gpu

MASKS = [(True, -1), (False, -1), (True, 100), (False, 100)]


@pytest.mark.parametrize("causal,wl", MASKS, ids=lambda v: str(v))
@pytest.mark.parametrize("force", [0, 2])
def test_split_items_every_row(causal, wl, force):
    # packed rows 80, 128, 68 (GQA 4): one Q tile each; 2, 3, 5 and 8 key tiles
    pb = workloads.make_paged_batch([20, 32, 17, 30], [129, 300, 520, 1000], 8, 2, 128, 16,
                                    "bf16", 9100 + force)
    out, lse, plan = run_gpu(pb, causal, wl, force_kv_chunks=force)
    info = plan.info()
    assert info["kernel_name"] == "prefill_m128", info
    assert_close(pb, out, lse, causal, wl, what="split items %s" % info)


@pytest.mark.parametrize("causal,wl", [(True, -1), (False, 300)], ids=lambda v: str(v))
@pytest.mark.parametrize("force", [0, 3])
def test_split_and_pair_items_mixed_sampled(causal, wl, force):
    rng = np.random.default_rng(9200 + force)
    B = 48
    ql = rng.integers(10, 101, size=B)             # 40..400 packed rows: 1 or 2 Q tiles per item
    kl = ql + rng.integers(0, 901, size=B)
    pb = workloads.make_paged_batch(ql, kl, 8, 2, 128, 16, "f16", 9300 + force)
    out, lse, plan = run_gpu(pb, causal, wl, force_kv_chunks=force)
    info = plan.info()
    assert info["kernel_name"] == "prefill_m128", info
    toks, heads = sample(pb, 600, 17 + force)
    assert_close(pb, out, lse, causal, wl, toks, heads, what="mixed items %s" % info)
