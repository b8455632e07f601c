"""The short-query kernel (every request of at most 32 packed rows) against
the oracle: GQA groups 1..16, decode, verify, ragged short prefill, the
32-row pair consumer, split-KV with several query rows per work item, and
run-to-run determinism.
"""
import numpy as np
import pytest
import torch

import workloads
from tests._util import assert_close, run_gpu

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("hq,hk", [(16, 2), (32, 2), (8, 8), (16, 8), (64, 4)])
@pytest.mark.parametrize("force", [0, 5])
def test_decode_groups(hq, hk, force):
    """Groups 8 and 16 (one and two fragment row halves) and 1, 2, 4."""
    lens = [1, 9, 64, 130, 511, 2000, 77]
    pb = workloads.make_paged_batch([1] * len(lens), lens, hq, hk, 128, 16, "bf16", 900 + hq + hk)
    out, lse, plan = run_gpu(pb, False, -1, mode="decode", force_kv_chunks=force)
    assert plan.info()["kernel_name"] == "decode"
    assert_close(pb, out, lse, False, -1, what="decode g=%d force=%d" % (hq // hk, force))


@pytest.mark.parametrize("hq,hk,qlen", [(8, 4, 4), (32, 8, 4), (16, 2, 2), (16, 16, 16), (4, 4, 3)])
@pytest.mark.parametrize("window_left", [-1, 5])
@pytest.mark.parametrize("force", [0, 4])
def test_verify_rows(hq, hk, qlen, window_left, force):
    """Verify: qlen draft rows per request, causal, with and without a
    window, with the key range split so several query rows share a chunk."""
    kv = [qlen, qlen + 3, 97, 700, 1500]
    pb = workloads.make_paged_batch([qlen] * len(kv), kv, hq, hk, 128, 16, "bf16", 40 + qlen + hq)
    out, lse, plan = run_gpu(pb, True, window_left, mode="verify", force_kv_chunks=force,
                             q_len_per_req=qlen)
    assert plan.info()["kernel_name"] == "decode"
    assert_close(pb, out, lse, True, window_left,
                 what="verify g=%d q=%d wl=%d force=%d" % (hq // hk, qlen, window_left, force))


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("window_left", [-1, 0, 40])
@pytest.mark.parametrize("head_dim,dtype", [(128, "bf16"), (64, "f16")])
def test_ragged_short_prefill(causal, window_left, head_dim, dtype):
    """Prefill whose requests all fit 16 packed rows (g = 4: up to 4 query
    rows) with ragged query and key lengths, including an empty request."""
    q_lens = [1, 4, 2, 3, 0, 4]
    kv_lens = [1, 4, 300, 33, 10, 2049]
    pb = workloads.make_paged_batch(q_lens, kv_lens, 16, 4, head_dim, 16, dtype, 71 + head_dim)
    out, lse, plan = run_gpu(pb, causal, window_left, mode="prefill")
    assert plan.info()["kernel_name"] == "decode"
    assert_close(pb, out, lse, causal, window_left,
                 what="short prefill causal=%s wl=%d d=%d" % (causal, window_left, head_dim))


def test_runs_are_bitwise_reproducible():
    """The cross-warp merge adds in a fixed order: two runs agree bit for bit."""
    pb = workloads.speculative_verify(batch=8)
    a = run_gpu(pb, True, -1, mode="verify", q_len_per_req=4)
    b = run_gpu(pb, True, -1, mode="verify", q_len_per_req=4)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    pb = workloads.batch_decode(batch=16)
    a = run_gpu(pb, False, -1, mode="decode")
    b = run_gpu(pb, False, -1, mode="decode")
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


@pytest.mark.parametrize("force", [0, 4])
@pytest.mark.parametrize("window_left", [-1, 6])
def test_verify_32_rows_in_one_tile(force, window_left):
    """8 draft rows at GQA 4: 32 packed rows in one tile of the pair
    consumer (two M tiles over complementary key halves)."""
    kv = [8, 11, 300, 1200, 77]
    pb = workloads.make_paged_batch([8] * len(kv), kv, 32, 8, 128, 16, "bf16", 61)
    out, lse, plan = run_gpu(pb, True, window_left, mode="verify", force_kv_chunks=force,
                             q_len_per_req=8)
    info = plan.info()
    assert info["kernel_name"] == "decode" and info["tile_rows"] == 32
    assert_close(pb, out, lse, True, window_left, what="verify 32 rows f=%d wl=%d" % (
        force, window_left))


@pytest.mark.parametrize("hq,hk,qlen", [(8, 8, 20), (16, 8, 9), (32, 8, 5), (64, 8, 3),
                                         (32, 2, 2), (16, 16, 32)])
@pytest.mark.parametrize("head_dim,dtype", [(128, "bf16"), (64, "f16")])
@pytest.mark.parametrize("force", [0, 3])
def test_pair_consumer_groups(hq, hk, qlen, head_dim, dtype, force):
    """17 to 32 packed rows for every group (1, 2, 4, 8, 16), both head
    dims and dtypes, split or not: rows past the request's own (a 20-row
    tile of group 1, an 18-row tile of group 2) stay unwritten padding."""
    kv = [qlen, qlen + 5, 130, 999, 64]
    pb = workloads.make_paged_batch([qlen] * len(kv), kv, hq, hk, head_dim, 16, dtype,
                                    300 + hq + qlen + head_dim)
    out, lse, plan = run_gpu(pb, True, -1, mode="verify", force_kv_chunks=force,
                             q_len_per_req=qlen)
    info = plan.info()
    g = hq // hk
    assert info["kernel_name"] == "decode" and info["tile_rows"] == (32 // g) * g
    assert_close(pb, out, lse, True, -1, what="pair g=%d q=%d d=%d f=%d" % (g, qlen, head_dim,
                                                                                force))


def test_pair_consumer_mixed_rows_and_window():
    """Ragged short prefill mixing 1..32 packed rows (GQA 4: 1..8 query rows)
    with a window: tiles of the pair consumer with fewer live rows than 32."""
    q_lens = [8, 5, 1, 7, 0, 6]
    kv_lens = [8, 40, 300, 2100, 10, 6]
    pb = workloads.make_paged_batch(q_lens, kv_lens, 16, 4, 128, 16, "bf16", 91)
    for causal, wl in ((True, -1), (False, 33), (True, 7)):
        out, lse, plan = run_gpu(pb, causal, wl, mode="prefill")
        info = plan.info()
        assert info["kernel_name"] == "decode" and info["tile_rows"] == 32
        assert_close(pb, out, lse, causal, wl, what="pair mixed causal=%s wl=%d" % (causal, wl))
