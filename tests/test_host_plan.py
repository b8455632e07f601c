"""Host-side logic of libfi, on the CPU through the C ABI with host-only plans:
refusals, plan transactionality, graph-mode capacity and frozen shapes, and
exact-cover properties of the work list. No GPU is touched."""
import ctypes

import numpy as np
import pytest
import torch

import paged_kv_attention_13_gb300 as fi
import workloads


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_attention_13_gb300 import build
    build.build()


def _plan(**kw):
    return fi.Plan(None, **kw)


def _status(exc):
    return exc.value.status_name


# --------------------------------------------------------------- refusals
def test_gqa_indivisible_and_zero_kv_heads_refused():
    p = _plan()
    for hq, hk in [(12, 8), (4, 8), (8, 0)]:
        with pytest.raises(fi.FiError) as e:
            p.plan([0, 4], [0, 1], [4], 16, hq, hk, 128)
        assert _status(e) == "FI_ERR_GQA_INDIVISIBLE"


def test_unsupported_head_dim_and_dtype():
    p = _plan()
    with pytest.raises(fi.FiError) as e:
        p.plan([0, 4], [0, 1], [4], 16, 8, 2, 96)
    assert _status(e) == "FI_ERR_UNSUPPORTED"
    with pytest.raises(fi.FiError) as e:
        p.plan([0, 4], [0, 1], [4], 16, 8, 2, 128, dtype=torch.float32)
    assert _status(e) == "FI_ERR_UNSUPPORTED"


def test_kv_shorter_than_q_under_causal_refused_from_metadata():
    p = _plan()
    with pytest.raises(fi.FiError) as e:  # Lk = 3 < Lq = 5
        p.plan([0, 5], [0, 1], [3], 16, 8, 2, 128, causal=True)
    assert _status(e) == "FI_ERR_KV_SHORTER_THAN_Q"
    assert "kv_len=3" in str(e.value) and "qo_len=5" in str(e.value)
    # non-causal accepts it
    p.plan([0, 5], [0, 1], [3], 16, 8, 2, 128, causal=False)
    # verify: the page metadata says 16 tokens, the draft is 32 rows
    with pytest.raises(fi.FiError) as e:
        p.plan(None, [0, 1], [16], 16, 8, 2, 128, q_len_per_req=32)
    assert _status(e) == "FI_ERR_KV_SHORTER_THAN_Q"


def test_bad_metadata_refused():
    p = _plan()
    cases = [
        dict(qo=[0, 4], kv=[0, 1], last=[17]),   # last_page_len > page_size
        dict(qo=[0, 4], kv=[0, 1], last=[0]),    # last_page_len 0 with a page
        dict(qo=[1, 4], kv=[0, 1], last=[4]),    # qo_indptr[0] != 0
        dict(qo=[0, 4, 3], kv=[0, 1, 2], last=[4, 4]),  # qo_indptr decreasing
        dict(qo=[0, 4, 5], kv=[0, 2, 1], last=[4, 4]),  # kv_indptr decreasing
    ]
    for c in cases:
        with pytest.raises(fi.FiError) as e:
            p.plan(c["qo"], c["kv"], c["last"], 16, 8, 2, 128)
        assert _status(e) == "FI_ERR_INVALID_ARG", c
    with pytest.raises(fi.FiError) as e:
        p.plan([0, 4], [0, 1], [4], 16, 8, 2, 128, window_left=-2)
    assert _status(e) == "FI_ERR_INVALID_ARG"
    with pytest.raises(fi.FiError) as e:  # decode plans derive qo_indptr themselves
        p.plan([0, 1], [0, 1], [4], 16, 8, 2, 128, q_len_per_req=1)
    assert _status(e) == "FI_ERR_INVALID_ARG"


def test_rejected_plan_leaves_previous_plan_usable():
    p = _plan()
    p.plan([0, 3, 10], [0, 2, 5], [7, 16], 16, 8, 2, 128, causal=True)
    before = p.info(with_arrays=True)
    # a *different* page table that is refused: nothing may change
    with pytest.raises(fi.FiError):
        p.plan([0, 30, 40], [0, 1, 2], [16, 16], 16, 8, 2, 128, causal=True)
    after = p.info(with_arrays=True)
    for k in ("batch", "total_rows", "num_items"):
        assert before[k] == after[k]
    assert np.array_equal(before["items"], after["items"])


def test_run_before_plan_and_run_refusals():
    lib = fi.load()
    p = _plan()
    T, Hq, Hk, d, P = 9, 8, 2, 128, 16
    q = torch.zeros((T, Hq, d), dtype=torch.bfloat16)
    k = torch.zeros((4, P, Hk, d), dtype=torch.bfloat16)
    v = torch.zeros_like(k)
    idx = torch.zeros(4, dtype=torch.int32)
    out = torch.zeros_like(q)
    lse = torch.zeros((T, Hq), dtype=torch.float32)

    def run(qq=q, kk=k, vv=v, ii=idx, oo=out, ll=lse, decode=False):
        f = fi.fi_batch_decode_paged if decode else fi.fi_batch_prefill_paged
        with pytest.raises(fi.FiError) as e:
            f(p, qq, kk, vv, ii, 0.1, out=oo, lse=ll)
        return _status(e), str(e.value)

    assert run()[0] == "FI_ERR_NOT_PLANNED"
    p.plan([0, 4, 9], [0, 2, 4], [5, 16], P, Hq, Hk, d, causal=True)
    # strided last dim refused, never copied
    wide = torch.zeros((T, Hq, 2 * d), dtype=torch.bfloat16)
    assert run(qq=wide[..., ::2])[0] == "FI_ERR_STRIDED_LAST_DIM"
    kw = torch.zeros((4, P, Hk, 2 * d), dtype=torch.bfloat16)
    assert run(kk=kw[..., ::2])[0] == "FI_ERR_STRIDED_LAST_DIM"
    # plan-vs-run mismatches name the field, the planned and the given value
    st, msg = run(qq=torch.zeros((T, 4, d), dtype=torch.bfloat16))
    assert st == "FI_ERR_PLAN_MISMATCH" and "num_qo_heads" in msg and "8" in msg and "4" in msg
    st, msg = run(kk=torch.zeros((4, 8, Hk, d), dtype=torch.bfloat16))
    assert st == "FI_ERR_PLAN_MISMATCH" and "page_size" in msg
    st, msg = run(qq=torch.zeros((T - 1, Hq, d), dtype=torch.bfloat16))
    assert st == "FI_ERR_PLAN_MISMATCH" and "rows" in msg
    st, msg = run(qq=torch.zeros((1, T, Hq, d), dtype=torch.bfloat16))
    assert st == "FI_ERR_PLAN_MISMATCH" and "rank" in msg
    st, _ = run(qq=q.half())
    assert st == "FI_ERR_PLAN_MISMATCH"
    st, _ = run(decode=True)  # a prefill plan run through the decode entry point
    assert st == "FI_ERR_PLAN_MISMATCH"
    # outputs must be packed
    obig = torch.zeros((T, Hq + 1, d), dtype=torch.bfloat16)
    assert run(oo=obig[:, :Hq])[0] == "FI_ERR_NONCONTIGUOUS_OUTPUT"
    lbig = torch.zeros((T, 2 * Hq), dtype=torch.float32)
    assert run(ll=lbig[:, ::2])[0] == "FI_ERR_STRIDED_LAST_DIM"
    # kv_indices shorter than the plan's page count
    assert run(ii=idx[:3])[0] == "FI_ERR_PLAN_MISMATCH"
    # a valid run on a host-only plan stops before any launch
    st, msg = run()
    assert st == "FI_ERR_INVALID_ARG" and "workspace" in msg
    # q padded with extra rows is accepted up to the launch
    st, msg = run(qq=torch.zeros((T + 5, Hq, d), dtype=torch.bfloat16),
                  oo=torch.zeros((T + 5, Hq, d), dtype=torch.bfloat16),
                  ll=torch.zeros((T + 5, Hq), dtype=torch.float32))
    assert st == "FI_ERR_INVALID_ARG" and "workspace" in msg


def test_graph_mode_capacity_and_frozen_shape():
    p = _plan(enable_graph_capture=True, max_batch=4, max_total_rows=16)
    p.plan(None, [0, 1, 2], [8, 9], 16, 32, 8, 128, q_len_per_req=4)
    assert p.info()["graph_mode"] == 1
    with pytest.raises(fi.FiError) as e:  # batch beyond capacity
        p.plan(None, [0, 1, 2, 3, 4, 5], [8, 9, 10, 11, 12], 16, 32, 8, 128, q_len_per_req=4)
    assert _status(e) == "FI_ERR_CAPACITY"
    with pytest.raises(fi.FiError) as e:  # draft length frozen, both directions
        p.plan(None, [0, 1, 2], [8, 9], 16, 32, 8, 128, q_len_per_req=1)
    assert _status(e) == "FI_ERR_CAPACITY" and "q_len_per_req" in str(e.value)
    with pytest.raises(fi.FiError) as e:
        p.plan(None, [0, 1, 2], [8, 9], 16, 64, 8, 128, q_len_per_req=4)
    assert _status(e) == "FI_ERR_CAPACITY"
    p.plan(None, [0, 3, 4], [8, 9], 16, 32, 8, 128, q_len_per_req=4)  # same shape: fine


def _check_cover(p, pb, causal, wl, forced):
    info = p.info(with_arrays=True)
    items = info["items"]
    g = pb.num_qo_heads // pb.num_kv_heads
    tile = info["tile_rows"]
    assert tile % g == 0 and tile >= g
    qo = pb.qo_indptr.numpy()
    # every (request, packed row, kv head) is covered by exactly one tile
    seen = {}
    for it in items:
        b, hk, row0, kb, ke, chunk, nch, base = (int(x) for x in it)
        if b < 0:  # schedule padding of the persistent grid
            continue
        seen.setdefault((b, hk, row0), set()).add((chunk, kb, ke, nch, base))
    for b in range(len(qo) - 1):
        lq = qo[b + 1] - qo[b]
        lk = pb.kv_lens[b]
        rows = list(range(0, lq * g, tile))
        for hk in range(pb.num_kv_heads):
            for row0 in rows:
                chunks = sorted(seen.pop((b, hk, row0)))
                nch = chunks[0][2 + 1]
                assert all(c[3] == nch for c in chunks) and len(chunks) == nch
                if nch == 1:
                    assert chunks[0][0] == -1
                else:
                    assert [c[0] for c in chunks] == list(range(nch))
                # chunks partition one contiguous key range
                spans = [(c[1], c[2]) for c in chunks]
                for (a0, a1), (b0, b1) in zip(spans, spans[1:]):
                    assert a1 == b0
                if forced:
                    assert spans[0][0] == 0 and spans[-1][1] == lk
                else:
                    n_rows = min(tile, lq * g - row0)
                    i0, i1 = row0 // g, (row0 + n_rows) // g - 1
                    hi = min(lk, i1 + lk - lq + 1) if causal else lk
                    lo = max(0, lk - lq + i0 - wl) if wl >= 0 else 0
                    lo = min(lo, hi)
                    assert spans[0][0] == lo and spans[-1][1] == hi
    assert not seen, "items for rows that do not exist: %s" % list(seen)[:3]
    # merge index: tokens of split tiles own num_chunks partial slots
    merge = info["merge_indptr"]
    assert merge[0] == 0 and np.all(np.diff(merge) >= 0)
    assert merge[-1] == info["num_partials"]
    assert info["num_merge_rows"] == int(np.sum(np.diff(merge) > 1))
    for it in items:
        if it[0] >= 0 and it[5] >= 0:
            b, row0, nch, base = int(it[0]), int(it[2]), int(it[6]), int(it[7])
            t = qo[b] + row0 // g
            assert merge[t] == base and merge[t + 1] - merge[t] == nch


@pytest.mark.parametrize("forced", [0, 5])
@pytest.mark.parametrize("causal,wl", [(True, -1), (True, 100), (False, 33), (False, -1)])
def test_work_list_is_an_exact_cover(forced, causal, wl):
    pb = workloads.batch_prefill(batch=6, q_lo=1, q_hi=300, prefix_lo=0, prefix_hi=900,
                                 num_qo_heads=12, num_kv_heads=4, head_dim=64)
    p = _plan()
    p.plan(pb.qo_indptr, pb.kv_indptr, pb.last_page_len, 16, 12, 4, 64, causal=causal,
           window_left=wl, force_kv_chunks=forced)
    _check_cover(p, pb, causal, wl, forced)


def test_decode_split_cover_and_long_context_split():
    pb = workloads.batch_decode(batch=64)
    p = _plan()
    p.plan(None, pb.kv_indptr, pb.last_page_len, 16, 32, 8, 128, q_len_per_req=1)
    info = p.info()
    assert info["kernel_name"] == "decode"
    _check_cover(p, pb, True, -1, 0)
    pb = workloads.long_context()
    for forced in (0, 8, 32):
        p.plan(pb.qo_indptr, pb.kv_indptr, pb.last_page_len, 16, 64, 8, 128, causal=True,
               force_kv_chunks=forced)
        _check_cover(p, pb, True, -1, forced)
        if forced:
            assert p.info()["max_chunks"] == forced


def _meta_batch(ql, kl, hq, hk, P):
    """Plan metadata only (no tensors): qo/kv indptr, last_page_len, kv_lens."""
    from types import SimpleNamespace
    pages = [(k + P - 1) // P for k in kl]
    return SimpleNamespace(
        qo_indptr=torch.tensor(np.concatenate([[0], np.cumsum(ql)]), dtype=torch.int32),
        kv_indptr=torch.tensor(np.concatenate([[0], np.cumsum(pages)]), dtype=torch.int32),
        last_page_len=torch.tensor([k - (n - 1) * P if n else 0 for k, n in zip(kl, pages)],
                                   dtype=torch.int32),
        kv_lens=list(kl), num_qo_heads=hq, num_kv_heads=hk)


@pytest.mark.parametrize("seed", range(12))
def test_random_plans_are_exact_covers(seed):
    """Seeded random batches through every planning path (prefill on each
    kernel, decode, verify, forced and planner-chosen splits, few long units
    that take the chunk-length search): the work list covers every
    (request, row tile, kv head) once and each tile's chunks partition its
    live key range."""
    rng = np.random.default_rng(7000 + seed)
    hk = int(rng.choice([1, 2, 8]))
    g = int(rng.choice([1, 4, 8]))
    d = int(rng.choice([64, 128]))
    B = int(rng.integers(1, 12))
    mode = ["prefill", "decode", "verify", "long"][seed % 4]
    causal = bool(rng.integers(0, 2)) or mode == "verify"
    wl = int(rng.choice([-1, -1, 0, 37, 500]))
    forced = int(rng.choice([0, 0, 3]))
    if mode == "long":  # few long units: the makespan-chosen chunk length
        kl = [int(rng.integers(20000, 40000))] * B
        ql = [int(rng.integers(1, 17))] * B
    else:
        kl = [int(x) for x in rng.integers(1, 3000, size=B)]
        ql = [1] * B if mode == "decode" else (
            [4] * B if mode == "verify" else [int(x) for x in rng.integers(1, 400, size=B)])
    if causal:
        kl = [max(k, q) for k, q in zip(kl, ql)]
    pb = _meta_batch(ql, kl, g * hk, hk, 16)
    p = _plan()
    if mode in ("decode", "verify"):
        p.plan(None, pb.kv_indptr, pb.last_page_len, 16, g * hk, hk, d, causal=causal,
               window_left=wl, q_len_per_req=ql[0], force_kv_chunks=forced)
    else:
        p.plan(pb.qo_indptr, pb.kv_indptr, pb.last_page_len, 16, g * hk, hk, d, causal=causal,
               window_left=wl, force_kv_chunks=forced)
    _check_cover(p, pb, causal or mode == "verify", wl, forced)


def test_workspace_bytes_grows_with_chunks():
    a = fi.workspace_bytes(64, 64, 32, 128, 1)
    b = fi.workspace_bytes(64, 64, 32, 128, 32)
    assert 0 < a < b
    assert b >= 64 * 32 * 32 * 129 * 4


def test_schedule_balances_the_persistent_grid():
    """Items are laid out so CTA c runs positions c, c + grid, ...: the
    balanced spans keep every CTA's share of keys within a few percent of
    the mean on the batch-decode workload."""
    pb = workloads.batch_decode()
    p = _plan()
    p.plan(None, pb.kv_indptr, pb.last_page_len, 16, 32, 8, 128, q_len_per_req=1)
    info = p.info(with_arrays=True)
    items, G = info["items"], info["grid"]
    assert len(items) % G == 0
    kv = np.array(pb.kv_lens)
    load = np.zeros(G)
    for i, it in enumerate(items):
        if it[0] >= 0:
            load[i % G] += max(0, min(int(it[4]), kv[it[0]]) - int(it[3])) + 32
    assert load.max() / load.mean() < 1.03


def _tc_step_loads(info, pb, causal, page_size):
    """Per-CTA time of a tcgen05 prefill plan in tile steps: each item pays its
    128-key tiles (counted from the K/V box boundary at or below its first live
    key) once per 128-row Q tile, plus 2 steps for its start and epilogue."""
    items, G = info["items"], info["grid"]
    g = pb.num_qo_heads // pb.num_kv_heads
    qo = pb.qo_indptr.numpy()
    kv = np.array(pb.kv_lens)
    box = int(np.gcd(page_size, 128))
    load = np.zeros(G)
    for i, it in enumerate(items):
        b, row0, kb, ke = int(it[0]), int(it[2]), int(it[3]), int(it[4])
        if b < 0:
            continue
        lq, lk = int(qo[b + 1] - qo[b]), int(kv[b])
        rows = min(info["tile_rows"], lq * g - row0)
        i1 = (row0 + rows) // g - 1
        hi = min(ke, min(lk, i1 + lk - lq + 1) if causal else lk)
        lo = kb
        n_kt = (hi - lo // box * box + 127) // 128 if hi > lo else 0
        load[i % G] += n_kt * (2 if rows > 128 else 1) + 2
    return load


@pytest.mark.parametrize("causal,page", [(True, 16), (False, 16), (True, 1024)])
def test_tcgen05_prefill_schedule_is_balanced(causal, page):
    """The unsplit batch-16 prefill on the tcgen05 kernel: items dealt longest
    first by their tile steps leave no CTA more than 2% above the mean (a
    schedule by live keys x rows left the longest 4% above it)."""
    pb = workloads.batch_prefill(page_size=page)
    p = _plan()
    p.plan(pb.qo_indptr, pb.kv_indptr, pb.last_page_len, page, 32, 8, 128, causal=causal)
    info = p.info(with_arrays=True)
    assert info["kernel_name"] == "prefill_m128" and info["max_chunks"] == 1
    load = _tc_step_loads(info, pb, causal, page)
    assert load.max() / load.mean() < 1.02
    _check_cover(p, pb, causal, -1, 0)


def test_tcgen05_split_plan_weighs_q_tiles():
    """The head_dim-64 prefill (4 q / 2 kv heads) is split into spans: a
    request's last, partial Q tile is weighed as the whole 128-row tile the
    kernel computes, so no CTA carries more than 10% above the mean in tile
    steps (weighing it by its live rows left one 23% above)."""
    pb = workloads.batch_prefill_hd64()
    p = _plan()
    p.plan(pb.qo_indptr, pb.kv_indptr, pb.last_page_len, 16, 4, 2, 64, causal=True,
           dtype=torch.float16)
    info = p.info(with_arrays=True)
    assert info["kernel_name"] == "prefill_m128" and info["max_chunks"] > 1
    load = _tc_step_loads(info, pb, True, 16)
    assert load.max() / load.mean() < 1.10
    _check_cover(p, pb, True, -1, 0)


def _cta_loads(info, kv_lens):
    items, G = info["items"], info["grid"]
    load = np.zeros(G)
    for i, it in enumerate(items):
        if it[0] >= 0:
            load[i % G] += max(0, min(int(it[4]), kv_lens[it[0]]) - int(it[3]))
    return load


def test_long_context_split_is_balanced():
    """A few long units over many CTAs: 8 requests x 8 kv heads of 32768 keys
    on the 152-CTA tcgen05 grid. The chunk length is chosen by the simulated
    makespan, so no CTA carries much more than the mean (an even 5-way cut
    leaves 16 CTAs with a third chunk, 24% above it)."""
    pb = workloads.long_context()
    p = _plan()
    for causal in (True, False):
        p.plan(pb.qo_indptr, pb.kv_indptr, pb.last_page_len, 16, 64, 8, 128, causal=causal)
        info = p.info(with_arrays=True)
        assert info["kernel_name"] == "prefill_m128"
        load = _cta_loads(info, np.array(pb.kv_lens))
        assert load.sum() == 8 * 8 * 32768  # every key of every unit, once
        assert load.max() / load.mean() < 1.05
        _check_cover(p, pb, causal, -1, 0)


def _span_costs(info, rows_of):
    """Per-CTA cost of a short-query plan: (keys + 32) x rows per item, the
    span scheduler's own cost model."""
    items, G = info["items"], info["grid"]
    cost = np.zeros(G)
    for i, it in enumerate(items):
        if it[0] >= 0:
            cost[i % G] += (int(it[4]) - int(it[3]) + 32) * rows_of(it)
    return cost


@pytest.mark.parametrize("which", ["verify", "tree", "decode"])
def test_short_query_spans_are_balanced(which):
    """Split short-query plans cut the keys of all tiles, end to end, into one
    span per bundle of kv-head CTAs: every CTA's cost is within a few percent
    of the mean, the kv heads of a piece run side by side, and the work list
    stays an exact cover."""
    p = _plan()
    if which == "verify":
        pb = workloads.speculative_verify(batch=32)
        p.plan(None, pb.kv_indptr, pb.last_page_len, 16, 32, 8, 128, q_len_per_req=4)
    elif which == "tree":
        pb = workloads.tree_verify(batch=32)
        p.plan_masked(pb.qo_indptr, pb.kv_indptr, pb.last_page_len, 16, 32, 8, 128,
                      pb.extra["mask_indptr"].numpy(), causal=True)
    else:
        pb = workloads.batch_decode()
        p.plan(None, pb.kv_indptr, pb.last_page_len, 16, 32, 8, 128, q_len_per_req=1)
    info = p.info(with_arrays=True)
    assert info["kernel_name"] == "decode" and info["max_chunks"] > 1
    cost = _span_costs(info, lambda it: info["tile_rows"])
    used = cost[cost > 0]
    assert len(used) == info["grid"]
    assert used.max() / used.mean() < 1.03
    items, G = info["items"], info["grid"]
    for i in range(0, len(items), 8):  # a bundle: the 8 kv heads of one piece
        blk = items[i:i + 8]
        if blk[0][0] >= 0:
            assert [int(x[1]) for x in blk] == list(range(8))
            assert len({(int(x[0]), int(x[3]), int(x[4])) for x in blk}) == 1
    # far fewer item ends than fixed chunks: at most 5 items per CTA
    per_cta = np.bincount(np.nonzero(info["items"][:, 0] >= 0)[0] % info["grid"])
    assert per_cta.max() <= 5
    _check_cover(p, pb, True, -1, 0)


@pytest.mark.parametrize("seed", range(40))
def test_short_query_spans_terminate_and_cover(seed):
    """Random short-query batches (1 to 300 requests, 1 to 20000 keys, one
    to eight query rows) plan quickly and exactly cover their keys."""
    import time
    rng = np.random.default_rng(9100 + seed)
    hk = int(rng.choice([1, 2, 4, 8]))
    g = int(rng.choice([1, 2, 4, 8]))
    B = int(rng.choice([1, 2, 5, 17, 64, 300]))
    q = int(rng.choice([1, 2, 4, 8]))
    hi = int(rng.choice([40, 700, 5000, 20000]))
    kl = [max(q, int(x)) for x in rng.integers(1, hi + 1, size=B)]
    pb = _meta_batch([q] * B, kl, g * hk, hk, 16)
    p = _plan()
    t0 = time.perf_counter()
    p.plan(None, pb.kv_indptr, pb.last_page_len, 16, g * hk, hk, 128, q_len_per_req=q)
    assert time.perf_counter() - t0 < 2.0
    _check_cover(p, pb, True, -1, 0)


# ----------------------------------------------------------- ragged prefill

def _ragged(q_lens, kv_lens, hq=8, hk=2, d=128, seed=3):
    """A batch whose page-size-1, unpermuted cache is the contiguous K/V."""
    return workloads.make_paged_batch(q_lens, kv_lens, hq, hk, d, 1, "bf16", seed,
                                      permute_pages=False)


@pytest.mark.parametrize("causal,wl,forced", [(True, -1, 0), (False, 7, 0), (True, 3, 5)])
def test_ragged_plan_is_an_exact_cover(causal, wl, forced):
    pb = _ragged([5, 300, 0, 17, 2000], [5, 400, 9, 17, 2100])
    p = _plan()
    p.plan_ragged(pb.qo_indptr, pb.kv_indptr, 8, 2, 128, causal=causal, window_left=wl,
                  force_kv_chunks=forced)
    _check_cover(p, pb, causal, wl, forced)


def test_ragged_plan_refusals():
    p = _plan()
    # decreasing row offsets
    with pytest.raises(fi.FiError) as e:
        p.plan_ragged([0, 4, 8], [0, 10, 5], 8, 2, 128)
    assert _status(e) == "FI_ERR_INVALID_ARG"
    # fewer keys than query rows under the causal mask (kv_len from the offsets)
    with pytest.raises(fi.FiError) as e:
        p.plan_ragged([0, 4, 8], [0, 10, 13], 8, 2, 128, causal=True)
    assert _status(e) == "FI_ERR_KV_SHORTER_THAN_Q"
    p.plan_ragged([0, 4, 8], [0, 10, 13], 8, 2, 128, causal=False)


def test_ragged_and_paged_plans_do_not_cross():
    """A ragged plan refuses the paged run calls and a paged plan the ragged
    one (checked on the host, before any launch)."""
    pb = _ragged([3, 4], [10, 12])
    T = int(pb.qo_indptr[-1])
    q = torch.zeros((T, 8, 128), dtype=torch.bfloat16)
    kv = torch.zeros((22, 2, 128), dtype=torch.bfloat16)
    out = torch.zeros_like(q)
    p = _plan()
    p.plan_ragged(pb.qo_indptr, pb.kv_indptr, 8, 2, 128)
    with pytest.raises(fi.FiError) as e:
        fi.fi_batch_prefill_paged(p, q, pb.k_cache, pb.v_cache, pb.kv_indices, 0.1, out=out)
    assert _status(e) == "FI_ERR_PLAN_MISMATCH"
    p2 = _plan()
    p2.plan(pb.qo_indptr, pb.kv_indptr, pb.last_page_len, 1, 8, 2, 128)
    with pytest.raises(fi.FiError) as e:
        fi.fi_batch_prefill_ragged(p2, q, kv, kv, 0.1, out=out)
    assert _status(e) == "FI_ERR_PLAN_MISMATCH"
    # K/V with fewer rows than the plan's last offset
    with pytest.raises(fi.FiError) as e:
        fi.fi_batch_prefill_ragged(p, q, kv[:21], kv[:21], 0.1, out=out)
    assert _status(e) == "FI_ERR_PLAN_MISMATCH"


# ------------------------------------------------------------ custom masks

def test_masked_plan_refusals_and_kernel_choice():
    pb = workloads.tree_verify(batch=3, n_draft=4, kv_lo=20, kv_hi=40)
    mi = pb.extra["mask_indptr"].numpy()
    p = _plan()
    p.plan_masked(pb.qo_indptr, pb.kv_indptr, pb.last_page_len, 16, 32, 8, 128, mi, causal=True)
    assert p.info()["kernel_name"] == "decode"  # 16 packed rows, page 16
    # a segment one byte short of its request's bits
    short = mi.copy()
    short[1:] -= 1
    short[1] = max(short[1], 0)
    with pytest.raises(fi.FiError) as e:
        p.plan_masked(pb.qo_indptr, pb.kv_indptr, pb.last_page_len, 16, 32, 8, 128, short)
    assert _status(e) == "FI_ERR_INVALID_ARG"
    # more than 32 packed rows: the tcgen05 kernel reads the mask too; at a
    # page size it cannot tile (2), the mma.sync M = 64 kernel
    pb2 = workloads.tree_verify(batch=2, n_draft=40, kv_lo=100, kv_hi=200)
    p.plan_masked(pb2.qo_indptr, pb2.kv_indptr, pb2.last_page_len, 16, 32, 8, 128,
                  pb2.extra["mask_indptr"].numpy())
    assert p.info()["kernel_name"] == "prefill_m128"
    pb3 = workloads.tree_verify(batch=2, n_draft=40, kv_lo=100, kv_hi=200, page_size=2)
    p.plan_masked(pb3.qo_indptr, pb3.kv_indptr, pb3.last_page_len, 2, 32, 8, 128,
                  pb3.extra["mask_indptr"].numpy())
    assert p.info()["kernel_name"] == "prefill_m64"


def test_masked_and_unmasked_plans_do_not_cross():
    pb = workloads.tree_verify(batch=2, n_draft=4, kv_lo=20, kv_hi=30)
    T = int(pb.qo_indptr[-1])
    q = torch.zeros((T, 32, 128), dtype=torch.bfloat16)
    out = torch.zeros_like(q)
    args = (q, pb.k_cache, pb.v_cache, pb.kv_indices)
    p = _plan()
    p.plan_masked(pb.qo_indptr, pb.kv_indptr, pb.last_page_len, 16, 32, 8, 128,
                  pb.extra["mask_indptr"].numpy())
    with pytest.raises(fi.FiError) as e:
        fi.fi_batch_prefill_paged(p, *args, 0.1, out=out)
    assert _status(e) == "FI_ERR_PLAN_MISMATCH"
    # a mask tensor shorter than the plan's segments
    with pytest.raises(fi.FiError) as e:
        fi.fi_batch_prefill_paged_masked(p, *args, pb.extra["mask"][:-1], 0.1, out=out)
    assert _status(e) == "FI_ERR_PLAN_MISMATCH"
    p2 = _plan()
    p2.plan(pb.qo_indptr, pb.kv_indptr, pb.last_page_len, 16, 32, 8, 128)
    with pytest.raises(fi.FiError) as e:
        fi.fi_batch_prefill_paged_masked(p2, *args, pb.extra["mask"], 0.1, out=out)
    assert _status(e) == "FI_ERR_PLAN_MISMATCH"


def test_plan_metadata_inputs_are_equivalent():
    """The binding takes host metadata as int32/int64 tensors (contiguous or
    not), numpy arrays or lists; every form gives the same plan."""
    pb = workloads.speculative_verify(batch=8, kv_lo=64, kv_hi=900)
    base = pb.kv_indptr.to(torch.int32)
    last = pb.last_page_len.to(torch.int32)
    forms = [
        (base, last),
        (base.to(torch.int64), last.to(torch.int64)),
        (base.numpy(), last.numpy()),
        (base.tolist(), last.tolist()),
        (torch.stack([base, base], 1)[:, 0], torch.stack([last, last], 1)[:, 1]),  # strided
    ]
    ref = None
    for kv, lp in forms:
        p = _plan()
        p.plan(None, kv, lp, 16, 32, 8, 128, causal=True, q_len_per_req=4)
        info = p.info(with_arrays=True)
        got = (info["items"].tobytes(), info["merge_indptr"].tobytes(), info["grid"])
        if ref is None:
            ref = got
        assert got == ref


def test_tensor_desc_shapes_and_strides():
    t = torch.zeros((5, 3, 4, 8), dtype=torch.bfloat16)
    d = fi.tensor_desc(t.permute(0, 2, 1, 3))
    assert d.ndim == 4 and list(d.shape) == [5, 4, 3, 8] and list(d.stride) == [96, 8, 32, 1]
    assert d.data == t.data_ptr()
    d = fi.tensor_desc(torch.zeros(7, dtype=torch.int32))
    assert d.ndim == 1 and list(d.shape) == [7, 0, 0, 0] and list(d.stride) == [1, 0, 0, 0]
    with pytest.raises(ValueError):
        fi.tensor_desc(torch.zeros((1, 1, 1, 1, 1)))
    with pytest.raises(ValueError):
        fi.tensor_desc(torch.zeros(3, dtype=torch.float64))
