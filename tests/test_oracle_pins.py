"""Pins for the CPU oracle: it is checked against things other than itself.

- hand-worked mask examples from the pages' inequalities (tests/golden);
- closed forms: with all keys equal, lse - s = ln(#valid keys) for every row,
  and with v_j = j the output is the mean valid index;
- textbook reductions: torch's scaled_dot_product_attention on the CPU in
  fp64, with no mask and with its lower-right (bottom-right) causal bias;
- library decoding of fp16/bf16 inputs;
- the invariants the pages fix (window >= kv_len is no window, causal with one
  query row is full attention, split + merge is the unsplit result, page size
  does not matter, GQA is MHA with repeated K/V heads, windowed differs from
  unwindowed);
- a numpy brute force with an explicit mask matrix on tiny inputs.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import brute
from oracle.reference import attention_all, attention_rows, key_valid, kv_len, merge_states
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "mask_worked_examples.txt")


def _contig_paged(K, V, page_size, rng, extra_pages=0):
    """Page a dense [Lk, Hk, d] K/V into a permuted pool (test helper)."""
    lk, hk, d = K.shape
    n = (lk + page_size - 1) // page_size
    pool = n + extra_pages
    perm = rng.permutation(pool)[:n].astype(np.int32)
    kc = np.zeros((max(pool, 1), page_size, hk, d), K.dtype)
    vc = np.zeros_like(kc)
    for p in range(n):
        rows = slice(p * page_size, min((p + 1) * page_size, lk))
        cnt = rows.stop - rows.start
        kc[perm[p], :cnt] = K[rows]
        vc[perm[p], :cnt] = V[rows]
    last = lk - (n - 1) * page_size if n else 0
    return kc, vc, perm, np.array([0, n], np.int32), np.array([last], np.int32)


def _single(q, K, V, page_size, causal, wl, scale, rng):
    kc, vc, idx, kvp, last = _contig_paged(K, V, page_size, rng)
    qo = np.array([0, q.shape[0]], np.int32)
    return attention_all(q, kc, vc, idx, qo, kvp, last, page_size, causal, wl, scale)


def _count_closed_form(i, lq, lk, causal, wl):
    hi = min(lk - 1, i + lk - lq) if causal else lk - 1
    lo = max(0, lk - lq + i - wl) if wl >= 0 else 0
    return max(0, hi - lo + 1), lo, hi


# --------------------------------------------------------------- golden mask
def _golden_cases():
    cases = []
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        head, keys = line.split(":")
        lq, lk, causal, wl, row = (int(x) for x in head.split())
        cases.append((lq, lk, causal, wl, row, [int(x) for x in keys.split()]))
    return cases


@pytest.mark.parametrize("case", _golden_cases())
def test_mask_matches_hand_worked_examples(case):
    lq, lk, causal, wl, row, keys = case
    got = [j for j in range(lk) if key_valid(row, j, lq, lk, causal, wl)]
    assert got == keys
    assert [j for j in range(lk) if brute.mask_matrix(lq, lk, causal, wl)[row, j]] == keys


def test_golden_examples_through_attention_counts():
    """Constant keys: lse - s equals ln(#valid) for the hand-worked rows."""
    for lq, lk, causal, wl, row, keys in _golden_cases():
        d = 4
        q = np.zeros((lq, 1, d), np.float32)
        q[:, 0, 0] = 0.5
        K = np.ones((lk, 1, d), np.float32)
        V = np.zeros((lk, 1, d), np.float32)
        V[:, 0, 0] = np.arange(lk)
        o, lse = _single(q, K, V, 2, bool(causal), wl, 1.0, np.random.default_rng(1))
        if keys:
            assert lse[row, 0] - 0.5 == pytest.approx(math.log(len(keys)), abs=1e-12)
            assert o[row, 0, 0] == pytest.approx(np.mean(keys), abs=1e-12)
        else:
            assert lse[row, 0] == -np.inf and np.all(o[row, 0] == 0)


# --------------------------------------------------------------- closed forms
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("wl", [-1, 0, 1, 3, 7, 40])
@pytest.mark.parametrize("lq,lk", [(1, 1), (1, 9), (4, 9), (9, 9), (7, 30), (6, 3)])
def test_constant_keys_count_and_mean_index(causal, wl, lq, lk):
    if causal and lk < lq:
        pytest.skip("kv shorter than q under causal is refused by the library")
    rng = np.random.default_rng(lq * 100 + lk + wl)
    d = 8
    q = rng.standard_normal((lq, 2, d)).astype(np.float32)
    kvec = rng.standard_normal(d).astype(np.float32)
    K = np.tile(kvec, (lk, 1, 1)).astype(np.float32)  # [lk, 1, d]
    V = np.zeros((lk, 1, d), np.float32)
    V[:, 0, 3] = np.arange(lk)
    scale = 0.37
    for P in (1, 3, 16):
        o, lse = _single(q, K, V, P, causal, wl, scale, rng)
        for i in range(lq):
            cnt, lo, hi = _count_closed_form(i, lq, lk, causal, wl)
            for h in range(2):
                s = scale * float(np.dot(q[i, h].astype(np.float64), kvec.astype(np.float64)))
                if cnt == 0:
                    assert lse[i, h] == -np.inf
                    assert np.all(o[i, h] == 0)
                else:
                    assert lse[i, h] - s == pytest.approx(math.log(cnt), abs=1e-10)
                    assert o[i, h, 3] == pytest.approx((lo + hi) / 2.0, abs=1e-9)


def test_last_row_sees_every_key_under_causal():
    """The bottom-right causal mask lets the last query row attend to all keys."""
    for lq, lk in [(1, 5), (4, 9), (16, 16)]:
        assert all(key_valid(lq - 1, j, lq, lk, True, -1) for j in range(lk))
        assert not key_valid(0, lk - lq + 1, lq, lk, True, -1) or lq == 1


# --------------------------------------------------------------- textbook
def _sdpa64(q, K, V, scale, attn_mask=None):
    qt = torch.from_numpy(q.astype(np.float64)).permute(1, 0, 2)[None]
    kt = torch.from_numpy(K.astype(np.float64)).permute(1, 0, 2)[None]
    vt = torch.from_numpy(V.astype(np.float64)).permute(1, 0, 2)[None]
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=attn_mask,
                                                         scale=scale)
    return o[0].permute(1, 0, 2).numpy()


@pytest.mark.parametrize("lq,lk", [(5, 17), (17, 17), (1, 40)])
def test_unmasked_matches_sdpa(lq, lk):
    rng = np.random.default_rng(3)
    d, H = 16, 3
    q = rng.standard_normal((lq, H, d)).astype(np.float32)
    K = rng.standard_normal((lk, H, d)).astype(np.float32)
    V = rng.standard_normal((lk, H, d)).astype(np.float32)
    o, lse = _single(q, K, V, lk, False, -1, 0.25, rng)
    ref = _sdpa64(q, K, V, 0.25)
    np.testing.assert_allclose(o, ref, atol=1e-12, rtol=0)
    # lse: the log of the softmax denominator, from torch.logsumexp
    S = torch.einsum("qhd,khd->hqk", torch.from_numpy(q).double(), torch.from_numpy(K).double())
    np.testing.assert_allclose(lse, torch.logsumexp(0.25 * S, -1).T.numpy(), atol=1e-12)


@pytest.mark.parametrize("lq,lk", [(5, 17), (12, 12), (1, 9)])
def test_causal_matches_sdpa_lower_right(lq, lk):
    from torch.nn.attention.bias import causal_lower_right
    rng = np.random.default_rng(4)
    d, H = 16, 2
    q = rng.standard_normal((lq, H, d)).astype(np.float32)
    K = rng.standard_normal((lk, H, d)).astype(np.float32)
    V = rng.standard_normal((lk, H, d)).astype(np.float32)
    o, _ = _single(q, K, V, 4, True, -1, 0.3, rng)
    bias = causal_lower_right(lq, lk)
    ref = _sdpa64(q, K, V, 0.3, attn_mask=bias)
    np.testing.assert_allclose(o, ref, atol=1e-12, rtol=0)


def test_input_decoding_matches_library_casts():
    """fp16 and bf16 bit patterns decode to the values numpy/torch give them."""
    rng = np.random.default_rng(5)
    vals = np.concatenate([rng.standard_normal(2000) * 10, [0.0, -0.0, 6.1e-5, 5.96e-8,
                                                            65504.0, -3.0e-6]])
    for name in ("f16", "bf16"):
        t = torch.from_numpy(vals.astype(np.float32)).to(workloads.TORCH_DTYPE[name])
        raw = t.view(torch.int16).numpy().view(np.uint16)
        n = len(vals)
        # identity attention: one key with q=0 -> o = v exactly, per element
        q = np.zeros((1, 1, n), np.uint16)
        kc = np.zeros((1, 1, 1, n), np.uint16)
        vc = raw.reshape(1, 1, 1, n)
        o, lse = attention_rows(q, kc, vc, np.array([0], np.int32), np.array([0, 1], np.int32),
                                np.array([0, 1], np.int32), np.array([1], np.int32), 1,
                                False, -1, 1.0, np.array([0]), np.array([0]), dtype=name)
        np.testing.assert_array_equal(o[0], t.double().numpy())
        assert lse[0] == 0.0


# --------------------------------------------------------------- invariants
def test_window_at_least_kv_len_is_no_window():
    pb = workloads.pr1_reference()
    args = pb.oracle_args()
    for causal in (True, False):
        o1, l1 = attention_all(*args, causal, -1, pb.sm_scale, dtype="f16")
        for wl in (256, 257, 10_000):
            o2, l2 = attention_all(*args, causal, wl, pb.sm_scale, dtype="f16")
            np.testing.assert_array_equal(o1, o2)
            np.testing.assert_array_equal(l1, l2)


def test_windowed_differs_from_unwindowed():
    """Anti-vacuity guard: on the 64x256 workload the window changes the answer."""
    pb = workloads.pr1_reference()
    args = pb.oracle_args()
    for causal in (True, False):
        o1, _ = attention_all(*args, causal, -1, pb.sm_scale, dtype="f16")
        o2, _ = attention_all(*args, causal, 31, pb.sm_scale, dtype="f16")
        assert np.abs(o1 - o2).max() > 0.1


def test_causal_with_one_query_row_is_full_attention():
    pb = workloads.batch_decode(batch=3, kv_lo=5, kv_hi=70, num_qo_heads=4, num_kv_heads=2,
                                head_dim=16)
    args = pb.oracle_args()
    o1, l1 = attention_all(*args, True, -1, pb.sm_scale)
    o2, l2 = attention_all(*args, False, -1, pb.sm_scale)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


def test_split_then_merge_equals_unsplit():
    """Non-causal, unwindowed: attention over two halves of the keys, merged by
    LSE, equals attention over all keys."""
    rng = np.random.default_rng(6)
    lq, lk, d, H = 3, 23, 8, 2
    q = rng.standard_normal((lq, H, d)).astype(np.float32)
    K = rng.standard_normal((lk, H, d)).astype(np.float32)
    V = rng.standard_normal((lk, H, d)).astype(np.float32)
    o, lse = _single(q, K, V, 4, False, -1, 0.4, rng)
    parts = [(0, 5), (5, 6), (6, 23)]
    os_, ss = [], []
    for a, b in parts:
        oi, li = _single(q, K[a:b], V[a:b], 4, False, -1, 0.4, rng)
        os_.append(oi)
        ss.append(li)
    v = np.stack(os_, axis=2).reshape(lq * H, len(parts), d)
    s = np.stack(ss, axis=2).reshape(lq * H, len(parts))
    vm, sm = merge_states(v, s)
    np.testing.assert_allclose(vm, o.reshape(lq * H, d), atol=1e-12)
    np.testing.assert_allclose(sm, lse.reshape(lq * H), atol=1e-12)


def test_merge_closed_forms():
    rng = np.random.default_rng(7)
    v = rng.standard_normal((4, 1, 5))
    s = rng.standard_normal((4, 1))
    # a state merged with itself: same o, lse + ln 2
    vm, sm = merge_states(np.concatenate([v, v], 1), np.concatenate([s, s], 1))
    np.testing.assert_allclose(vm, v[:, 0], atol=1e-14)
    np.testing.assert_allclose(sm, s[:, 0] + math.log(2), atol=1e-14)
    # an empty (-inf) state is the identity
    vm, sm = merge_states(np.concatenate([v, v * 0 + 9], 1),
                          np.concatenate([s, np.full_like(s, -np.inf)], 1))
    np.testing.assert_allclose(vm, v[:, 0], atol=1e-14)
    np.testing.assert_allclose(sm, s[:, 0], atol=1e-14)
    # all empty -> o = 0, lse = -inf
    vm, sm = merge_states(v * 0 + 3, np.full_like(s, -np.inf))
    assert np.all(vm == 0) and np.all(sm == -np.inf)
    # two states: weights are the logistic of the lse difference
    va, vb = rng.standard_normal((2, 6))
    sa, sb = 0.3, -1.1
    vm, sm = merge_states(np.stack([va, vb])[None], np.array([[sa, sb]]))
    wa = 1.0 / (1.0 + math.exp(sb - sa))
    np.testing.assert_allclose(vm[0], wa * va + (1 - wa) * vb, atol=1e-14)
    assert sm[0] == pytest.approx(math.log(math.exp(sa) + math.exp(sb)), abs=1e-14)


@pytest.mark.parametrize("P", [1, 16, 1024])
def test_page_size_does_not_change_the_result(P):
    rng = np.random.default_rng(8)
    lq, lk, d, H = 6, 45, 8, 2
    q = rng.standard_normal((lq, H, d)).astype(np.float32)
    K = rng.standard_normal((lk, H, d)).astype(np.float32)
    V = rng.standard_normal((lk, H, d)).astype(np.float32)
    for causal, wl in [(True, -1), (True, 5), (False, 9)]:
        ref = _single(q, K, V, lk, causal, wl, 0.3, np.random.default_rng(0))
        got = _single(q, K, V, P, causal, wl, 0.3, rng)
        np.testing.assert_allclose(got[0], ref[0], atol=1e-13)
        np.testing.assert_allclose(got[1], ref[1], atol=1e-13)


def test_gqa_equals_mha_with_repeated_kv_heads():
    rng = np.random.default_rng(9)
    lq, lk, d, Hq, Hk = 5, 30, 8, 6, 2
    g = Hq // Hk
    q = rng.standard_normal((lq, Hq, d)).astype(np.float32)
    K = rng.standard_normal((lk, Hk, d)).astype(np.float32)
    V = rng.standard_normal((lk, Hk, d)).astype(np.float32)
    a = _single(q, K, V, 4, True, 7, 0.3, rng)
    b = _single(q, np.repeat(K, g, axis=1), np.repeat(V, g, axis=1), 4, True, 7, 0.3, rng)
    np.testing.assert_allclose(a[0], b[0], atol=1e-13)
    np.testing.assert_allclose(a[1], b[1], atol=1e-13)


def test_kv_len_comes_from_page_metadata():
    kv_indptr = np.array([0, 3, 3, 4], np.int32)
    last = np.array([5, 0, 16], np.int32)
    assert kv_len(kv_indptr, last, 0, 16) == 2 * 16 + 5
    assert kv_len(kv_indptr, last, 1, 16) == 0
    assert kv_len(kv_indptr, last, 2, 16) == 16


# --------------------------------------------------------------- brute force
@pytest.mark.parametrize("seed", range(6))
def test_c_oracle_agrees_with_brute_force(seed):
    rng = np.random.default_rng(100 + seed)
    B = int(rng.integers(1, 4))
    g = int(rng.integers(1, 4))
    Hk = int(rng.integers(1, 3))
    d = int(rng.integers(1, 9))
    P = int(rng.integers(1, 4))
    causal = bool(seed % 2)
    wl = int(rng.choice([-1, 0, 1, 2, 5]))
    ql, kl = [], []
    for _ in range(B):
        lk = int(rng.integers(0, 9))
        lq = int(rng.integers(0 if lk == 0 else 1, (lk if causal else 8) + 1)) if lk else 0
        ql.append(lq)
        kl.append(lk)
    pb = workloads.make_paged_batch(ql, kl, g * Hk, Hk, d, P, "bf16", 1000 + seed,
                                    extra_pool_pages=2)
    args = pb.oracle_args()
    o, lse = attention_all(*args, causal, wl, 0.7)
    ob, lb = brute.attention(pb.q.double().numpy(), pb.k_cache.double().numpy(),
                             pb.v_cache.double().numpy(), pb.kv_indices.numpy(),
                             pb.qo_indptr.numpy(), pb.kv_indptr.numpy(),
                             pb.last_page_len.numpy(), P, causal, wl, 0.7)
    np.testing.assert_allclose(o, ob, atol=1e-12)
    np.testing.assert_allclose(lse, lb, atol=1e-12)


def test_oracle_rejects_indivisible_heads():
    with pytest.raises(ValueError):
        attention_rows(np.zeros((1, 3, 4), np.float32), np.zeros((1, 1, 2, 4), np.float32),
                       np.zeros((1, 1, 2, 4), np.float32), np.array([0], np.int32),
                       np.array([0, 1], np.int32), np.array([0, 1], np.int32),
                       np.array([1], np.int32), 1, False, -1, 1.0, np.array([0]),
                       np.array([0]))


# ------------------------------------------------------ custom (tree) masks
# A tree draft needs a topology mask: the causal one lets a draft attend to a
# sibling on another branch ("Support speculative-decode verify on ROCm, and
# stop auto routing short-query prefill to AITER" (#362), "Architecture /
# design notes"). The mask is ANDed into the causal / window mask.

def _mask_batch(seed, causal, n_req=3):
    """Tiny requests with random boolean masks (each row keeps >= 0 keys)."""
    rng = np.random.default_rng(seed)
    ql, kl, masks = [], [], []
    for _ in range(n_req):
        lk = int(rng.integers(1, 9))
        lq = int(rng.integers(1, lk + 1))
        ql.append(lq)
        kl.append(lk)
        masks.append(rng.random((lq, lk)) < 0.6)
    d, Hk, g = 5, 2, 2
    pb = workloads.make_paged_batch(ql, kl, g * Hk, Hk, d, 3, "bf16", seed + 7,
                                    extra_pool_pages=1)
    packed, indptr = workloads.pack_masks(masks)
    return pb, masks, packed, indptr


def test_custom_mask_bit_order():
    """Bit n of a request's segment is bit n % 8 of byte n / 8 (LSB first),
    segments start on their own byte."""
    m0 = np.zeros((3, 5), bool)
    m0[0, 0] = m0[1, 2] = m0[2, 4] = True  # bits 0, 7, 14
    m1 = np.zeros((1, 2), bool)
    m1[0, 1] = True                         # bit 1 of request 1's segment
    packed, indptr = workloads.pack_masks([m0, m1])
    assert list(indptr) == [0, 2, 3]
    assert list(packed) == [0b10000001, 0b01000000, 0b00000010]
    from oracle.reference import custom_bit
    for b, m in enumerate((m0, m1)):
        for i in range(m.shape[0]):
            for j in range(m.shape[1]):
                assert custom_bit(packed, indptr, b, i, j, m.shape[1]) == int(m[i, j])


@pytest.mark.parametrize("seed", range(5))
@pytest.mark.parametrize("causal,wl", [(False, -1), (True, -1), (True, 2), (False, 1)])
def test_custom_mask_c_oracle_agrees_with_brute_force(seed, causal, wl):
    """The C oracle (reads packed bits) and the brute force (dense booleans)
    agree with random masks ANDed into every causal / window combination."""
    pb, masks, packed, indptr = _mask_batch(200 + seed, causal)
    o, lse = attention_all(*pb.oracle_args(), causal, wl, 0.6, custom_mask=packed,
                           mask_indptr=indptr)
    ob, lb = brute.attention(pb.q.double().numpy(), pb.k_cache.double().numpy(),
                             pb.v_cache.double().numpy(), pb.kv_indices.numpy(),
                             pb.qo_indptr.numpy(), pb.kv_indptr.numpy(),
                             pb.last_page_len.numpy(), pb.page_size, causal, wl, 0.6,
                             custom=masks)
    np.testing.assert_allclose(o, ob, atol=1e-12)
    np.testing.assert_array_equal(np.isneginf(lse), np.isneginf(lb))
    fin = ~np.isneginf(lb)
    np.testing.assert_allclose(lse[fin], lb[fin], atol=1e-12)


def test_all_ones_mask_is_no_mask_and_causal_pattern_is_causal():
    pb, masks, _, _ = _mask_batch(300, True)
    args = pb.oracle_args()
    ones = [np.ones_like(m) for m in masks]
    p1, i1 = workloads.pack_masks(ones)
    for causal in (True, False):
        o0, l0 = attention_all(*args, causal, -1, 0.6)
        o1, l1 = attention_all(*args, causal, -1, 0.6, custom_mask=p1, mask_indptr=i1)
        np.testing.assert_array_equal(o0, o1)
        np.testing.assert_array_equal(l0, l1)
    # the bottom-right causal pattern as a custom mask on a non-causal plan
    cm = [np.array([[j <= i + m.shape[1] - m.shape[0] for j in range(m.shape[1])]
                    for i in range(m.shape[0])]) for m in masks]
    pc, ic = workloads.pack_masks(cm)
    o0, l0 = attention_all(*args, True, -1, 0.6)
    o1, l1 = attention_all(*args, False, -1, 0.6, custom_mask=pc, mask_indptr=ic)
    np.testing.assert_array_equal(o0, o1)
    np.testing.assert_array_equal(l0, l1)


def test_tree_mask_closed_form():
    """Constant keys under a tree mask: lse - s = ln(#keys the row sees), the
    prefix plus the node's depth + 1 (its ancestors and itself)."""
    parents = [-1, 0, 0, 1, 1, 2, 4]
    prefix = 5
    m = workloads.tree_masks(parents, prefix)
    depth = []
    for i in range(len(parents)):
        k, a = 0, i
        while a >= 0:
            k, a = k + 1, parents[a]
        depth.append(k)
    assert [int(r.sum()) for r in m] == [prefix + x for x in depth]
    lq, lk, d = len(parents), prefix + len(parents), 6
    rng = np.random.default_rng(5)
    q = rng.standard_normal((lq, 1, d)).astype(np.float32)
    kvec = rng.standard_normal(d).astype(np.float32)
    K = np.tile(kvec, (lk, 1, 1)).astype(np.float32)
    V = np.zeros((lk, 1, d), np.float32)
    V[:, 0, 0] = np.arange(lk)
    packed, indptr = workloads.pack_masks([m])
    kc = K.reshape(lk, 1, 1, d)
    vc = V.reshape(lk, 1, 1, d)
    o, lse = attention_all(q, kc, vc, np.arange(lk, dtype=np.int32),
                           np.array([0, lq], np.int32), np.array([0, lk], np.int32),
                           np.array([1], np.int32), 1, True, -1, 0.5, custom_mask=packed,
                           mask_indptr=indptr)
    for i in range(lq):
        s = 0.5 * float(np.dot(q[i, 0].astype(np.float64), kvec.astype(np.float64)))
        assert lse[i, 0] - s == pytest.approx(math.log(prefix + depth[i]), abs=1e-10)
        seen = np.nonzero(m[i])[0]
        assert o[i, 0, 0] == pytest.approx(seen.mean(), abs=1e-9)
