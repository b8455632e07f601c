"""Pins for the chain speculative-sampling oracle, against things other than
itself: numpy's searchsorted for the inverse-CDF draw, the special cases the
acceptance rule fixes, closed forms of the draw margin and the residual
fallback, and the defining property of speculative sampling
(Leviathan et al. 2023, Theorem 1): with the draft token drawn from q, the
first emitted token is distributed exactly as the target p.
"""
import numpy as np
import pytest

from oracle.speculative import (accept_draft, chain_speculative_sampling, draw_margin, residual,
                                sample_inverse_cdf)
import workloads


def test_inverse_cdf_matches_searchsorted():
    rng = np.random.default_rng(0)
    for _ in range(200):
        V = int(rng.integers(1, 40))
        w = rng.random(V)
        w[rng.random(V) < 0.3] = 0.0
        if w.sum() == 0:
            w[0] = 1.0
        u = float(rng.random())
        c = np.cumsum(w)
        want = int(np.searchsorted(c, u * c[-1], side="right"))
        assert sample_inverse_cdf(w, u) == min(want, V - 1)


def test_equal_draft_and_target_accept_every_draft():
    """p == q: u * q(x) <= q(x) for u < 1, so every draft is accepted and the
    bonus token comes from p_n (one-hot here, so it is known)."""
    B, n, V = 3, 4, 11
    rng = np.random.default_rng(1)
    p = rng.random((B, n + 1, V)).astype(np.float32)
    p /= p.sum(-1, keepdims=True)
    p[:, n] = 0
    p[:, n, 7] = 1
    q = p[:, :n].copy()
    ids = rng.integers(0, V, (B, n)).astype(np.int32)
    tok, acc, pos = chain_speculative_sampling(q, ids, p, rng.random((B, n)), rng.random(B))
    assert list(acc) == [n] * B and list(pos) == [n] * B
    assert np.array_equal(tok[:, :n], ids) and list(tok[:, n]) == [7] * B


def test_draft_the_target_rules_out_is_rejected():
    """p(x) = 0 < q(x): rejected at once for any u > 0; the draw comes from
    max(0, p - q), so it lands where p exceeds q."""
    V = 6
    q = np.array([[[0.5, 0.1, 0.1, 0.1, 0.1, 0.1]]], np.float32)
    p = np.array([[[0.0, 0.1, 0.6, 0.1, 0.2, 0.0], [1, 0, 0, 0, 0, 0]]], np.float32)
    for u in (0.01, 0.5, 0.99):
        tok, acc, pos = chain_speculative_sampling(q, np.array([[0]], np.int32), p,
                                                   np.array([[0.3]], np.float32), np.array([u]))
        assert acc[0] == 0 and pos[0] == 0 and tok[0, 1] == -1
        assert tok[0, 0] in (2, 4)  # the tokens where p > q
    r = residual(p[0, 0], q[0, 0])
    np.testing.assert_allclose(r, [0, 0, 0.5, 0, 0.1, 0], atol=1e-7)


def test_acceptance_rule_edge_cases():
    assert accept_draft(0.999, 0.2, 0.2)        # p == q
    assert not accept_draft(0.5, 0.4, 0.1)      # u > p / q
    assert accept_draft(0.25, 0.4, 0.1)         # u = p / q exactly (fp32 0.1 == 0.25 * 0.4)
    assert accept_draft(0.9, 0.1, 0.8)          # p > q always accepts


@pytest.mark.parametrize("seed", [0, 1])
def test_first_emitted_token_follows_the_target(seed):
    """Monte Carlo over x ~ q and uniform u: the first emitted token's
    frequencies match p_0 within 5 standard errors (a wrong residual, a
    reversed test or a dropped normalisation shifts them by far more)."""
    rng = np.random.default_rng(10 + seed)
    V, N = 5, 60000
    p0 = rng.random(V)
    p0[rng.integers(V)] = 0
    p0 /= p0.sum()
    q0 = rng.random(V)
    q0 /= q0.sum()
    p = np.stack([p0, np.full(V, 1.0 / V)])[None].astype(np.float32)
    q = q0[None, None].astype(np.float32)
    counts = np.zeros(V)
    cq = np.cumsum(q0)
    for _ in range(N):
        x = min(int(np.searchsorted(cq, rng.random() * cq[-1], side="right")), V - 1)
        tok, _, _ = chain_speculative_sampling(q, np.array([[x]], np.int32), p,
                                               rng.random((1, 1)).astype(np.float32),
                                               np.array([rng.random()]))
        counts[tok[0, 0]] += 1
    freq = counts / N
    se = np.sqrt(np.maximum(p0 * (1 - p0), 1e-12) / N)
    assert np.all(np.abs(freq - p0) <= 5 * se + 1e-9), (freq, p0)


def test_generator_shapes_and_rows_are_distributions():
    d = workloads.spec_sampling_batch(batch=3, n_draft=2, vocab=50)
    assert tuple(d["target_probs"].shape) == (3, 3, 50)
    assert tuple(d["draft_probs"].shape) == (3, 2, 50)
    np.testing.assert_allclose(d["target_probs"].double().sum(-1).numpy(), 1.0, atol=1e-5)
    np.testing.assert_allclose(d["draft_probs"].double().sum(-1).numpy(), 1.0, atol=1e-5)
    assert int(d["draft_ids"].max()) < 50


def test_draw_margin_closed_forms():
    """Weights [1, 1, 2] have cumulative fractions 0.25, 0.5, 1: the margin of
    u is its distance to the nearest of them (an off-by-one cumsum or a
    missing normalisation moves these values)."""
    w = [1.0, 1.0, 2.0]
    assert draw_margin(w, 0.25) == 0.0
    assert abs(draw_margin(w, 0.3) - 0.05) < 1e-15
    assert abs(draw_margin(w, 0.45) - 0.05) < 1e-15
    assert abs(draw_margin(w, 0.8) - 0.2) < 1e-15
    assert abs(draw_margin(w, 0.0) - 0.25) < 1e-15
    assert draw_margin([0.0, 0.0], 0.5) == np.inf  # no mass: no boundary


def test_draw_margin_zero_only_on_a_boundary():
    """Brute force: the margin is zero exactly where the inverse-CDF draw
    switches token, and a draw with margin m does not change for any u'
    within m of u."""
    rng = np.random.default_rng(5)
    w = rng.random(9) + 0.05
    us = np.linspace(0.0, 0.999, 400)
    for u in us:
        m = draw_margin(w, u)
        t = sample_inverse_cdf(w, u)
        for du in (-0.9 * m, 0.9 * m):
            uu = min(max(u + du, 0.0), 0.999999)
            if m > 1e-12:
                assert sample_inverse_cdf(w, uu) == t


def test_residual_falls_back_to_the_target_when_all_zero():
    """q >= p everywhere (here q == p): max(0, p - q) has no mass, so the draw
    uses p itself; otherwise the residual is max(0, p - q) elementwise."""
    p = np.array([0.1, 0.6, 0.3], np.float32)
    assert np.array_equal(residual(p, p), p)
    q = np.array([0.5, 0.5, 0.0], np.float32)
    r = residual(p, q)
    assert np.array_equal(r, np.array([0.0, np.float32(0.6) - np.float32(0.5), 0.3], np.float32))
    # a full chain through the fallback: draft = target, u_accept above 1 so
    # the first draft is rejected; the draw must then follow p_0 (one-hot)
    V = 5
    tp = np.zeros((1, 2, V), np.float32)
    tp[0, :, 3] = 1.0
    dp = tp[:, :1].copy()
    toks, acc, pos = chain_speculative_sampling(dp, np.array([[3]]), tp,
                                                np.array([[1.5]], np.float32),
                                                np.array([0.4], np.float32))
    assert acc[0] == 0 and pos[0] == 0 and toks[0, 0] == 3 and toks[0, 1] == -1
