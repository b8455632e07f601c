"""Chain speculative sampling on the GPU against the oracle.

The acceptance decisions are taken in fp32 on both sides, so the accepted
prefix must match exactly. The final draw picks a token from a cumulative
sum: where u * total lies farther than 1e-5 (relative) from a cumulative
boundary the token must match exactly; closer than that the two summation
orders may legitimately pick a neighbour, so the kernel's token is checked
to be a valid draw instead (positive weight, and its cumulative range
within 1e-5 of the target).
"""
import numpy as np
import pytest
import torch

import workloads
from oracle.speculative import chain_speculative_sampling, draw_margin, residual

pytestmark = pytest.mark.gpu

TOL = 1e-5


def run(d):
    import paged_kv_attention_13_gb300 as fi
    dev = {k: (v if v.is_cuda else v.cuda()) for k, v in d.items()}
    tok, acc, emi = fi.fi_chain_speculative_sampling(dev["draft_probs"], dev["draft_ids"],
                                                     dev["target_probs"], dev["u_accept"],
                                                     dev["u_sample"])
    torch.cuda.synchronize()
    return tok.cpu().numpy(), acc.cpu().numpy(), emi.cpu().numpy()


def check(d, tok, acc, emi):
    dp = d["draft_probs"].numpy()
    tp = d["target_probs"].numpy()
    t_ref, a_ref, pos = chain_speculative_sampling(dp, d["draft_ids"].numpy(), tp,
                                                   d["u_accept"].numpy(), d["u_sample"].numpy())
    n = tp.shape[1] - 1
    np.testing.assert_array_equal(acc, a_ref)
    np.testing.assert_array_equal(emi, a_ref + 1)
    for b in range(tp.shape[0]):
        a = int(a_ref[b])
        np.testing.assert_array_equal(tok[b, :a], t_ref[b, :a])
        assert np.all(tok[b, a + 1:] == -1)
        w = tp[b, n] if a == n else residual(tp[b, a], dp[b, a])
        u = float(d["u_sample"][b])
        if draw_margin(w, u) > TOL:
            assert tok[b, a] == t_ref[b, a], (b, tok[b, a], t_ref[b, a])
        else:  # a boundary draw: any valid neighbour
            t = int(tok[b, a])
            w64 = np.asarray(w, np.float64)
            c = np.cumsum(w64) / w64.sum()
            assert w64[t] > 0
            assert (c[t - 1] if t > 0 else 0.0) <= u + TOL and c[t] >= u - TOL


@pytest.mark.parametrize("vocab", [128256, 32000, 50257, 7, 1])
@pytest.mark.parametrize("n", [0, 1, 4, 40])
def test_against_oracle(vocab, n):
    d = workloads.spec_sampling_batch(batch=24, n_draft=n, vocab=vocab, variant=vocab % 7)
    check(d, *run(d))


def test_equal_draft_and_target_accept_all():
    d = workloads.spec_sampling_batch(batch=8, n_draft=5, vocab=1000)
    d["draft_probs"] = d["target_probs"][:, :5].clone()
    tok, acc, emi = run(d)
    assert np.all(acc == 5)
    check(d, tok, acc, emi)


def test_forced_rejection_and_zero_residual_fallback():
    d = workloads.spec_sampling_batch(batch=6, n_draft=3, vocab=4096, variant=3)
    tp = d["target_probs"].clone()
    ids = d["draft_ids"]
    for b in range(3):  # the target rules out the first draft: rejected at once
        tp[b, 0, ids[b, 0]] = 0.0
    # requests 3..5: an unnormalised target below the draft everywhere at row 0,
    # so the residual is all zero and the draw falls back to the target row
    for b in range(3, 6):
        tp[b, 0] = d["draft_probs"][b, 0] * 0.5
        d["u_accept"][b, 0] = 0.9
    d["target_probs"] = tp
    tok, acc, emi = run(d)
    assert np.all(acc == 0)
    check(d, tok, acc, emi)


def test_strided_probability_rows():
    """Rows taken from wider tensors (non-packed batch / position strides)."""
    d = workloads.spec_sampling_batch(batch=5, n_draft=2, vocab=2048, variant=5)
    wide_t = torch.zeros((5, 4, 2048 + 64))
    wide_t[:, :3, :2048] = d["target_probs"]
    wide_d = torch.zeros((5, 3, 2048 + 64))
    wide_d[:, :2, :2048] = d["draft_probs"]
    e = dict(d)
    e["target_probs"] = wide_t.cuda()[:, :3, :2048]  # sliced on the device: strides kept
    e["draft_probs"] = wide_d.cuda()[:, :2, :2048]
    assert not e["target_probs"].is_contiguous()
    tok, acc, emi = run(e)
    check(d, tok, acc, emi)
