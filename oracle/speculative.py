"""Oracle for the chain speculative-sampling acceptance step (test
infrastructure only: the tests, the smoke check and the benchmark's CPU leg
call it; the product never does).

The step consumes the verify pass of a chain of n draft tokens per request
("Support speculative-decode verify on ROCm, and stop auto routing
short-query prefill to AITER" (#362), "Summary": the acceptance sampler
chain_speculative_sampling is fed by the multi-token verify; "Architecture /
design notes": it takes (batch_size, num_speculate_tokens), a chain, not a
tree). The pages give no formula; the steps here are the published
speculative sampling of Leviathan, Kalman and Matias (2023) and Chen et al.
(2023), in their order:

  for i = 0 .. n-1, draft token x_i with draft probability q_i(x_i) and
  target probability p_i(x_i): accept it while u_i * q_i(x_i) <= p_i(x_i)
  (the test u_i <= p/q without a division; product and compare in fp32, the
  precision the kernel decides in). At the first rejection i, draw one token
  from the residual max(0, p_i - q_i) (normalised; p_i itself if the residual
  is all zero). If all n are accepted, draw the bonus token from p_n. A draw
  with uniform u from weights w picks the smallest token t whose cumulative
  weight exceeds u * sum(w).

Outputs per request: tokens [n + 1] = the accepted drafts, the drawn token,
then -1; accepted = the number of drafts accepted before the first rejection
(the tokens emitted are accepted + 1).
"""
import numpy as np


def sample_inverse_cdf(w, u):
    """Smallest t with sum(w[:t+1]) > u * sum(w), in fp64, by a plain loop
    (the last token with positive weight if rounding leaves none)."""
    w = np.asarray(w, np.float64)
    total = float(w.sum())
    target = float(u) * total
    acc = 0.0
    last = -1
    for t in range(w.shape[0]):
        if w[t] > 0:
            last = t
        acc += w[t]
        if acc > target:
            return t
    return last


def accept_draft(u, q_x, p_x):
    """The acceptance test u * q(x) <= p(x), product and compare in fp32."""
    return bool(np.float32(u) * np.float32(q_x) <= np.float32(p_x))


def residual(p, q):
    """max(0, p - q) in fp32 (the kernel's precision); p if it is all zero."""
    r = np.maximum(np.float32(0), np.asarray(p, np.float32) - np.asarray(q, np.float32))
    return r if float(r.astype(np.float64).sum()) > 0 else np.asarray(p, np.float32)


def chain_speculative_sampling(draft_probs, draft_ids, target_probs, u_accept, u_sample):
    """draft_probs [B, n, V], draft_ids [B, n], target_probs [B, n+1, V],
    u_accept [B, n], u_sample [B] -> (tokens [B, n+1] int32, accepted [B]
    int32, position [B] int32: the row whose distribution was drawn from)."""
    draft_probs = np.asarray(draft_probs, np.float32)
    target_probs = np.asarray(target_probs, np.float32)
    B, n, V = draft_probs.shape
    tokens = np.full((B, n + 1), -1, np.int32)
    accepted = np.zeros(B, np.int32)
    position = np.zeros(B, np.int32)
    for b in range(B):
        i = 0
        while i < n:
            x = int(draft_ids[b, i])
            if not accept_draft(u_accept[b, i], draft_probs[b, i, x], target_probs[b, i, x]):
                break
            tokens[b, i] = x
            i += 1
        accepted[b] = i
        position[b] = i
        w = target_probs[b, n] if i == n else residual(target_probs[b, i], draft_probs[b, i])
        tokens[b, i] = sample_inverse_cdf(w, u_sample[b])
    return tokens, accepted, position


def draw_margin(w, u):
    """How far u * sum(w) lies from the nearest cumulative-weight boundary,
    relative to sum(w) (fp64): draws closer than rounding to a boundary may
    legitimately land on either neighbour in another summation order."""
    w = np.asarray(w, np.float64)
    total = w.sum()
    if total <= 0:
        return np.inf
    c = np.cumsum(w) / total
    return float(np.min(np.abs(c - float(u))))
