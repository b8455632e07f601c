"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module holds no attention arithmetic: it only draws lengths, page tables
and N(0, 1) tensors. Both the CUDA path and the CPU oracle read what it makes.

Recipe:
  * ``numpy.random.default_rng(seed)``, seed = 20261202 + 100 * config + variant;
  * q, k, v ~ N(0, 1) drawn in fp32, then cast (round-to-nearest-even) to the
    run's dtype; everybody reads the cast values;
  * integer lengths uniform over the inclusive range;
  * the page pool holds exactly the pages the batch needs, and ``kv_indices`` is
    a seeded permutation of that pool, so consecutive keys of a request land in
    scattered pages;
  * sm_scale = 1 / sqrt(head_dim).

The workloads follow the shapes of the pages' own measurements (AMD-Ecosystem
FlashInfer PRs #339, #362, #399): a 64x256 GQA-2 paged prefill, a batch-64
decode over mixed lengths, 4-row speculative verify, batch prefill with
prefixes and windows, and long-context short-query split-KV.
"""
from dataclasses import dataclass, field
from typing import List, Optional

import numpy as np
import torch

BASE_SEED = 20261202

TORCH_DTYPE = {"bf16": torch.bfloat16, "f16": torch.float16}


def seed_for(config: int, variant: int = 0) -> int:
    return BASE_SEED + 100 * config + variant


@dataclass
class PagedBatch:
    """One synthetic batch (CPU tensors) in the library's layouts.

    q [T, Hq, d]; k_cache, v_cache [num_pages, P, Hk, d] (NHD);
    qo_indptr, kv_indptr [B+1], last_page_len [B], kv_indices [kv_indptr[B]]
    are int32.
    """
    q: torch.Tensor
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    kv_indices: torch.Tensor
    qo_indptr: torch.Tensor
    kv_indptr: torch.Tensor
    last_page_len: torch.Tensor
    q_lens: List[int]
    kv_lens: List[int]
    page_size: int
    num_qo_heads: int
    num_kv_heads: int
    head_dim: int
    dtype: str
    sm_scale: float
    extra: dict = field(default_factory=dict)

    def raw(self, t: torch.Tensor) -> np.ndarray:
        """Raw 16-bit pattern of a 16-bit tensor (what the oracle reads)."""
        if t.dtype in (torch.bfloat16, torch.float16):
            return t.contiguous().view(torch.int16).numpy().view(np.uint16)
        return t.contiguous().numpy()

    def oracle_args(self):
        """Positional inputs for the oracle's attention functions."""
        return (self.raw(self.q), self.raw(self.k_cache), self.raw(self.v_cache),
                self.kv_indices.numpy(), self.qo_indptr.numpy(), self.kv_indptr.numpy(),
                self.last_page_len.numpy(), self.page_size)


def _normal(rng, shape, dtype):
    x = rng.standard_normal(size=shape, dtype=np.float32)
    return torch.from_numpy(x).to(TORCH_DTYPE[dtype])


def make_paged_batch(q_lens, kv_lens, num_qo_heads, num_kv_heads, head_dim, page_size,
                     dtype, seed, permute_pages=True, extra_pool_pages=0) -> PagedBatch:
    """Random q and a randomly paged K/V cache for the given lengths."""
    rng = np.random.default_rng(seed)
    q_lens = [int(x) for x in q_lens]
    kv_lens = [int(x) for x in kv_lens]
    B = len(q_lens)
    assert len(kv_lens) == B
    pages_per_req = [(lk + page_size - 1) // page_size for lk in kv_lens]
    total_pages = sum(pages_per_req)
    pool = total_pages + extra_pool_pages
    kv_indptr = np.zeros(B + 1, np.int32)
    kv_indptr[1:] = np.cumsum(pages_per_req)
    qo_indptr = np.zeros(B + 1, np.int32)
    qo_indptr[1:] = np.cumsum(q_lens)
    last = np.array([(lk - (n - 1) * page_size) if n > 0 else 0
                     for lk, n in zip(kv_lens, pages_per_req)], np.int32)
    if permute_pages:
        indices = rng.permutation(pool)[:total_pages].astype(np.int32)
    else:
        indices = np.arange(total_pages, dtype=np.int32)
    T = int(qo_indptr[-1])
    q = _normal(rng, (T, num_qo_heads, head_dim), dtype)
    k = _normal(rng, (max(pool, 1), page_size, num_kv_heads, head_dim), dtype)
    v = _normal(rng, (max(pool, 1), page_size, num_kv_heads, head_dim), dtype)
    return PagedBatch(q=q, k_cache=k, v_cache=v, kv_indices=torch.from_numpy(indices),
                      qo_indptr=torch.from_numpy(qo_indptr),
                      kv_indptr=torch.from_numpy(kv_indptr),
                      last_page_len=torch.from_numpy(last), q_lens=q_lens, kv_lens=kv_lens,
                      page_size=page_size, num_qo_heads=num_qo_heads,
                      num_kv_heads=num_kv_heads, head_dim=head_dim, dtype=dtype,
                      sm_scale=1.0 / float(np.sqrt(head_dim)))


# ---------------------------------------------------------------------------
# The five workloads. Each returns a PagedBatch; its run options (causal,
# window_left, ...) are listed by the matching *_CASES table.
# ---------------------------------------------------------------------------

def pr1_reference(variant: int = 0) -> PagedBatch:
    """Single-request paged prefill: qo_len 64, kv_len 256, 4 q / 2 kv heads,
    head_dim 64, fp16, page 16, 16 pages in seeded random order."""
    return make_paged_batch([64], [256], 4, 2, 64, 16, "f16", seed_for(1, variant))


PR1_CASES = [dict(causal=c, window_left=w) for c in (True, False) for w in (-1, 31)]


def batch_decode(variant: int = 0, batch: int = 64, kv_lo: int = 512, kv_hi: int = 8192,
                 num_qo_heads: int = 32, num_kv_heads: int = 8, head_dim: int = 128,
                 page_size: int = 16, dtype: str = "bf16") -> PagedBatch:
    """Batch decode: one query row per request, kv_len uniform in [kv_lo, kv_hi]."""
    rng = np.random.default_rng(seed_for(2, variant) + 7)
    kv = rng.integers(kv_lo, kv_hi + 1, size=batch)
    return make_paged_batch([1] * batch, kv, num_qo_heads, num_kv_heads, head_dim,
                            page_size, dtype, seed_for(2, variant))


def speculative_verify(batch: int = 32, variant: int = 0, q_len_per_req: int = 4,
                       kv_lo: int = 1024, kv_hi: int = 4096, num_qo_heads: int = 32,
                       num_kv_heads: int = 8, head_dim: int = 128, page_size: int = 16,
                       dtype: str = "bf16") -> PagedBatch:
    """Verify: q_len_per_req draft rows per request; kv_len includes the drafts."""
    rng = np.random.default_rng(seed_for(3, variant) + 7 + batch)
    kv = rng.integers(kv_lo, kv_hi + 1, size=batch)
    pb = make_paged_batch([q_len_per_req] * batch, kv, num_qo_heads, num_kv_heads,
                          head_dim, page_size, dtype, seed_for(3, variant) + batch)
    pb.extra["q_len_per_req"] = q_len_per_req
    return pb


def batch_prefill(page_size: int = 16, variant: int = 0, batch: int = 16,
                  q_lo: int = 512, q_hi: int = 2048, prefix_lo: int = 0,
                  prefix_hi: int = 4096, num_qo_heads: int = 32, num_kv_heads: int = 8,
                  head_dim: int = 128, dtype: str = "bf16") -> PagedBatch:
    """Batch paged prefill: qo_len uniform, kv_len = qo_len + uniform prefix."""
    rng = np.random.default_rng(seed_for(4, variant) + 7)
    ql = rng.integers(q_lo, q_hi + 1, size=batch)
    pre = rng.integers(prefix_lo, prefix_hi + 1, size=batch)
    return make_paged_batch(ql, ql + pre, num_qo_heads, num_kv_heads, head_dim, page_size,
                            dtype, seed_for(4, variant) + page_size)


def batch_prefill_hd64(page_size: int = 16, variant: int = 0) -> PagedBatch:
    """The batch-prefill lengths at head_dim 64, 4 q / 2 kv heads, fp16."""
    return batch_prefill(page_size=page_size, variant=variant, num_qo_heads=4, num_kv_heads=2,
                         head_dim=64, dtype="f16")


def ragged_prefill(variant: int = 0, batch: int = 16, q_lo: int = 512, q_hi: int = 2048,
                   prefix_lo: int = 0, prefix_hi: int = 4096, num_qo_heads: int = 32,
                   num_kv_heads: int = 8, head_dim: int = 128, dtype: str = "bf16") -> PagedBatch:
    """The batch-prefill shapes over contiguous K/V: a page-size-1 cache with
    an unpermuted page table, whose rows are the ragged K/V in request order
    (k_cache.reshape(rows, Hk, d)); kv_indptr is then each request's first row."""
    rng = np.random.default_rng(seed_for(4, variant) + 7)
    ql = rng.integers(q_lo, q_hi + 1, size=batch)
    pre = rng.integers(prefix_lo, prefix_hi + 1, size=batch)
    return make_paged_batch(ql, ql + pre, num_qo_heads, num_kv_heads, head_dim, 1, dtype,
                            seed_for(4, variant) + 1, permute_pages=False)


def pack_masks(masks):
    """Bit-pack per-request boolean [Lq, Lk] masks: request b's bits (row-major,
    i * Lk + j) start on byte mask_indptr[b], least significant bit first.
    Returns (uint8 array, int32 byte offsets [batch + 1])."""
    segs = [np.packbits(np.asarray(m, dtype=np.uint8).reshape(-1), bitorder="little")
            for m in masks]
    indptr = np.zeros(len(segs) + 1, np.int32)
    indptr[1:] = np.cumsum([len(x) for x in segs])
    data = np.concatenate(segs) if segs else np.zeros(0, np.uint8)
    if data.size == 0:
        data = np.zeros(1, np.uint8)  # never empty, so it always has an address
    return data.astype(np.uint8), indptr


def tree_masks(parents, prefix_len):
    """Topology mask of one request's draft tree: row i (draft node i) sees
    every prefix key and the keys of its ancestors and itself; parents[i] < i
    (parents[0] = -1, the root under the prefix)."""
    n = len(parents)
    m = np.zeros((n, prefix_len + n), dtype=bool)
    m[:, :prefix_len] = True
    for i in range(n):
        a = i
        while a >= 0:
            m[i, prefix_len + a] = True
            a = parents[a]
    return m


def tree_verify(batch: int = 32, variant: int = 0, n_draft: int = 8, kv_lo: int = 1024,
                kv_hi: int = 4096, num_qo_heads: int = 32, num_kv_heads: int = 8,
                head_dim: int = 128, page_size: int = 16, dtype: str = "bf16") -> PagedBatch:
    """Tree verify: n_draft draft nodes per request with random parents
    (node i's parent uniform in [0, i)), kv_len = prefix + n_draft; the
    topology masks are in extra["masks"] (dense) and packed in
    extra["mask"] / extra["mask_indptr"]."""
    rng = np.random.default_rng(seed_for(6, variant) + batch)
    kv = rng.integers(kv_lo, kv_hi + 1, size=batch)
    masks = []
    for b in range(batch):
        parents = [-1] + [int(rng.integers(0, i)) for i in range(1, n_draft)]
        masks.append(tree_masks(parents, int(kv[b]) - n_draft))
    pb = make_paged_batch([n_draft] * batch, kv, num_qo_heads, num_kv_heads, head_dim,
                          page_size, dtype, seed_for(6, variant) + 3 * batch)
    packed, indptr = pack_masks(masks)
    pb.extra["masks"] = masks
    pb.extra["mask"] = torch.from_numpy(packed)
    pb.extra["mask_indptr"] = torch.from_numpy(indptr)
    return pb


def spec_sampling_batch(batch: int = 64, n_draft: int = 4, vocab: int = 128256,
                        variant: int = 0, temperature: float = 0.7, draft_noise: float = 0.5):
    """Inputs of the chain speculative-sampling step: target probabilities
    [B, n+1, V] (softmax of N(0,1) logits / temperature, fp32), draft
    probabilities [B, n, V] (the same logits plus N(0, draft_noise) noise), draft
    tokens drawn from the draft rows, and the uniforms of the acceptance tests
    [B, n] and of the final draw [B]. Returns a dict of CPU torch tensors."""
    rng = np.random.default_rng(seed_for(7, variant) + batch + n_draft)
    logits = rng.standard_normal((batch, n_draft + 1, vocab), dtype=np.float32)
    noise = rng.standard_normal((batch, n_draft, vocab), dtype=np.float32) * draft_noise

    def softmax(x):
        x = x / temperature
        x = x - x.max(axis=-1, keepdims=True)
        e = np.exp(x)
        return (e / e.sum(axis=-1, keepdims=True)).astype(np.float32)

    target = softmax(logits)
    draft = softmax(logits[:, :n_draft] + noise)
    ids = np.zeros((batch, n_draft), np.int32)
    for b in range(batch):
        for i in range(n_draft):
            c = np.cumsum(draft[b, i].astype(np.float64))
            ids[b, i] = min(int(np.searchsorted(c, rng.random() * c[-1], side="right")), vocab - 1)
    u_accept = rng.random((batch, n_draft), dtype=np.float32)
    u_sample = rng.random(batch, dtype=np.float32)
    return {"draft_probs": torch.from_numpy(draft), "draft_ids": torch.from_numpy(ids),
            "target_probs": torch.from_numpy(target), "u_accept": torch.from_numpy(u_accept),
            "u_sample": torch.from_numpy(u_sample)}


PREFILL_CASES = ([dict(causal=True, window_left=w) for w in (-1, 0, 127, 4095)]
                 + [dict(causal=False, window_left=w) for w in (-1, 127)])


def long_context(variant: int = 0, batch: int = 8, qo_len: int = 16, kv_len: int = 32768,
                 num_qo_heads: int = 64, num_kv_heads: int = 8, head_dim: int = 128,
                 page_size: int = 16, dtype: str = "bf16") -> PagedBatch:
    """Long-context short-query batch for split-KV (GQA 8)."""
    return make_paged_batch([qo_len] * batch, [kv_len] * batch, num_qo_heads, num_kv_heads,
                            head_dim, page_size, dtype, seed_for(5, variant))


# {causal, 127} and {non-causal, 127} are the workload's two cases; the
# unwindowed causal case is added as the bandwidth-bound split-KV stress case.
LONG_CONTEXT_CASES = [dict(causal=True, window_left=127), dict(causal=False, window_left=127),
                      dict(causal=True, window_left=-1)]
LONG_CONTEXT_CHUNKS = (8, 16, 32)


def sample_rows(pb: PagedBatch, n: int, seed: int, must_include: Optional[list] = None):
    """A seeded sample of (token, head) rows, always including each request's
    first and last row and any rows in ``must_include``."""
    rng = np.random.default_rng(seed)
    T = int(pb.qo_indptr[-1])
    Hq = pb.num_qo_heads
    toks = list(rng.integers(0, T, size=n))
    heads = list(rng.integers(0, Hq, size=n))
    qo = pb.qo_indptr.numpy()
    for b in range(len(qo) - 1):
        if qo[b + 1] > qo[b]:
            for t in (qo[b], qo[b + 1] - 1):
                toks.append(int(t))
                heads.append(int(rng.integers(0, Hq)))
    for t, h in (must_include or []):
        toks.append(int(t))
        heads.append(int(h))
    return np.array(toks, np.int64), np.array(heads, np.int32)
