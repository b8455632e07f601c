"""Brute-force paged attention for tiny inputs (test infrastructure only).

A second, deliberately naive route to the same definition as the C oracle:
it copies each request's keys out of the page table into a dense matrix,
fills an explicit boolean mask matrix cell by cell from the two inequalities
of the pages (bottom-right causal bound, left-only window: "Route non-causal
windowed prefill to AITER's masked kernel", section "Why window_size_right
stays -1"), and applies a dense masked softmax with numpy. Inputs are float
arrays already holding the quantised values (float64 is fine).
"""
import numpy as np


def dense_kv(cache, kv_indices, kv_indptr, last_page_len, b, page_size):
    """Keys (or values) of request b as a dense [Lk, Hk, d] array."""
    pages = kv_indices[kv_indptr[b]:kv_indptr[b + 1]]
    if len(pages) == 0:
        return cache[:0, 0]
    rows = [cache[p] for p in pages]  # each [P, Hk, d]
    full = np.concatenate(rows, axis=0)
    lk = (len(pages) - 1) * page_size + int(last_page_len[b])
    return full[:lk]


def mask_matrix(lq, lk, causal, window_left):
    """Boolean [lq, lk] matrix, one cell at a time."""
    m = np.zeros((lq, lk), dtype=bool)
    for i in range(lq):
        for j in range(lk):
            ok = True
            if causal and not (j <= i + lk - lq):
                ok = False
            if window_left >= 0 and not (j + lq + window_left >= lk + i):
                ok = False
            m[i, j] = ok
    return m


def attention(q, k_cache, v_cache, kv_indices, qo_indptr, kv_indptr, last_page_len,
              page_size, causal, window_left, sm_scale, custom=None):
    """o [T, Hq, d] and natural-log lse [T, Hq], both float64. custom: per
    request a boolean [Lq, Lk] matrix ANDed into the mask (a tree topology),
    or None."""
    q = np.asarray(q, np.float64)
    k_cache = np.asarray(k_cache, np.float64)
    v_cache = np.asarray(v_cache, np.float64)
    T, Hq, d = q.shape
    Hk = k_cache.shape[2]
    g = Hq // Hk
    o = np.zeros((T, Hq, d))
    lse = np.full((T, Hq), -np.inf)
    for b in range(len(qo_indptr) - 1):
        q0, q1 = int(qo_indptr[b]), int(qo_indptr[b + 1])
        lq = q1 - q0
        K = dense_kv(k_cache, kv_indices, kv_indptr, last_page_len, b, page_size)
        V = dense_kv(v_cache, kv_indices, kv_indptr, last_page_len, b, page_size)
        lk = K.shape[0]
        if lq == 0:
            continue
        mask = mask_matrix(lq, lk, causal, window_left)
        if custom is not None:
            mask = mask & np.asarray(custom[b], dtype=bool)
        for h in range(Hq):
            S = sm_scale * (q[q0:q1, h, :] @ K[:, h // g, :].T)  # [lq, lk]
            for i in range(lq):
                sel = mask[i]
                if not sel.any():
                    continue
                s = S[i, sel]
                mx = s.max()
                w = np.exp(s - mx)
                tot = w.sum()
                lse[q0 + i, h] = mx + np.log(tot)
                o[q0 + i, h] = (w / tot) @ V[sel, h // g, :]
    return o, lse
