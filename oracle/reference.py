"""ctypes wrapper around the fp64 C oracle (test infrastructure only).

Inputs are numpy arrays. 16-bit floating inputs are passed as their raw bits
(``uint16``/``int16`` views of fp16 or bf16) together with a dtype name, so the
oracle reads exactly the quantised values the GPU reads.
"""
import ctypes
import numpy as np

from .build import build_oracle, build_oracle_fp32omp

_DT = {"f16": 0, "bf16": 1, "f32": 2}
_lib = None
_lib_fast = None


def _bind(lib):
    P = ctypes.c_void_p
    i32, i64, dbl = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
    lib.oracle_attention_rows.restype = ctypes.c_int
    lib.oracle_attention_rows.argtypes = [
        P, ctypes.c_int, P, P, ctypes.c_int, P, P, P, P, i32, i32, i32, i32, i32,
        ctypes.c_int, i32, dbl, i64, P, P, P, P, P, P]
    lib.oracle_custom_bit.restype = ctypes.c_int
    lib.oracle_custom_bit.argtypes = [P, P, i32, i64, i64, i64]
    lib.oracle_merge_states.restype = None
    lib.oracle_merge_states.argtypes = [P, P, i64, i64, i64, P, P]
    lib.oracle_kv_len.restype = i64
    lib.oracle_kv_len.argtypes = [P, P, i32, i32]
    lib.oracle_key_valid.restype = ctypes.c_int
    lib.oracle_key_valid.argtypes = [i64, i64, i64, i64, ctypes.c_int, i64]
    lib.oracle_set_threads.restype = None
    lib.oracle_set_threads.argtypes = [ctypes.c_int]
    lib.oracle_threads.restype = ctypes.c_int
    lib.oracle_threads.argtypes = []
    lib.oracle_acc_is_float.restype = ctypes.c_int
    lib.oracle_acc_is_float.argtypes = []
    return lib


def _load():
    """The fp64 parity build."""
    global _lib
    if _lib is None:
        _lib = _bind(ctypes.CDLL(build_oracle()))
    return _lib


def _load_fast():
    """The fp32-accumulate OpenMP build of the same source (timed baseline)."""
    global _lib_fast
    if _lib_fast is None:
        _lib_fast = _bind(ctypes.CDLL(build_oracle_fp32omp()))
    return _lib_fast


def fp32omp_threads(n=None):
    """Set (when n is given) and return the thread count of the timed build."""
    lib = _load_fast()
    if n is not None:
        lib.oracle_set_threads(int(n))
    return int(lib.oracle_threads())


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dt):
    return np.ascontiguousarray(a, dtype=dt)


def kv_len(kv_indptr, last_page_len, b, page_size):
    kv_indptr = _c(kv_indptr, np.int32)
    last_page_len = _c(last_page_len, np.int32)
    return _load().oracle_kv_len(_ptr(kv_indptr), _ptr(last_page_len), b, page_size)


def key_valid(i, j, lq, lk, causal, window_left):
    return bool(_load().oracle_key_valid(i, j, lq, lk, int(causal), window_left))


def _as_raw(a, dtype):
    """(contiguous array, oracle dtype name) for a float32, float16 or raw-bits array."""
    if a.dtype == np.float32:
        return _c(a, np.float32), "f32"
    if a.dtype == np.float16:
        return _c(a.view(np.uint16), np.uint16), "f16"
    if a.dtype in (np.uint16, np.int16):
        return _c(a.view(np.uint16), np.uint16), dtype
    raise TypeError("unsupported oracle input dtype %s" % a.dtype)


def custom_bit(custom_mask, mask_indptr, b, i, j, lk):
    """Bit (i * lk + j) of request b's packed custom mask, as the oracle reads it."""
    custom_mask = _c(custom_mask, np.uint8)
    mask_indptr = _c(mask_indptr, np.int64)
    return _load().oracle_custom_bit(_ptr(custom_mask), _ptr(mask_indptr), b, i, j, lk)


def attention_rows(q, k_cache, v_cache, kv_indices, qo_indptr, kv_indptr, last_page_len,
                   page_size, causal, window_left, sm_scale, sel_token, sel_head,
                   dtype="bf16", custom_mask=None, mask_indptr=None, fp32omp=False):
    """fp64 (o [n, d], lse [n]) for rows (sel_token[r], sel_head[r]).
    fp32omp=True runs the timed baseline build instead (fp32 accumulation,
    OpenMP over the rows); its results are not the parity oracle's.

    q [T, Hq, d]; k_cache/v_cache [num_pages, P, Hk, d]. Arrays are float32,
    float16, or uint16/int16 raw bits of ``dtype`` ("bf16" or "f16").
    custom_mask (uint8, bit-packed per request) / mask_indptr (byte offsets,
    [batch + 1]): a mask ANDed into the causal / window mask, or None.
    """
    q, q_dt = _as_raw(q, dtype)
    k_cache, kv_dt = _as_raw(k_cache, dtype)
    v_cache, v_dt = _as_raw(v_cache, dtype)
    assert kv_dt == v_dt
    assert q.ndim == 3 and k_cache.ndim == 4 and v_cache.shape == k_cache.shape
    T, Hq, d = q.shape
    _, P, Hk, d2 = k_cache.shape
    assert d == d2 and P == page_size
    kv_indices = _c(kv_indices, np.int32)
    qo_indptr = _c(qo_indptr, np.int32)
    kv_indptr = _c(kv_indptr, np.int32)
    last_page_len = _c(last_page_len, np.int32)
    sel_token = _c(sel_token, np.int64)
    sel_head = _c(sel_head, np.int32)
    n = sel_token.shape[0]
    o = np.zeros((n, d), np.float64)
    lse = np.zeros((n,), np.float64)
    cm = mi = None
    if custom_mask is not None:
        cm = _c(custom_mask, np.uint8)
        mi = _c(mask_indptr, np.int64)
    lib = _load_fast() if fp32omp else _load()
    rc = lib.oracle_attention_rows(
        _ptr(q), _DT[q_dt], _ptr(k_cache), _ptr(v_cache), _DT[kv_dt], _ptr(kv_indices),
        _ptr(qo_indptr), _ptr(kv_indptr), _ptr(last_page_len), len(qo_indptr) - 1,
        page_size, Hq, Hk, d, int(bool(causal)), int(window_left), float(sm_scale), n,
        _ptr(sel_token), _ptr(sel_head), _ptr(o), _ptr(lse),
        _ptr(cm) if cm is not None else None, _ptr(mi) if mi is not None else None)
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    return o, lse


def attention_all(q, k_cache, v_cache, kv_indices, qo_indptr, kv_indptr, last_page_len,
                  page_size, causal, window_left, sm_scale, dtype="bf16", custom_mask=None,
                  mask_indptr=None):
    """fp64 o [T, Hq, d] and lse [T, Hq] for every row."""
    T, Hq, d = q.shape
    tok = np.repeat(np.arange(T, dtype=np.int64), Hq)
    head = np.tile(np.arange(Hq, dtype=np.int32), T)
    o, lse = attention_rows(q, k_cache, v_cache, kv_indices, qo_indptr, kv_indptr,
                            last_page_len, page_size, causal, window_left, sm_scale,
                            tok, head, dtype, custom_mask, mask_indptr)
    return o.reshape(T, Hq, d), lse.reshape(T, Hq)


def merge_states(v, s):
    """Merge states along axis 1: v [rows, n, d], s [rows, n] -> ([rows, d], [rows])."""
    v = _c(v, np.float64)
    s = _c(s, np.float64)
    rows, n, d = v.shape
    vo = np.zeros((rows, d), np.float64)
    so = np.zeros((rows,), np.float64)
    _load().oracle_merge_states(_ptr(v), _ptr(s), rows, n, d, _ptr(vo), _ptr(so))
    return vo, so
