"""Python binding of libfi with the C ABI's names (argument marshalling only).

Every computation happens in libfi's CUDA kernels; this module turns torch
tensors into ``fi_tensor`` descriptors, passes the current CUDA stream, and
raises ``FiError`` with the library's message on any non-OK status.
"""
import ctypes
import struct

import numpy as np
import torch

from . import _lib
from ._lib import FiPlanInfo, FiTensor

_DTYPES = {torch.float16: _lib.FI_F16, torch.bfloat16: _lib.FI_BF16,
           torch.float32: _lib.FI_F32, torch.int32: _lib.FI_I32, torch.uint8: _lib.FI_U8}

KERNEL_NAMES = {0: "decode", 1: "prefill_m16", 2: "prefill_m64", 3: "prefill_m128"}


class FiError(RuntimeError):
    """A refusal or failure reported by libfi."""

    def __init__(self, status: int, message: str):
        self.status = status
        self.status_name = _lib.STATUS_NAMES.get(status, str(status))
        super().__init__("%s: %s" % (self.status_name, message))


def _check(status: int):
    if status != _lib.FI_OK:
        msg = _lib.load().fi_last_error().decode(errors="replace")
        raise FiError(status, msg)


_I64x4 = ctypes.c_int64 * 4


def tensor_desc(t: torch.Tensor) -> FiTensor:
    """fi_tensor view of a torch tensor (no copy; strides in elements)."""
    nd = t.dim()
    if nd < 1 or nd > 4:
        raise ValueError("fi_tensor supports ranks 1..4, got %d" % nd)
    code = _DTYPES.get(t.dtype)
    if code is None:
        raise ValueError("unsupported dtype %s" % t.dtype)
    # one constructor call: per-field assignment costs several microseconds
    return FiTensor(t.data_ptr(), code, nd, _I64x4(*t.shape), _I64x4(*t.stride()))


# fi_tensor as packed bytes (void*, dtype, ndim, shape[4], stride[4]): about
# half the cost of building the ctypes structure, which matters on the run()
# path where six descriptors are made per call.
_FMT = struct.Struct("<Qii4q4q")
_Z4 = (0, 0, 0, 0)


def _desc(t: torch.Tensor) -> bytes:
    """fi_tensor bytes of a torch tensor (no copy of its data)."""
    code = _DTYPES.get(t.dtype)
    nd = t.dim()
    if code is None or nd < 1 or nd > 4:
        return bytes(tensor_desc(t))  # raises the descriptive error
    return _FMT.pack(t.data_ptr(), code, nd, *(tuple(t.shape) + _Z4)[:4],
                     *(t.stride() + _Z4)[:4])


_PI32 = ctypes.POINTER(ctypes.c_int32)


def _host_i32(x):
    if x is None:
        return None, None
    if isinstance(x, torch.Tensor):
        if x.dtype == torch.int32 and x.device.type == "cpu" and x.is_contiguous():
            # already host int32: pass its storage (the caller keeps x alive)
            return x, ctypes.cast(x.data_ptr(), _PI32)
        x = x.detach().cpu().numpy()
    a = np.ascontiguousarray(np.asarray(x), dtype=np.int32)
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream_handle(stream, t=None):
    """The cudaStream_t to pass: `stream`, else torch's current stream (on
    tensor t's device when t is given)."""
    if stream is None:
        if t is not None and t.is_cuda and _raw_stream is not None:
            return _raw_stream(t.get_device())
        if torch.cuda.is_available() and torch.cuda.is_initialized():
            return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        return ctypes.c_void_p(0)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def workspace_bytes(max_batch: int, max_total_rows: int, num_qo_heads: int, head_dim: int,
                    max_kv_chunks: int) -> int:
    return int(_lib.load().fi_workspace_bytes(max_batch, max_total_rows, num_qo_heads, head_dim,
                                              max_kv_chunks))


class Plan:
    """An ``fi_plan_t`` bound to a caller-owned device workspace.

    ``workspace`` is a CUDA uint8 tensor (kept alive by the plan) or None for a
    host-only plan (validation and planning without a GPU).
    """

    def __init__(self, workspace=None, enable_graph_capture=False, max_batch=0, max_total_rows=0):
        lib = _lib.load()
        self._lib = lib
        self.workspace = workspace
        ptr = ctypes.c_void_p()
        ws_ptr = workspace.data_ptr() if workspace is not None else None
        ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
        _check(lib.fi_plan_create(ctypes.byref(ptr), ws_ptr, ws_bytes, int(bool(enable_graph_capture)),
                                  int(max_batch), int(max_total_rows)))
        self._h = ptr
        self.q_len_per_req = None

    def close(self):
        if getattr(self, "_h", None):
            self._lib.fi_plan_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def handle(self):
        if not self._h:
            raise RuntimeError("plan is closed")
        return self._h

    def plan(self, qo_indptr, kv_indptr, last_page_len, page_size, num_qo_heads, num_kv_heads,
             head_dim, causal=False, window_left=-1, dtype=torch.bfloat16, q_len_per_req=0,
             force_kv_chunks=0, stream=None):
        """fi_plan: host int32 metadata (tensors, arrays or lists)."""
        qo, qo_p = _host_i32(qo_indptr)
        kv, kv_p = _host_i32(kv_indptr)
        last, last_p = _host_i32(last_page_len)
        batch = len(kv) - 1 if kv is not None else 0
        _check(self._lib.fi_plan(self.handle, qo_p, kv_p, last_p, batch, int(page_size),
                                 int(num_qo_heads), int(num_kv_heads), int(head_dim),
                                 int(bool(causal)), int(window_left), _DTYPES[dtype],
                                 int(q_len_per_req), int(force_kv_chunks), _stream_handle(stream)))
        self.q_len_per_req = q_len_per_req
        return self

    def plan_masked(self, qo_indptr, kv_indptr, last_page_len, page_size, num_qo_heads,
                    num_kv_heads, head_dim, mask_indptr, causal=False, window_left=-1,
                    dtype=torch.bfloat16, force_kv_chunks=0, stream=None):
        """fi_plan_masked: a paged prefill with a custom (tree) mask whose
        request b starts at byte mask_indptr[b] (host int32)."""
        qo, qo_p = _host_i32(qo_indptr)
        kv, kv_p = _host_i32(kv_indptr)
        last, last_p = _host_i32(last_page_len)
        mi, mi_p = _host_i32(mask_indptr)
        batch = len(kv) - 1 if kv is not None else 0
        _check(self._lib.fi_plan_masked(self.handle, qo_p, kv_p, last_p, batch, int(page_size),
                                        int(num_qo_heads), int(num_kv_heads), int(head_dim),
                                        int(bool(causal)), int(window_left), _DTYPES[dtype], mi_p,
                                        int(force_kv_chunks), _stream_handle(stream)))
        self.q_len_per_req = 0
        return self

    def plan_ragged(self, qo_indptr, kv_indptr, num_qo_heads, num_kv_heads, head_dim,
                    causal=False, window_left=-1, dtype=torch.bfloat16, force_kv_chunks=0,
                    stream=None):
        """fi_plan_ragged: kv_indptr holds each request's first row of a
        contiguous [rows, Hk, d] K/V (host int32 tensors, arrays or lists)."""
        qo, qo_p = _host_i32(qo_indptr)
        kv, kv_p = _host_i32(kv_indptr)
        batch = len(kv) - 1 if kv is not None else 0
        _check(self._lib.fi_plan_ragged(self.handle, qo_p, kv_p, batch, int(num_qo_heads),
                                        int(num_kv_heads), int(head_dim), int(bool(causal)),
                                        int(window_left), _DTYPES[dtype], int(force_kv_chunks),
                                        _stream_handle(stream)))
        self.q_len_per_req = 0
        return self

    def info(self, with_arrays=False):
        inf = FiPlanInfo()
        _check(self._lib.fi_plan_get_info(self.handle, ctypes.byref(inf), None, 0, None, 0))
        out = {n: getattr(inf, n) for n, _ in FiPlanInfo._fields_}
        out["kernel_name"] = KERNEL_NAMES.get(out["kernel"], "?")
        if with_arrays:
            items = np.zeros(max(out["num_items"], 1) * 8, np.int32)
            merge = np.zeros(out["total_rows"] + 1, np.int32)
            _check(self._lib.fi_plan_get_info(
                self.handle, None, items.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                items.size, merge.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), merge.size))
            out["items"] = items[: out["num_items"] * 8].reshape(-1, 8)
            out["merge_indptr"] = merge
        return out

    def read_device(self, stream=None):
        inf = self.info()
        items = np.zeros(max(inf["num_items"], 1) * 8, np.int32)
        merge = np.zeros(inf["total_rows"] + 1, np.int32)
        _check(self._lib.fi_plan_read_device(
            self.handle, items.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), items.size,
            merge.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), merge.size,
            _stream_handle(stream)))
        return items[: inf["num_items"] * 8].reshape(-1, 8), merge


    def device_error(self, clear=False, stream=None) -> int:
        """fi_plan_device_error: a bit set, 0 when nothing went wrong since the
        last plan / clear; 1 = a kernel gave up an expired bounded wait, 2 =
        the page-table check found entries outside the cache."""
        v = ctypes.c_int32(0)
        _check(self._lib.fi_plan_device_error(self.handle, ctypes.byref(v), int(bool(clear)),
                                              _stream_handle(stream)))
        return int(v.value)

    def set_wait_limit(self, limit_ns: int):
        """fi_plan_set_wait_limit: the bounded-wait limit of this plan's kernels
        from the next plan on (0 = the default 2 s)."""
        _check(self._lib.fi_plan_set_wait_limit(self.handle, int(limit_ns)))

    def check_kv_indices(self, kv_indices, num_pages: int, stream=None):
        """fi_check_kv_indices: count page-table entries outside [0, num_pages)
        on the device (read back with device_error(), bit 2)."""
        d = tensor_desc(kv_indices)
        _check(self._lib.fi_check_kv_indices(self.handle, ctypes.byref(d), int(num_pages),
                                             _stream_handle(stream)))


def fi_plan(plan: Plan, *args, **kwargs) -> Plan:
    return plan.plan(*args, **kwargs)


def _run(fn, plan, q, k_cache, v_cache, kv_indices, sm_scale, out, lse, return_lse, stream):
    if out is None:
        out = torch.empty(q.shape, dtype=q.dtype, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty(q.shape[:2], dtype=torch.float32, device=q.device)
    st = fn(plan.handle, _desc(q), _desc(k_cache), _desc(v_cache), _desc(kv_indices),
            sm_scale, _desc(out), _desc(lse) if lse is not None else None,
            _stream_handle(stream, q))
    if st:
        _check(st)
    return out, lse


def fi_batch_prefill_paged(plan, q, k_cache, v_cache, kv_indices, sm_scale, out=None, lse=None,
                           return_lse=True, stream=None):
    """Batched paged prefill; returns (out, lse)."""
    return _run(_lib.load().fi_batch_prefill_paged, plan, q, k_cache, v_cache, kv_indices,
                sm_scale, out, lse, return_lse, stream)


def fi_batch_decode_paged(plan, q, k_cache, v_cache, kv_indices, sm_scale, out=None, lse=None,
                          return_lse=True, stream=None):
    """Batched paged decode / speculative verify; returns (out, lse)."""
    return _run(_lib.load().fi_batch_decode_paged, plan, q, k_cache, v_cache, kv_indices,
                sm_scale, out, lse, return_lse, stream)


def fi_batch_prefill_paged_masked(plan, q, k_cache, v_cache, kv_indices, custom_mask, sm_scale,
                                  out=None, lse=None, return_lse=True, stream=None):
    """Paged prefill with a custom (tree) mask: custom_mask is a device uint8
    tensor of bit-packed per-request masks; returns (out, lse)."""
    if out is None:
        out = torch.empty(q.shape, dtype=q.dtype, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty(q.shape[:2], dtype=torch.float32, device=q.device)
    descs = [tensor_desc(t) for t in (q, k_cache, v_cache, kv_indices, custom_mask, out)]
    ld = tensor_desc(lse) if lse is not None else None
    _check(_lib.load().fi_batch_prefill_paged_masked(
        plan.handle, *[ctypes.byref(d) for d in descs[:5]], ctypes.c_float(sm_scale),
        ctypes.byref(descs[5]), ctypes.byref(ld) if ld is not None else None,
        _stream_handle(stream)))
    return out, lse


def fi_chain_speculative_sampling(draft_probs, draft_token_ids, target_probs, uniform_accept,
                                  uniform_sample, output_token_ids=None, accepted_num=None,
                                  emitted_num=None, stream=None):
    """Chain speculative-sampling acceptance step on the device; returns
    (output_token_ids [B, n+1], accepted_num [B], emitted_num [B])."""
    B, n1 = target_probs.shape[0], target_probs.shape[1]
    dev = target_probs.device
    if output_token_ids is None:
        output_token_ids = torch.empty((B, n1), dtype=torch.int32, device=dev)
    if accepted_num is None:
        accepted_num = torch.empty((B,), dtype=torch.int32, device=dev)
    if emitted_num is None:
        emitted_num = torch.empty((B,), dtype=torch.int32, device=dev)
    n = n1 - 1
    ins = [tensor_desc(t) if n > 0 else None
           for t in (draft_probs, draft_token_ids)] + [tensor_desc(target_probs)]
    ua = tensor_desc(uniform_accept) if n > 0 else None
    us = tensor_desc(uniform_sample)
    outs = [tensor_desc(t) for t in (output_token_ids, accepted_num, emitted_num)]
    ref = lambda d: ctypes.byref(d) if d is not None else None  # noqa: E731
    _check(_lib.load().fi_chain_speculative_sampling(
        ref(ins[0]), ref(ins[1]), ref(ins[2]), ref(ua), ref(us), *[ref(d) for d in outs],
        _stream_handle(stream)))
    return output_token_ids, accepted_num, emitted_num


def fi_batch_prefill_ragged(plan, q, k, v, sm_scale, out=None, lse=None, return_lse=True,
                            stream=None):
    """Batched prefill over contiguous K/V [rows, Hk, d]; returns (out, lse)."""
    if out is None:
        out = torch.empty(q.shape, dtype=q.dtype, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty(q.shape[:2], dtype=torch.float32, device=q.device)
    qd, kd, vd, od = tensor_desc(q), tensor_desc(k), tensor_desc(v), tensor_desc(out)
    ld = tensor_desc(lse) if lse is not None else None
    _check(_lib.load().fi_batch_prefill_ragged(
        plan.handle, ctypes.byref(qd), ctypes.byref(kd), ctypes.byref(vd), ctypes.c_float(sm_scale),
        ctypes.byref(od), ctypes.byref(ld) if ld is not None else None, _stream_handle(stream)))
    return out, lse


def fi_merge_state(v_a, s_a, v_b, s_b, v_out=None, s_out=None, num_rows_dev=None, stream=None):
    """Merge two attention states by LSE; returns (v_out, s_out)."""
    if v_out is None:
        v_out = torch.empty(v_a.shape, dtype=v_a.dtype, device=v_a.device)
    if s_out is None:
        s_out = torch.empty(s_a.shape, dtype=torch.float32, device=s_a.device)
    descs = [tensor_desc(t) for t in (v_a, s_a, v_b, s_b, v_out, s_out)]
    _check(_lib.load().fi_merge_state(*[ctypes.byref(d) for d in descs],
                                      num_rows_dev.data_ptr() if num_rows_dev is not None else None,
                                      _stream_handle(stream)))
    return v_out, s_out


def fi_merge_states(v, s, merge_indptr, rows, v_out=None, s_out=None, out_dtype=torch.float32,
                    num_rows_dev=None, return_lse=True, stream=None):
    """Variable-length merge: row r merges states merge_indptr[r]..[r+1]-1."""
    if v_out is None:
        v_out = torch.empty((rows,) + tuple(v.shape[1:]), dtype=out_dtype, device=v.device)
    if s_out is None and return_lse:
        s_out = torch.empty((rows, v.shape[1]), dtype=torch.float32, device=v.device)
    vd, sd, vod = tensor_desc(v), tensor_desc(s), tensor_desc(v_out)
    sod = tensor_desc(s_out) if s_out is not None else None
    _check(_lib.load().fi_merge_states(
        ctypes.byref(vd), ctypes.byref(sd), merge_indptr.data_ptr(), int(rows), ctypes.byref(vod),
        ctypes.byref(sod) if sod is not None else None,
        num_rows_dev.data_ptr() if num_rows_dev is not None else None, _stream_handle(stream)))
    return v_out, s_out


def fi_batch_decode_paged_noalloc(q, k_cache, v_cache, kv_indices, kv_indptr, last_page_len,
                                  sm_scale, window_left=-1, kv_chunks=4, out=None, lse=None,
                                  return_lse=True, stream=None):
    """Batch decode whose split-KV scratch is a fixed device array inside the
    library: the call itself allocates no device memory (``out``/``lse`` are
    allocated here only when not passed; with ``return_lse=False`` no lse is
    written and NULL is passed). kv_indptr / last_page_len are device int32
    tensors; the batch is ``len(kv_indptr) - 1``."""
    lib = _lib.load()
    batch = kv_indptr.shape[0] - 1
    if out is None:
        out = torch.empty(q.shape, dtype=q.dtype, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty(q.shape[:2], dtype=torch.float32, device=q.device)
    descs = [tensor_desc(t) for t in (q, k_cache, v_cache, kv_indices)]
    od = tensor_desc(out)
    ld = tensor_desc(lse) if lse is not None else None
    st = lib.fi_batch_decode_paged_noalloc(
        *[ctypes.byref(d) for d in descs], kv_indptr.data_ptr(), last_page_len.data_ptr(),
        int(batch), int(window_left), int(kv_chunks), ctypes.c_float(sm_scale), ctypes.byref(od),
        ctypes.byref(ld) if ld is not None else None, _stream_handle(stream))
    if st != _lib.FI_OK:
        raise FiError(st, lib.fi_noalloc_last_error().decode(errors="replace"))
    return out, lse


def fi_noalloc_device_error(clear=False, stream=None) -> int:
    """fi_noalloc_device_error: 1 when the latest no-allocation decode on the
    current device gave up an expired bounded wait, else 0."""
    lib = _lib.load()
    v = ctypes.c_int32(0)
    st = lib.fi_noalloc_device_error(ctypes.byref(v), int(bool(clear)), _stream_handle(stream))
    if st != _lib.FI_OK:
        raise FiError(st, lib.fi_noalloc_last_error().decode(errors="replace"))
    return int(v.value)
