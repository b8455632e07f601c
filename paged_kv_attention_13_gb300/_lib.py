"""ctypes declarations of libfi.so (the C ABI in include/fi.h).

Argument marshalling only. Loading fails loudly when the library is missing:
there is no fallback implementation anywhere in this package.
"""
import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libfi.so")

FI_OK = 0
STATUS_NAMES = {
    0: "FI_OK", 1: "FI_ERR_INVALID_ARG", 2: "FI_ERR_STRIDED_LAST_DIM",
    3: "FI_ERR_NONCONTIGUOUS_OUTPUT", 4: "FI_ERR_GQA_INDIVISIBLE", 5: "FI_ERR_PLAN_MISMATCH",
    6: "FI_ERR_NOT_PLANNED", 7: "FI_ERR_KV_SHORTER_THAN_Q", 8: "FI_ERR_CAPACITY",
    9: "FI_ERR_UNSUPPORTED", 10: "FI_ERR_CUDA",
}
FI_F16, FI_BF16, FI_F32, FI_I32, FI_U8 = 0, 1, 2, 3, 4

# Every symbol include/fi.h declares.
EXPORTED = [
    "fi_workspace_bytes", "fi_plan_create", "fi_plan", "fi_batch_prefill_paged",
    "fi_batch_decode_paged", "fi_merge_state", "fi_merge_states", "fi_plan_get_info",
    "fi_plan_read_device", "fi_plan_destroy", "fi_last_error", "fi_status_str",
    "fi_batch_decode_paged_noalloc", "fi_noalloc_scratch_bytes", "fi_noalloc_last_error",
    "fi_plan_device_error", "fi_plan_ragged", "fi_batch_prefill_ragged", "fi_plan_masked",
    "fi_batch_prefill_paged_masked", "fi_chain_speculative_sampling",
    "fi_plan_set_wait_limit", "fi_check_kv_indices", "fi_noalloc_device_error",
]


class FiTensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int), ("ndim", ctypes.c_int32),
                ("shape", ctypes.c_int64 * 4), ("stride", ctypes.c_int64 * 4)]


class FiPlanInfo(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "batch", "total_rows", "kernel", "tile_rows", "num_items", "num_partials",
        "num_merge_rows", "max_chunks", "grid", "graph_mode")]


_lib = None


def load():
    """Load libfi.so (built by ``paged_kv_attention_13_gb300.build``)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            "libfi.so is not built (%s); run `python -c \"import __graft_entry__ as g; g.build()\"` "
            "or `python paged_kv_attention_13_gb300/build.py`" % LIB_PATH)
    lib = ctypes.CDLL(LIB_PATH)
    P = ctypes.c_void_p
    i32 = ctypes.c_int32
    PT = ctypes.POINTER(FiTensor)
    pi32 = ctypes.POINTER(ctypes.c_int32)
    lib.fi_workspace_bytes.restype = ctypes.c_size_t
    lib.fi_workspace_bytes.argtypes = [i32, i32, i32, i32, i32]
    lib.fi_plan_create.restype = ctypes.c_int
    lib.fi_plan_create.argtypes = [ctypes.POINTER(P), P, ctypes.c_size_t, i32, i32, i32]
    lib.fi_plan.restype = ctypes.c_int
    lib.fi_plan.argtypes = [P, pi32, pi32, pi32, i32, i32, i32, i32, i32, i32, i32, ctypes.c_int,
                            i32, i32, P]
    for name in ("fi_batch_prefill_paged", "fi_batch_decode_paged"):
        f = getattr(lib, name)
        f.restype = ctypes.c_int
        # tensor descriptors as void*: a ctypes byref or the packed bytes
        f.argtypes = [P, P, P, P, P, ctypes.c_float, P, P, P]
    lib.fi_merge_state.restype = ctypes.c_int
    lib.fi_merge_state.argtypes = [PT, PT, PT, PT, PT, PT, P, P]
    lib.fi_merge_states.restype = ctypes.c_int
    lib.fi_merge_states.argtypes = [PT, PT, P, i32, PT, PT, P, P]
    lib.fi_plan_get_info.restype = ctypes.c_int
    lib.fi_plan_get_info.argtypes = [P, ctypes.POINTER(FiPlanInfo), pi32, i32, pi32, i32]
    lib.fi_plan_read_device.restype = ctypes.c_int
    lib.fi_plan_read_device.argtypes = [P, pi32, i32, pi32, i32, P]
    lib.fi_chain_speculative_sampling.restype = ctypes.c_int
    lib.fi_chain_speculative_sampling.argtypes = [PT, PT, PT, PT, PT, PT, PT, PT, P]
    lib.fi_plan_masked.restype = ctypes.c_int
    lib.fi_plan_masked.argtypes = [P, pi32, pi32, pi32, i32, i32, i32, i32, i32, i32, i32,
                                   ctypes.c_int, pi32, i32, P]
    lib.fi_batch_prefill_paged_masked.restype = ctypes.c_int
    lib.fi_batch_prefill_paged_masked.argtypes = [P, PT, PT, PT, PT, PT, ctypes.c_float, PT, PT, P]
    lib.fi_plan_ragged.restype = ctypes.c_int
    lib.fi_plan_ragged.argtypes = [P, pi32, pi32, i32, i32, i32, i32, i32, i32, ctypes.c_int, i32, P]
    lib.fi_batch_prefill_ragged.restype = ctypes.c_int
    lib.fi_batch_prefill_ragged.argtypes = [P, PT, PT, PT, ctypes.c_float, PT, PT, P]
    lib.fi_plan_device_error.restype = ctypes.c_int
    lib.fi_plan_device_error.argtypes = [P, pi32, ctypes.c_int, P]
    lib.fi_plan_set_wait_limit.restype = ctypes.c_int
    lib.fi_plan_set_wait_limit.argtypes = [P, ctypes.c_uint64]
    lib.fi_check_kv_indices.restype = ctypes.c_int
    lib.fi_check_kv_indices.argtypes = [P, PT, ctypes.c_int64, P]
    lib.fi_noalloc_device_error.restype = ctypes.c_int
    lib.fi_noalloc_device_error.argtypes = [pi32, ctypes.c_int, P]
    lib.fi_plan_destroy.restype = None
    lib.fi_plan_destroy.argtypes = [P]
    lib.fi_last_error.restype = ctypes.c_char_p
    lib.fi_last_error.argtypes = []
    lib.fi_status_str.restype = ctypes.c_char_p
    lib.fi_status_str.argtypes = [ctypes.c_int]
    lib.fi_batch_decode_paged_noalloc.restype = ctypes.c_int
    lib.fi_batch_decode_paged_noalloc.argtypes = [PT, PT, PT, PT, P, P, i32, i32, i32,
                                                  ctypes.c_float, PT, PT, P]
    lib.fi_noalloc_scratch_bytes.restype = ctypes.c_size_t
    lib.fi_noalloc_scratch_bytes.argtypes = []
    lib.fi_noalloc_last_error.restype = ctypes.c_char_p
    lib.fi_noalloc_last_error.argtypes = []
    _lib = lib
    return lib
