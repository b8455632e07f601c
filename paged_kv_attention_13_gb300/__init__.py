"""Paged-KV attention for one NVIDIA GB300 (sm_103a).

The product is the C-ABI library ``libfi.so`` (declared in ``include/fi.h``):
batched prefill, decode and speculative verify over a paged KV cache, and
LSE merging of split-KV partial states. This package holds its CUDA sources
(``csrc/``), its build script and a thin ctypes binding with the C names.
"""
from .api import (FiError, Plan, fi_batch_decode_paged, fi_batch_decode_paged_noalloc,  # noqa: F401
                  fi_batch_prefill_paged, fi_batch_prefill_paged_masked, fi_batch_prefill_ragged,
                  fi_chain_speculative_sampling, fi_merge_state, fi_merge_states,
                  fi_noalloc_device_error, fi_plan, tensor_desc, workspace_bytes)
from ._lib import EXPORTED, LIB_PATH, load  # noqa: F401
