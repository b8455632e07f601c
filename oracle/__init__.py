"""CPU oracle for paged-KV attention and LSE state merging.

TEST INFRASTRUCTURE ONLY: the tests, the package smoke check and the
benchmark's CPU-baseline leg are the only callers. The product library never
imports, links or runs anything here, and nothing here imports the product.

- ``attention_oracle.c``: the plain fp64 definition, one row at a time, with
  its own paged indexing (built into ``liboracle.so`` by ``build.py``).
- ``reference.py``: ctypes wrapper around it.
- ``brute.py``: a numpy brute force for tiny inputs that materialises the
  boolean mask matrix element by element.
- ``speculative.py``: the chain speculative-sampling acceptance step.
"""
from .build import build_oracle  # noqa: F401
from .reference import attention_rows, attention_all, merge_states, kv_len  # noqa: F401
