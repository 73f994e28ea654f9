"""fp64 CPU oracle for grouped-query softmax attention.

TEST INFRASTRUCTURE: only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's
CPU-baseline leg may import this package.  The product library never does.
"""
from .attention import (SOURCE, Oracle, build_library, compile_library, decode,
                        default_threads, kv_append, kv_append_ring, prefill)

__all__ = ["SOURCE", "Oracle", "build_library", "compile_library", "decode",
           "default_threads", "kv_append", "kv_append_ring", "prefill"]
