"""GB300-native paged attention over a block-table-addressed KV cache.

The compute path is the C-ABI library ``libpa.so`` built from ``csrc/``
(hand-written sm_103a CUDA kernels); ``binding`` is its thin ctypes binding
and ``workload`` holds the seeded synthetic input generators.  Importing this
package loads nothing: ``binding`` loads the library on first import and
raises if it is missing.
"""
__all__ = ["binding", "workload"]
