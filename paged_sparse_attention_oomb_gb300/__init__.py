"""Page-level sparse causal attention over a paged KV cache, for one GB300.

The compute lives in ``liboomb.so`` (hand-written CUDA for sm_103a behind a
C ABI declared in ``include/oomb.h``).  ``paged_sparse_attention_oomb_gb300.oomb``
is the thin Python binding with the same call names; it only marshals
arguments and raises if the native library is missing.  ``workloads`` holds
the named workloads and the seeded input generator.
"""
from .workloads import WORKLOADS, Workload, make_inputs  # noqa: F401

__all__ = ["WORKLOADS", "Workload", "make_inputs"]
