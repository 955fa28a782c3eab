"""Exact attention for GB300 (sm_103a): tcgen05/TMA kernels behind a C ABI.

The compute path is libfa_gb300.so (built by ``exact_attention_76_gb300.build``);
``exact_attention_76_gb300.api`` binds its entry points by name.  Importing
this package loads nothing; the library loads on the first API call and a
missing library is an error, never a fallback.
"""

__all__ = ["api", "inputs", "build"]
