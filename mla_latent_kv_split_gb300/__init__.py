"""Absorbed-form MLA split-KV decode for GB300 (sm_103a).

The compute lives in ``libmla_decode.so`` (hand-written CUDA kernels behind a C ABI,
declared in ``include/mla_decode.h``).  :mod:`.binding` marshals arguments to it;
:mod:`.workloads` draws seeded synthetic inputs.  Importing this package loads nothing;
the shared library is opened on first use and a missing library is an error.
"""
__all__ = ["binding", "workloads"]
