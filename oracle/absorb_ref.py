"""Test infrastructure only: float64 CPU oracle of the two per-head projections on either
side of the absorbed decode.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline leg may import it; the product path never does.

metrale ``kv_cache_mla.rs``, ``mla_batched_gemv``: one launch over all heads computes
``output[head, n] = sum_k weight[head, n, k] * input[head, k]`` in BF16, with the weight
contiguous per head and per-head input / output strides.  In the absorbed form of MLA it
serves both sides of the latent attention:

* Q absorption: ``q_lat[h, c] = sum_d W_UK[h, d, c] q_nope[h, d]`` (weight = W_UK^T per
  head, ``[512, 128]``), so that ``q_lat . c_t = q_nope . (W_UK c_t)``: scoring the latent
  cache row equals scoring the up-projected key.
* V up-projection: ``o[h, d] = sum_c W_UV[h, d, c] o_lat[h, c]`` (weight = W_UV, ``[128, 512]``).

Batched over tokens: ``out[t, h, n] = sum_k weight[h, n, k] x[t, h, k]``, accumulated
exactly (float64) here; the kernel accumulates in fp32 and rounds the result to bf16.
"""
from __future__ import annotations

import numpy as np

from .mla_ref import decode_bf16


def _values(a: np.ndarray) -> np.ndarray:
    a = np.asarray(a)
    return decode_bf16(a) if a.dtype == np.uint16 else a.astype(np.float64)


def batched_gemv_ref(x: np.ndarray, w: np.ndarray) -> np.ndarray:
    """``x [T, H, K]`` and ``w [H, N, K]`` (bf16 bit patterns as uint16, or real values)
    -> float64 ``[T, H, N]`` with ``out[t, h, n] = sum_k w[h, n, k] * x[t, h, k]``."""
    return np.einsum("hnk,thk->thn", _values(w), _values(x))
