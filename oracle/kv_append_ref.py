"""Test infrastructure only: float64 / exact-integer CPU oracle of the KV-cache append with
quantise-on-write.  Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s
CPU-baseline leg may import it; the product path never does.

What it computes (sources by page and section):

* tokenspeed ``tokenspeed_mla.py``, ``CuteDSLMLABackend.forward_decode``: before the decode,
  this step's latent ``k[..., :512]`` and rope ``k[..., 512:]`` of every new token are
  written into the paged cache at the token's flat cache location ``out_cache_loc``
  (``set_mla_kv_buffer``); a location is ``page * page_size + row``.
* metrale ``kv_cache_mla.rs``, ``mla_cache_assemble`` and the NVFP4 / FP8 paged decode
  launchers: a cache entry is the 576 values ``[latent | rope]``; an NVFP4 page holds the
  packed E2M1 data section followed by one E4M3 scale per 16 values; an FP8 cache holds one
  E4M3 code per value with one scalar scale.

The pages do not say how values are quantised.  Readings taken (the plainest ones the
layouts support):

* FP8: ``code = E4M3(x / kv_scale)``, the quotient taken in fp32 and rounded to the nearest
  E4M3 value, ties to the even code, saturating to +-448 (the caller's per-tensor scale).
* NVFP4: per group of 16 values, ``s = E4M3(amax / 6)`` (fp32 quotient, same rounding);
  ``code_i = E2M1(x_i / value(s))`` (fp32 quotient, nearest E2M1 value, ties to the even
  code, saturating to +-6); a group whose scale decodes to 0 stores all-zero codes.  No
  second-level scale.
* The sign of a result that rounds to zero is the sign of its input (IEEE rounding).
* bf16 tokens are stored unchanged.  Negative locations are padding and are skipped;
  locations past the cache are skipped (the kernel reports them).  Locations are distinct.

Rounding decisions are taken on fp32 quotients on both sides (the kernel computes in fp32),
so the stored bytes must agree exactly.
"""
from __future__ import annotations

import numpy as np

from .mla_ref import CACHE_DIM, E2M1_TABLE, E4M3_TABLE, LATENT_DIM, NVFP4_GROUP, ROPE_DIM, decode_bf16

# Non-negative finite codes in increasing order of value (codes 0..0x7E; 0x7F is NaN) and
# their values: E4M3 codes 0..126 and E2M1 codes 0..7 are both monotone in value.
_E4M3_POS = E4M3_TABLE[:0x7F]
_E2M1_POS = E2M1_TABLE[:8]


def _encode_nearest_even(x: np.ndarray, pos_values: np.ndarray, sign_bit: int) -> np.ndarray:
    """Nearest code of each value of ``x``: the magnitude goes to the nearest entry of
    ``pos_values`` (ties to the entry with an even code), saturating at the last entry; the
    sign bit is set when ``x`` has its sign bit set."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    top = len(pos_values) - 1
    hi = np.searchsorted(pos_values, a, side="left")  # first entry >= a
    hi = np.minimum(hi, top)
    lo = np.maximum(hi - 1, 0)
    exact_or_sat = (pos_values[hi] == a) | (a >= pos_values[top])
    d_lo = a - pos_values[lo]
    d_hi = pos_values[hi] - a
    pick = np.where(d_lo < d_hi, lo, np.where(d_hi < d_lo, hi, np.where(lo % 2 == 0, lo, hi)))
    code = np.where(exact_or_sat, np.where(a >= pos_values[top], top, hi), pick).astype(np.uint8)
    return code | (np.signbit(x).astype(np.uint8) * np.uint8(sign_bit))


def encode_e4m3(x) -> np.ndarray:
    """fp32 (or exactly representable) values -> OCP E4M3 codes: round to nearest, ties to
    even, saturate to +-448.  Inputs must be finite."""
    return _encode_nearest_even(x, _E4M3_POS, 0x80)


def encode_e2m1(x) -> np.ndarray:
    """Values -> OCP E2M1 codes (0..15): round to nearest, ties to even, saturate to +-6."""
    return _encode_nearest_even(x, _E2M1_POS, 0x8)


def quantize_token_fp8(x32: np.ndarray, kv_scale: float) -> np.ndarray:
    """One token's 576 fp32 values -> 576 E4M3 codes of ``x / kv_scale`` (fp32 quotient)."""
    q = np.asarray(x32, dtype=np.float32) / np.float32(kv_scale)
    return encode_e4m3(q)


def quantize_token_nvfp4(x32: np.ndarray):
    """One token's 576 fp32 values -> (288 packed E2M1 bytes, 36 E4M3 scale codes)."""
    g = np.asarray(x32, dtype=np.float32).reshape(CACHE_DIM // NVFP4_GROUP, NVFP4_GROUP)
    amax = np.abs(g).max(axis=1)
    s_code = encode_e4m3(amax / np.float32(6.0))
    s_val = E4M3_TABLE[s_code].astype(np.float32)
    nib = np.zeros_like(g, dtype=np.uint8)
    live = s_val > 0
    if live.any():
        nib[live] = encode_e2m1(g[live] / s_val[live, None])
    nib = nib.reshape(CACHE_DIM)
    packed = (nib[0::2] | (nib[1::2] << 4)).astype(np.uint8)
    return packed, s_code.astype(np.uint8)


def kv_append_ref(cache: np.ndarray, latent_bits: np.ndarray, rope_bits: np.ndarray, slots: np.ndarray,
                  kv_dtype: str, page_size: int, kv_scale: float = 1.0) -> np.ndarray:
    """A copy of ``cache`` with token ``t``'s ``[latent | rope]`` (bf16 bit patterns,
    ``[T, 512]`` and ``[T, 64]``) stored at flat location ``slots[t]`` in the cache's format
    (layouts as in :func:`oracle.mla_ref.dequant_pages`)."""
    out = cache.copy()
    num_slots = cache.shape[0] * page_size
    slots = np.asarray(slots, dtype=np.int64)
    for t in range(slots.shape[0]):
        s = int(slots[t])
        if s < 0 or s >= num_slots:
            continue
        page, row = divmod(s, page_size)
        bits = np.concatenate([np.asarray(latent_bits[t], np.uint16), np.asarray(rope_bits[t], np.uint16)])
        if kv_dtype == "bf16":
            out[page, row] = bits
            continue
        x32 = decode_bf16(bits).astype(np.float32)  # exact: bf16 is a truncated fp32
        if kv_dtype == "fp8":
            out[page, row] = quantize_token_fp8(x32, kv_scale)
        elif kv_dtype == "nvfp4":
            packed, scales = quantize_token_nvfp4(x32)
            data = page_size * CACHE_DIM // 2
            out[page, row * (CACHE_DIM // 2):(row + 1) * (CACHE_DIM // 2)] = packed
            out[page, data + row * (CACHE_DIM // NVFP4_GROUP):data + (row + 1) * (CACHE_DIM // NVFP4_GROUP)] = scales
        else:
            raise ValueError(f"unknown kv_dtype {kv_dtype!r}")
    return out


assert LATENT_DIM + ROPE_DIM == CACHE_DIM
