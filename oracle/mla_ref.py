"""Float64 CPU oracle for absorbed-form MLA decode over a paged 576-wide latent cache.

TEST INFRASTRUCTURE ONLY.  Plain, slow, obviously-correct NumPy in float64.  It shares
no code with the CUDA path and imports nothing from it; only the tests, the smoke
check and the bench's CPU-baseline leg use it.

What is computed (sources, by page and section):

* TileGym ``mla_decoding_split_kv.py``, ``_mla_decoding_split_kv.forward`` and the
  ``mla_decoding_split_kv`` entry point: per batch row and head, scores of the absorbed
  query ``[q (512) | qpe (64)]`` against the cache row ``[kv (512) | kpe (64)]``, a
  softmax with an explicit ``sm_scale``, and the same cache row's first 512 values used
  as V (the call passes ``KV`` for both K and V).  The KV sequence is cut into splits;
  each split yields a partial output and an fp32 log-sum-exp which ``splitk_reduce``
  combines.
* tokenspeed ``tokenspeed_mla.py``, ``CuteDSLMLABackend.forward_decode``: the cache is
  paged, ``[num_pages, page_size, 576]``, addressed through ``block_tables`` and
  ``seq_lens`` (which already count this step's ``q_len`` new tokens); FP8 E4M3 caches
  carry a per-tensor scale folded into the score.
* metrale ``kv_cache_mla.rs``, ``mla_paged_decode_nvfp4`` / ``mla_paged_decode_fp8``: a
  576-value token; an NVFP4 page holds packed E2M1 data followed by one E4M3 scale per
  16 values; FP8 pages hold one E4M3 byte per value with scalar scales.

Readings where the pages are silent (each also listed in the design notes):

* LSE is the natural log of ``sum_t exp(sm_scale * kv_scale * q.k_t)`` (scale included).
* Query ``i`` of ``q_len`` sees cache positions ``t < seq_len - q_len + i + 1``.
* Tokens at or past the visible length contribute exactly nothing, whatever bytes
  they hold; block-table entries past ``cdiv(seq_len, page_size)`` are never read.
* An empty split / empty query has ``lse = -inf`` and output 0.
* FP8: one ``kv_scale`` multiplies every stored value (the same bytes serve as K and V).
* NVFP4 page: token-major data, 288 bytes per token, element ``2j`` in the LOW nibble of
  byte ``j`` and ``2j+1`` in the high nibble; then token-major scales, 36 per token, scale
  ``g`` covering elements ``16g .. 16g+15`` (rope included); no second-level scale.
* Sliding window and attention sinks (metrale ``mla_paged_decode_fp8`` takes
  ``sliding_window`` and nullable per-head fp32 ``sinks`` without defining them): with a
  window ``W > 0`` query ``i`` sees only the last ``W`` of its visible positions,
  ``[max(0, V - W), V)``; a sink is one extra logit per head, in the units of the scaled
  scores ``x``, that enters the softmax normalisation and carries no value:
  ``lse = log(sum_t exp(x_t) + exp(sink))``, ``out = sum_t exp(x_t - lse) v_t``.
"""
from __future__ import annotations

import math

import numpy as np

LATENT_DIM = 512  # kv_lora_rank: the latent part, reused as V
ROPE_DIM = 64  # qk_rope_head_dim
CACHE_DIM = LATENT_DIM + ROPE_DIM  # 576 values per cached token
NVFP4_GROUP = 16  # one E4M3 scale per 16 values


# --------------------------------------------------------------------------------------
# Exact decoding of stored bytes (OCP 8-bit floating point / OCP MX v1.0 element types)
# --------------------------------------------------------------------------------------

def decode_bf16(bits: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns (uint16) -> float64, exactly (the top half of an IEEE f32)."""
    bits = np.asarray(bits, dtype=np.uint16)
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def _e4m3_value(code: int) -> float:
    """One OCP E4M3 ("FN") code -> its value: sign bit 7, exponent bits 6..3 with bias 7,
    mantissa bits 2..0; exponent 0 is subnormal (m/8 * 2^-6); S.1111.111 is NaN; there is
    no infinity, so the largest finite magnitude is 1.75 * 2^8 = 448."""
    sign = -1.0 if (code >> 7) & 1 else 1.0
    exp = (code >> 3) & 0xF
    man = code & 0x7
    if exp == 0xF and man == 0x7:
        return math.nan
    if exp == 0:
        return sign * (man / 8.0) * 2.0 ** -6
    return sign * (1.0 + man / 8.0) * 2.0 ** (exp - 7)


def _e2m1_value(nibble: int) -> float:
    """One OCP E2M1 (FP4) code -> its value: sign bit 3, exponent bits 2..1 with bias 1,
    mantissa bit 0; exponent 0 is subnormal (m * 0.5).  Magnitudes 0, .5, 1, 1.5, 2, 3, 4, 6."""
    sign = -1.0 if (nibble >> 3) & 1 else 1.0
    exp = (nibble >> 1) & 0x3
    man = nibble & 0x1
    if exp == 0:
        return sign * man * 0.5
    return sign * (1.0 + man / 2.0) * 2.0 ** (exp - 1)


E4M3_TABLE = np.array([_e4m3_value(c) for c in range(256)], dtype=np.float64)
E2M1_TABLE = np.array([_e2m1_value(c) for c in range(16)], dtype=np.float64)


def decode_e4m3(codes: np.ndarray) -> np.ndarray:
    return E4M3_TABLE[np.asarray(codes, dtype=np.uint8)]


def decode_e2m1(nibbles: np.ndarray) -> np.ndarray:
    return E2M1_TABLE[np.asarray(nibbles, dtype=np.uint8) & 0xF]


def nvfp4_page_bytes(page_size: int) -> int:
    """Bytes of one NVFP4 page: the packed E2M1 data section, then the E4M3 scale section
    (metrale ``mla_paged_decode_nvfp4``: data section followed by one scale per 16)."""
    return page_size * CACHE_DIM // 2 + page_size * CACHE_DIM // NVFP4_GROUP


def dequant_pages(cache: np.ndarray, kv_dtype: str, page_size: int, kv_scale: float,
                  pages: np.ndarray) -> np.ndarray:
    """Decode whole pages ``pages`` of the cache to float64 ``[len(pages), page_size, 576]``.

    ``cache`` layouts:  bf16 -> uint16 ``[num_pages, page_size, 576]``;
    fp8 -> uint8 ``[num_pages, page_size, 576]`` (value = e4m3(code) * kv_scale);
    nvfp4 -> uint8 ``[num_pages, nvfp4_page_bytes(page_size)]``
    (value = e2m1(nibble) * e4m3(scale of its 16-value group)).
    """
    pages = np.asarray(pages, dtype=np.int64)
    if kv_dtype == "bf16":
        return decode_bf16(cache[pages])
    if kv_dtype == "fp8":
        return decode_e4m3(cache[pages]) * np.float64(np.float32(kv_scale))
    if kv_dtype == "nvfp4":
        raw = cache[pages]  # [n, page_bytes]
        n = raw.shape[0]
        data_bytes = page_size * CACHE_DIM // 2
        data = raw[:, :data_bytes].reshape(n, page_size, CACHE_DIM // 2)
        scales = raw[:, data_bytes:].reshape(n, page_size, CACHE_DIM // NVFP4_GROUP)
        lo = data & 0xF  # element 2j
        hi = data >> 4  # element 2j+1
        nib = np.empty((n, page_size, CACHE_DIM), dtype=np.uint8)
        nib[..., 0::2] = lo
        nib[..., 1::2] = hi
        elem = decode_e2m1(nib)
        sc = decode_e4m3(scales)  # [n, ps, 36]
        return elem * np.repeat(sc, NVFP4_GROUP, axis=-1)
    raise ValueError(f"unknown kv_dtype {kv_dtype!r}")


def gather_tokens(cache: np.ndarray, block_table_row: np.ndarray, n_tokens: int, kv_dtype: str,
                  page_size: int, kv_scale: float = 1.0) -> np.ndarray:
    """Cache rows of positions ``0 .. n_tokens-1`` of one request, float64 ``[n_tokens, 576]``:
    ``row(t) = cache[block_table_row[t // page_size], t % page_size, :]`` (tokenspeed
    ``forward_decode``: paged cache addressed by ``block_tables``).  Only the pages that
    hold positions below ``n_tokens`` are read."""
    if n_tokens <= 0:
        return np.zeros((0, CACHE_DIM), dtype=np.float64)
    n_pages = -(-n_tokens // page_size)
    pages = np.asarray(block_table_row[:n_pages], dtype=np.int64)
    rows = dequant_pages(cache, kv_dtype, page_size, kv_scale, pages)
    return rows.reshape(n_pages * page_size, CACHE_DIM)[:n_tokens]


def visible_len(seq_len: int, q_len: int, i: int) -> int:
    """Number of cache positions query ``i`` of ``q_len`` may attend to: the last ``q_len``
    positions are this step's new tokens and query ``i`` sees up to and including its own
    position, i.e. ``t < seq_len - q_len + i + 1``; never negative."""
    return max(0, int(seq_len) - int(q_len) + int(i) + 1)


# --------------------------------------------------------------------------------------
# The decode itself: plain softmax attention per (request, query, head)
# --------------------------------------------------------------------------------------

def _query_rows(q_nope_bits: np.ndarray, q_pe_bits: np.ndarray) -> np.ndarray:
    """``[H, 512]`` and ``[H, 64]`` bf16 bit patterns -> float64 ``[H, 576]`` = ``[q_nope | q_pe]``."""
    return np.concatenate([decode_bf16(q_nope_bits), decode_bf16(q_pe_bits)], axis=-1)


def mla_decode_one(q: np.ndarray, keys: np.ndarray, sm_scale: float, sink=None):
    """Softmax attention of ``q [H, 576]`` over ``keys [n, 576]`` with ``V = keys[:, :512]``.

    ``x[h, t] = sm_scale * q[h] . keys[t]``;  ``lse[h] = log(sum_t exp(x[h, t]) [+ exp(sink[h])])``;
    ``out[h] = sum_t exp(x[h, t] - lse[h]) * keys[t, :512]``.  ``sink [H]`` (optional) is an
    extra logit per head with no value.  With ``n = 0`` and no sink: out 0, lse -inf.
    """
    H = q.shape[0]
    n = keys.shape[0]
    x = np.float64(sm_scale) * (q @ keys.T) if n else np.zeros((H, 0))  # [H, n]
    logits = x if sink is None else np.concatenate([x, np.asarray(sink, np.float64)[:, None]], axis=1)
    if logits.shape[1] == 0:
        return np.zeros((H, LATENT_DIM)), np.full((H,), -np.inf)
    m = logits.max(axis=1)
    empty = np.isneginf(m)  # every logit -inf (nothing visible and a -inf sink): sum is 0
    ms = np.where(empty, 0.0, m)
    z = np.exp(logits - ms[:, None]).sum(axis=1)
    with np.errstate(divide="ignore"):
        lse = np.where(empty, -np.inf, ms + np.log(np.where(empty, 1.0, z)))
    p = np.exp(x - np.where(empty, 0.0, lse)[:, None])
    p[empty] = 0.0
    return p @ keys[:, :LATENT_DIM], lse


def window_range(n_visible: int, window: int):
    """Positions a query with ``n_visible`` visible positions attends under a sliding window
    of ``window`` (0: no window): ``[max(0, n_visible - window), n_visible)``."""
    lo = n_visible - window if window > 0 and n_visible > window else 0
    return lo, n_visible


def mla_decode_ref(q_nope_bits, q_pe_bits, cache, block_table, seq_lens, sm_scale: float,
                   kv_dtype: str = "bf16", kv_scale: float = 1.0, page_size: int = 64,
                   rows=None, window: int = 0, sinks=None):
    """Reference decode.  ``q_nope_bits [B, q_len, H, 512]`` / ``q_pe_bits [B, q_len, H, 64]``
    are bf16 bit patterns (uint16); ``block_table [B, max_pages]`` / ``seq_lens [B]`` int.
    Returns float64 ``out [B, q_len, H, 512]`` and ``lse [B, q_len, H]``.  ``rows`` (optional)
    restricts the work to a list of ``(b, i)`` pairs; the other entries stay NaN.
    ``window`` / ``sinks [H]``: the sliding window and per-head sinks (see the header)."""
    B, q_len, H, _ = q_nope_bits.shape
    out = np.full((B, q_len, H, LATENT_DIM), np.nan)
    lse = np.full((B, q_len, H), np.nan)
    want = rows if rows is not None else [(b, i) for b in range(B) for i in range(q_len)]
    cached = {}
    for b, i in want:
        L = int(seq_lens[b])
        if b not in cached:
            cached = {b: gather_tokens(cache, block_table[b], L, kv_dtype, page_size, kv_scale)}
        lo, hi = window_range(visible_len(L, q_len, i), window)
        keys = cached[b][lo:hi]
        q = _query_rows(q_nope_bits[b, i], q_pe_bits[b, i])
        out[b, i], lse[b, i] = mla_decode_one(q, keys, sm_scale, sink=sinks)
    return out, lse


# --------------------------------------------------------------------------------------
# The split model: partial (o_s, lse_s) per KV range, and the LSE-weighted combine
# --------------------------------------------------------------------------------------

def mla_partial_ref(q: np.ndarray, keys: np.ndarray, t0: int, t1: int, n_visible: int,
                    sm_scale: float):
    """Partial result of one split covering positions ``[t0, t1)``: the same softmax over
    the visible positions inside the range, normalised within the split.  ``o_s [H, 512]``,
    ``lse_s [H]``; a split with no visible position gives ``o_s = 0, lse_s = -inf``."""
    hi = min(t1, n_visible)
    return mla_decode_one(q, keys[t0:hi] if hi > t0 else keys[:0], sm_scale)


def combine_ref(o_parts, lse_parts):
    """LSE-weighted combine of split partials (TileGym ``splitk_reduce``):
    ``lse = M + log sum_s exp(lse_s - M)`` with ``M = max_s lse_s``, and
    ``out = sum_s exp(lse_s - lse) * o_s``.  If every split is empty: out 0, lse -inf."""
    o_parts = np.asarray(o_parts, dtype=np.float64)  # [S, H, 512]
    lse_parts = np.asarray(lse_parts, dtype=np.float64)  # [S, H]
    M = lse_parts.max(axis=0)  # [H]
    empty = ~np.isfinite(M)
    Ms = np.where(empty, 0.0, M)
    w = np.exp(lse_parts - Ms[None, :])  # exp(-inf) = 0 for empty splits
    tot = w.sum(axis=0)
    with np.errstate(divide="ignore"):
        lse = np.where(empty, -np.inf, Ms + np.log(np.where(empty, 1.0, tot)))
    wn = np.where(empty[None, :], 0.0, w / np.where(empty, 1.0, tot)[None, :])
    out = (wn[:, :, None] * o_parts).sum(axis=0)
    return out, lse


def forced_split_ranges(n_tokens: int, num_splits: int, tile: int = 64):
    """KV ranges for a forced split count: span = cdiv(n_tokens, num_splits) rounded up to
    a whole tile, so a 256-token request in 2 splits gives 2 x 128 (the TileGym call's
    power-of-two span of at least 128 for that case)."""
    if n_tokens <= 0:
        return [(0, 0)]
    span = -(-n_tokens // num_splits)
    span = -(-span // tile) * tile
    return [(t, min(t + span, n_tokens)) for t in range(0, n_tokens, span)]


def mla_decode_split_ref(q_nope_bits, q_pe_bits, cache, block_table, seq_lens, sm_scale: float,
                         splits_for, kv_dtype: str = "bf16", kv_scale: float = 1.0,
                         page_size: int = 64):
    """Split-KV decode in float64: for each ``(b, i)``, ``splits_for(b, i, n_visible)`` gives
    a list of ``(t0, t1)`` ranges; each range's partial is computed on its own and the
    partials are combined with :func:`combine_ref`.  Returns ``out, lse, partials`` where
    ``partials[(b, i)] = (o_parts [S, H, 512], lse_parts [S, H])``."""
    B, q_len, H, _ = q_nope_bits.shape
    out = np.zeros((B, q_len, H, LATENT_DIM))
    lse = np.zeros((B, q_len, H))
    partials = {}
    for b in range(B):
        L = int(seq_lens[b])
        keys = gather_tokens(cache, block_table[b], L, kv_dtype, page_size, kv_scale)
        for i in range(q_len):
            nv = visible_len(L, q_len, i)
            q = _query_rows(q_nope_bits[b, i], q_pe_bits[b, i])
            o_s, l_s = [], []
            for t0, t1 in splits_for(b, i, nv):
                o, l = mla_partial_ref(q, keys, t0, t1, nv, sm_scale)
                o_s.append(o)
                l_s.append(l)
            partials[(b, i)] = (np.stack(o_s), np.stack(l_s))
            out[b, i], lse[b, i] = combine_ref(o_s, l_s)
    return out, lse, partials


# Integer helpers of the TileGym wrapper (``next_power_of_2``, ``cdiv``) and its split
# heuristic; kept here so tests can state what that wrapper would choose.

def next_power_of_2(n: int) -> int:
    """Smallest power of two that is >= n (1 for n <= 0)."""
    return 1 if n <= 0 else 1 << (int(n) - 1).bit_length()


def cdiv(a: int, b: int) -> int:
    return -(-int(a) // int(b))


def tilegym_split_heuristic(num_sms: int, batch: int, s_kv: int, tile_n: int = 128):
    """TileGym ``forward``: estimate ``max(1, SMs // B)`` splits, span = next power of two of
    ``S_kv // estimate`` but at least one 128-token tile, split count = cdiv(S_kv, span)."""
    est = max(1, num_sms // batch)
    span = max(next_power_of_2(s_kv // est), tile_n)
    return span, cdiv(s_kv, span)


def workspace_bytes_formula(B: int, H: int, q_len: int, splits: int, D: int = LATENT_DIM,
                            acc_bytes: int = 4) -> int:
    """tokenspeed's split workspace size: ``B * H * q_len * splits * (D + 1) * acc_bytes``."""
    return B * H * q_len * splits * (D + 1) * acc_bytes
