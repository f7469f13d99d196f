"""Seeded synthetic inputs for paged MLA decode.

This module only DRAWS inputs: random queries, random page permutations, random cache
values and their storage encoding (bf16 rounding, FP8 E4M3 with a per-tensor scale,
NVFP4 = E2M1 nibbles with an E4M3 scale per 16 values).  It holds none of the decode's
arithmetic, so both the CUDA path's tests and the float64 oracle can take their inputs
from here without sharing any of the method.

Every array is produced on the CPU from one ``torch.Generator`` seeded per workload, in
a fixed draw order: ``seq_lens`` (ragged workloads), the page permutation, ``q_nope``,
``q_pe``, then the cache values, page-chunk by page-chunk.  Everything is returned as
NumPy arrays of the stored bit patterns (uint16 for bf16, uint8 for FP8 / NVFP4).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import numpy as np
import torch

LATENT = 512
ROPE = 64
DIM = LATENT + ROPE  # 576 values per cached token
GROUP = 16  # NVFP4: values per E4M3 block scale
E4M3_MAX = 448.0
E2M1_MAX = 6.0
KV_DTYPES = ("bf16", "fp8", "nvfp4")


def nvfp4_page_bytes(page_size: int) -> int:
    """Bytes per NVFP4 page: ``page_size * 288`` packed E2M1 bytes, then
    ``page_size * 36`` E4M3 scales."""
    return page_size * DIM // 2 + page_size * DIM // GROUP


@dataclass(frozen=True)
class Workload:
    """One decode call's shape and input recipe."""

    name: str
    B: int
    q_len: int
    H: int
    page_size: int
    kv_dtype: str
    seq_len: int | None = None  # uniform length; None -> ragged draw
    ragged: tuple[int, int] | None = None  # inclusive range of the ragged lengths
    sm_scale: float = 1.0 / math.sqrt(192.0)
    num_splits: int = 0  # 0 = schedule from the SM count, >0 = forced per request
    identity_table: bool = False  # contiguous cache: pages 0..n-1 in order
    seed: int = 0
    extra_pages: int = 0  # unused pages appended to the pool (poisoned with NaN/garbage)
    seq_lens_override: tuple[int, ...] | None = field(default=None)

    def scaled(self, **kw) -> "Workload":
        return replace(self, **kw)


# The five workloads the measurements and parity tests are quoted on.
WORKLOADS = {
    "tiny_contig_bf16": Workload("tiny_contig_bf16", B=1, q_len=1, H=16, page_size=64,
                                 kv_dtype="bf16", seq_len=256, num_splits=2,
                                 identity_table=True),
    "paged_bf16_uniform": Workload("paged_bf16_uniform", B=32, q_len=1, H=128, page_size=64,
                                   kv_dtype="bf16", seq_len=4096),
    "paged_bf16_ragged": Workload("paged_bf16_ragged", B=64, q_len=1, H=128, page_size=64,
                                  kv_dtype="bf16", ragged=(128, 32768)),
    "paged_fp8": Workload("paged_fp8", B=128, q_len=1, H=128, page_size=64, kv_dtype="fp8",
                          seq_len=8192),
    "paged_nvfp4_verify4": Workload("paged_nvfp4_verify4", B=8, q_len=4, H=128, page_size=64,
                                    kv_dtype="nvfp4", seq_len=131072),
}


def _bf16_bits(x: torch.Tensor) -> np.ndarray:
    """float32 tensor -> bf16 bit patterns (round to nearest even)."""
    return x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def quantize_e4m3_rne(x: torch.Tensor) -> np.ndarray:
    """float32 tensor (already within +-448) -> E4M3 codes, round to nearest even."""
    return x.clamp(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


_E2M1_MIDS = torch.tensor([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], dtype=torch.float32)


def quantize_e2m1_rne(v: torch.Tensor) -> torch.Tensor:
    """float32 tensor -> E2M1 codes (uint8, 0..15): nearest of +-{0,.5,1,1.5,2,3,4,6},
    ties to the even code, saturating at 6."""
    a = v.abs().clamp(max=E2M1_MAX)
    code = torch.searchsorted(_E2M1_MIDS, a.contiguous(), right=False)
    tie = a == _E2M1_MIDS[code.clamp(max=6)]
    code = code + (tie & (code % 2 == 1)).to(code.dtype)
    sign = (v < 0).to(code.dtype) << 3
    return (code | sign).to(torch.uint8)


def quantize_nvfp4_pages(x: torch.Tensor) -> np.ndarray:
    """float32 ``[n_pages, page_size, 576]`` -> NVFP4 pages ``[n_pages, page_bytes]`` uint8.

    Per 16-value group: ``s = RNE_e4m3(amax / 6)``; each element's code is the E2M1
    rounding of ``x / s`` (all zero when ``s`` is 0).  Data bytes are token-major with
    element ``2j`` in the low nibble of byte ``j``; the scale bytes follow, token-major.
    """
    n, ps, d = x.shape
    g = x.reshape(n, ps, d // GROUP, GROUP)
    amax = g.abs().amax(dim=-1)  # [n, ps, 36]
    s_code = (amax / E2M1_MAX).to(torch.float8_e4m3fn)
    s_val = s_code.to(torch.float32)
    safe = torch.where(s_val > 0, s_val, torch.ones_like(s_val))
    q = quantize_e2m1_rne(g / safe[..., None])
    q = torch.where((s_val > 0)[..., None], q, torch.zeros_like(q)).reshape(n, ps, d)
    packed = (q[..., 0::2] | (q[..., 1::2] << 4)).to(torch.uint8)  # [n, ps, 288]
    out = torch.cat([packed.reshape(n, -1), s_code.view(torch.uint8).reshape(n, -1)], dim=1)
    return out.numpy()


def draw_seq_lens(w: Workload, g: torch.Generator) -> np.ndarray:
    if w.seq_lens_override is not None:
        return np.asarray(w.seq_lens_override, dtype=np.int32)
    if w.ragged is not None:
        lo, hi = w.ragged
        return torch.randint(lo, hi + 1, (w.B,), generator=g, dtype=torch.int64).numpy().astype(np.int32)
    return np.full((w.B,), int(w.seq_len), dtype=np.int32)


def make_inputs(w: Workload, chunk_pages: int = 1024) -> dict:
    """Draw one workload's inputs.  Returns a dict of NumPy arrays and scalars:

    ``q_nope [B,q_len,H,512]`` / ``q_pe [B,q_len,H,64]`` (uint16 bf16 bits),
    ``cache`` (uint16 ``[P,ps,576]`` | uint8 ``[P,ps,576]`` | uint8 ``[P,page_bytes]``),
    ``block_table [B, max_pages]`` int32 (zero beyond each request's pages),
    ``seq_lens [B]`` int32, ``kv_scale`` (float; 1.0 unless FP8), ``num_pages``.
    """
    g = torch.Generator().manual_seed(w.seed)
    seq_lens = draw_seq_lens(w, g)
    ps = w.page_size
    pages_per = [-(-int(L) // ps) for L in seq_lens]
    n_used = int(sum(pages_per))
    num_pages = n_used + w.extra_pages
    max_pages = max(1, max(pages_per) if pages_per else 1)
    if w.identity_table:
        perm = np.arange(num_pages, dtype=np.int32)
    else:
        perm = torch.randperm(num_pages, generator=g).numpy().astype(np.int32)
    table = np.zeros((w.B, max_pages), dtype=np.int32)
    off = 0
    for b, n in enumerate(pages_per):
        table[b, :n] = perm[off:off + n]
        off += n
    q_nope = _bf16_bits(torch.randn((w.B, w.q_len, w.H, LATENT), generator=g))
    q_pe = _bf16_bits(torch.randn((w.B, w.q_len, w.H, ROPE), generator=g))

    kv_scale = 1.0
    if w.kv_dtype == "bf16":
        cache = np.empty((num_pages, ps, DIM), dtype=np.uint16)
    elif w.kv_dtype == "fp8":
        cache = np.empty((num_pages, ps, DIM), dtype=np.uint8)
    elif w.kv_dtype == "nvfp4":
        cache = np.empty((num_pages, nvfp4_page_bytes(ps)), dtype=np.uint8)
    else:
        raise ValueError(w.kv_dtype)

    state = g.get_state()
    if w.kv_dtype == "fp8":  # per-tensor scale needs the global amax first
        amax = 0.0
        for p0 in range(0, num_pages, chunk_pages):
            n = min(chunk_pages, num_pages - p0)
            amax = max(amax, float(torch.randn((n, ps, DIM), generator=g).abs().max()))
        g.set_state(state)
        kv_scale = float(np.float32(amax / E4M3_MAX)) if amax > 0 else 1.0
    for p0 in range(0, num_pages, chunk_pages):
        n = min(chunk_pages, num_pages - p0)
        x = torch.randn((n, ps, DIM), generator=g)
        if w.kv_dtype == "bf16":
            cache[p0:p0 + n] = _bf16_bits(x)
        elif w.kv_dtype == "fp8":
            cache[p0:p0 + n] = quantize_e4m3_rne(x / torch.tensor(kv_scale, dtype=torch.float32))
        else:
            cache[p0:p0 + n] = quantize_nvfp4_pages(x)
    return dict(q_nope=q_nope, q_pe=q_pe, cache=cache, block_table=table,
                seq_lens=seq_lens, kv_scale=kv_scale, num_pages=num_pages,
                workload=w)


def draw_sinks(H: int, seed: int = 0, lo: float = 0.0, hi: float = 12.0) -> np.ndarray:
    """Per-head sink logits ``[H]`` float32 for the attention-sink cases: uniform in
    ``[lo, hi]`` (the range of a decode's log-sum-exp over a few to tens of thousands of
    positions at these query/key scales), with every 8th head at -inf (a head without a
    sink) and head 1 at ``hi + 20`` (a sink that takes nearly all of the weight)."""
    g = torch.Generator().manual_seed(1000 + seed)
    s = (lo + (hi - lo) * torch.rand((H,), generator=g)).numpy().astype(np.float32)
    s[::8] = -np.inf
    if H > 1:
        s[1] = np.float32(hi + 20.0)
    return s


def poison_unused(inp: dict, rng_seed: int = 1) -> None:
    """Overwrite every cache position a request never reads (tails of its last page and
    whole unused pages) with NaN / garbage bytes, in place."""
    w: Workload = inp["workload"]
    cache = inp["cache"]
    ps = w.page_size
    used_rows = {}
    for b in range(w.B):
        L = int(inp["seq_lens"][b])
        n = -(-L // ps)
        for j in range(n):
            p = int(inp["block_table"][b, j])
            used_rows[p] = min(ps, L - j * ps) if j == n - 1 else ps
    rng = np.random.default_rng(rng_seed)
    for p in range(cache.shape[0]):
        k = used_rows.get(p, 0)
        if k >= ps:
            continue
        if w.kv_dtype == "bf16":
            cache[p, k:] = 0x7FC1  # quiet NaN
        elif w.kv_dtype == "fp8":
            cache[p, k:] = 0x7F  # E4M3 NaN
        else:
            data = cache[p, : ps * DIM // 2].reshape(ps, DIM // 2)
            scl = cache[p, ps * DIM // 2:].reshape(ps, DIM // GROUP)
            data[k:] = rng.integers(0, 256, size=data[k:].shape, dtype=np.uint8)
            scl[k:] = 0x7F  # NaN scale
