"""Queries across the whole bf16 range on the quantized caches.  FP8 and NVFP4 caches
multiply in f16, so each query row is brought into f16's range by a power of two chosen
from that row before the conversion and the partial scores are scaled back; rows far
above 65504 or far below f16's normal range must decode as exactly as ordinary ones.

The scale of the scores stays moderate through sm_scale (an explicit argument of the
call): rows multiplied by ~1e5..1e6 run with a small sm_scale, rows multiplied by
~1e-6..1e-5 with a large one, so that the log-sum-exp stays within the range where its
fp32 value resolves the 1e-3 tolerance."""
import math

import numpy as np
import pytest
import torch

from mla_latent_kv_split_gb300 import workloads as W

from gpu_util import assert_close, ensure_built, oracle_ref, run_decode

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()


def _scale_rows(bits: np.ndarray, f: np.ndarray) -> np.ndarray:
    """bf16 bit patterns [B, q_len, H, D] times a per-head factor f[H], rounded to bf16."""
    x = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float()
    y = (x * torch.from_numpy(f.astype(np.float32)).view(1, 1, -1, 1)).to(torch.bfloat16)
    return y.view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("kv_dtype", ["fp8", "nvfp4", "bf16"])
@pytest.mark.parametrize("band", ["large", "small", "mixed"])
def test_query_rows_across_the_bf16_range(kv_dtype, band):
    H = 64
    w = W.WORKLOADS["paged_fp8"].scaled(B=3, q_len=2, H=H, kv_dtype=kv_dtype, seq_lens_override=(700, 64, 1500))
    rng = np.random.default_rng({"large": 1, "small": 2, "mixed": 3}[band])
    base = 1.0 / math.sqrt(192.0)
    if band == "large":    # |q| up to ~4e6, far beyond f16's 65504
        f = 10.0 ** rng.uniform(5.0, 6.0, H)
        sm = base / 3e5
    elif band == "small":  # |q| down to ~1e-7, below f16's normal range
        f = 10.0 ** rng.uniform(-6.5, -5.0, H)
        sm = base * 3e5
    else:                  # unscaled rows next to scaled ones in the same warps
        f = np.where(np.arange(H) % 2 == 0, 1.0, 10.0 ** rng.uniform(-6.0, -5.0, H))
        sm = base
    w = w.scaled(sm_scale=sm)
    inp = W.make_inputs(w)
    inp["q_nope"] = _scale_rows(inp["q_nope"], f)
    inp["q_pe"] = _scale_rows(inp["q_pe"], f)
    out, lse, status, _ = run_decode(inp)
    assert status == 0, hex(status)
    ref_out, ref_lse = oracle_ref(inp)
    assert_close(out, lse, ref_out, ref_lse, what=f"{kv_dtype} q {band}")


@pytest.mark.parametrize("kv_dtype", ["fp8", "nvfp4"])
def test_query_range_with_forced_splits_and_a_window(kv_dtype):
    H = 32
    w = W.WORKLOADS["paged_fp8"].scaled(B=2, q_len=1, H=H, kv_dtype=kv_dtype, seq_lens_override=(900, 333),
                                        sm_scale=1.0 / math.sqrt(192.0) / 1e5)
    inp = W.make_inputs(w)
    f = np.full(H, 1e5)
    f[::4] = 3e5
    inp["q_nope"] = _scale_rows(inp["q_nope"], f)
    inp["q_pe"] = _scale_rows(inp["q_pe"], f)
    for ns, window in ((3, 0), (0, 200)):
        out, lse, status, _ = run_decode(inp, num_splits=ns, window=window)
        assert status == 0, hex(status)
        assert_close(out, lse, *oracle_ref(inp, window=window), what=f"{kv_dtype} n{ns} W{window}")
