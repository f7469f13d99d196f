"""GPU parity of the sliding window and the per-head attention sinks (metrale
"kv_cache_mla.rs", mla_paged_decode_fp8's sliding_window and sinks) against the float64
oracle: every cache format, page sizes 32 and 64, one and two queries per request, windows
inside, on and across tile edges and longer than the sequence, with the library's split
schedule and with forced splits (so the sink is applied both where a unit is written
directly and in the split-K combine), and requests that see nothing."""
import numpy as np
import pytest

import oracle
from mla_latent_kv_split_gb300 import workloads as W

from gpu_util import assert_close, ensure_built, oracle_ref, run_decode

pytestmark = pytest.mark.gpu

SEQ_LT_QLEN = 0x4  # a request shorter than its q_len (seq_len 0 here) is reported, not an error


def _expected_status(inp):
    return SEQ_LT_QLEN if int(np.min(inp["seq_lens"])) < inp["workload"].q_len else 0


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()


LENS = (0, 1, 63, 64, 65, 700, 2000, 129)


@pytest.mark.parametrize("num_splits", [0, 3])
@pytest.mark.parametrize("window", [1, 63, 64, 65, 100, 640, 5000])
@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8"])
def test_window_parity(kv_dtype, window, num_splits):
    w = W.WORKLOADS["paged_fp8"].scaled(B=len(LENS), H=32, kv_dtype=kv_dtype, seq_lens_override=LENS)
    inp = W.make_inputs(w)
    out, lse, status, _ = run_decode(inp, num_splits=num_splits, window=window)
    assert status == _expected_status(inp), hex(status)
    assert_close(out, lse, *oracle_ref(inp, window=window), what=f"{kv_dtype} W{window} n{num_splits}")


@pytest.mark.parametrize("num_splits", [0, 2, 5])
@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8", "nvfp4"])
def test_sinks_parity(kv_dtype, num_splits):
    w = W.WORKLOADS["paged_fp8"].scaled(B=len(LENS), H=64, kv_dtype=kv_dtype, seq_lens_override=LENS)
    inp = W.make_inputs(w)
    sinks = W.draw_sinks(w.H, seed=3)
    out, lse, status, _ = run_decode(inp, num_splits=num_splits, sinks=sinks)
    assert status == _expected_status(inp), hex(status)
    assert_close(out, lse, *oracle_ref(inp, sinks=sinks), what=f"{kv_dtype} sinks n{num_splits}")


@pytest.mark.parametrize("ps", [32, 64])
@pytest.mark.parametrize("num_splits", [0, 4])
@pytest.mark.parametrize("kv_dtype", ["fp8", "nvfp4", "bf16"])
def test_window_and_sinks_verify(kv_dtype, num_splits, ps):
    # two queries per request: each query's window ends at its own newest position
    w = W.WORKLOADS["paged_fp8"].scaled(B=5, q_len=2, H=32, page_size=ps, kv_dtype=kv_dtype,
                                        seq_lens_override=(1, 2, 300, 1025, 4000))
    inp = W.make_inputs(w)
    sinks = W.draw_sinks(w.H, seed=5)
    for window in (33, 128, 1000):
        out, lse, status, _ = run_decode(inp, num_splits=num_splits, window=window, sinks=sinks)
        assert status == _expected_status(inp), hex(status)
        assert_close(out, lse, *oracle_ref(inp, window=window, sinks=sinks),
                     what=f"{kv_dtype} ps{ps} W{window} n{num_splits}")


def test_full_size_fp8_window_sinks_every_row():
    # the FP8 workload at full size (B=128, 8192 tokens, H=128) with a 4096-token window and
    # sinks, in the library's own schedule; every row against the oracle
    w = W.WORKLOADS["paged_fp8"].scaled(seed=9)
    inp = W.make_inputs(w)
    sinks = W.draw_sinks(w.H, seed=9)
    out, lse, status, _ = run_decode(inp, window=4096, sinks=sinks)
    assert status == _expected_status(inp), hex(status)
    ref_out, ref_lse = oracle_ref(inp, window=4096, sinks=sinks)
    assert_close(out, lse, ref_out, ref_lse, what="fp8 full W4096 sinks")
