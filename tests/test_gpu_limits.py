"""GPU parity at the limits of the build: the largest q_len (8, causal verify), the largest
number of (b, i) units (1024, more work items per scheduling worker than the item ring
holds), forced split counts far above the tile count (every tile its own part) and the
sliding window at q_len 8."""
import numpy as np
import pytest

from mla_latent_kv_split_gb300 import workloads as W

from gpu_util import assert_close, ensure_built, oracle_ref, run_decode

pytestmark = pytest.mark.gpu

SEQ_LT_QLEN = 0x4


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8", "nvfp4"])
def test_q_len_8(kv_dtype):
    inp = W.make_inputs(W.WORKLOADS["paged_nvfp4_verify4"].scaled(
        B=4, q_len=8, H=32, kv_dtype=kv_dtype, seq_lens_override=(8, 9, 100, 1000)))
    out, lse, status, _ = run_decode(inp)
    assert status == 0, hex(status)
    assert_close(out, lse, *oracle_ref(inp), what=f"q_len 8 {kv_dtype}")


def test_q_len_8_window_and_forced_splits():
    inp = W.make_inputs(W.WORKLOADS["paged_fp8"].scaled(B=3, q_len=8, H=16, seq_lens_override=(70, 700, 2000)))
    sinks = W.draw_sinks(16, seed=8)
    for ns, window in ((0, 50), (5, 129)):
        out, lse, status, _ = run_decode(inp, num_splits=ns, window=window, sinks=sinks)
        assert status == 0, hex(status)
        assert_close(out, lse, *oracle_ref(inp, window=window, sinks=sinks), what=f"q8 W{window} n{ns}")


def test_max_units_many_items_per_worker():
    # 1024 short requests: ~13 work items per worker with 76 workers, several hundred with
    # fewer; every output row checked
    inp = W.make_inputs(W.WORKLOADS["paged_bf16_ragged"].scaled(B=1024, H=16, ragged=(0, 300), seed=4))
    out, lse, status, _ = run_decode(inp)
    want = SEQ_LT_QLEN if int(inp["seq_lens"].min()) < 1 else 0
    assert status == want, hex(status)
    assert_close(out, lse, *oracle_ref(inp), what="1024 units")


def test_max_units_q_len_8_sampled():
    inp = W.make_inputs(W.WORKLOADS["paged_fp8"].scaled(B=128, q_len=8, H=16, ragged=(8, 4000), seq_len=None,
                                                        seed=5))
    out, lse, status, _ = run_decode(inp)
    assert status == 0, hex(status)
    rows = [(b, i) for b in (0, 1, 64, 127) for i in range(8)]
    ref_out, ref_lse = oracle_ref(inp, rows=rows)
    assert_close(out, lse, ref_out, ref_lse, rows=rows, what="128 x q_len 8")


@pytest.mark.parametrize("num_splits", [64, 4096])
def test_split_count_above_tile_count(num_splits):
    inp = W.make_inputs(W.WORKLOADS["paged_bf16_uniform"].scaled(B=2, H=16, seq_lens_override=(3000, 65)))
    out, lse, status, _ = run_decode(inp, num_splits=num_splits)
    assert status == 0, hex(status)
    assert_close(out, lse, *oracle_ref(inp), what=f"splits {num_splits}")
