"""Host-side pieces of bench.py: the algorithmic work it divides by (cache rows read once per
request, the union of the query windows), and the code hash that keys recorded ncu traffic
(comments do not change it, code does)."""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from mla_latent_kv_split_gb300 import workloads as W  # noqa: E402


def test_algorithmic_work_counts_each_cache_row_once():
    w = W.WORKLOADS["paged_fp8"].scaled(B=3, q_len=2, H=16, seq_lens_override=(10, 300, 1))
    inp = W.make_inputs(w)
    nbytes, flops, kv = bench.algorithmic_work(inp)
    assert kv == (10 + 300 + 1) * 576
    # visible positions per query: (9, 10), (299, 300), (0, 1)
    assert flops == 2.0 * 16 * (576 + 512) * (9 + 10 + 299 + 300 + 0 + 1)
    io = 3 * 2 * 16 * (576 * 2 + 512 * 2 + 4)
    table = 4 * (1 + 5 + 1) + 4 * 3
    assert nbytes == kv + io + table


def test_algorithmic_work_with_a_window_reads_the_union_of_the_windows():
    w = W.WORKLOADS["paged_fp8"].scaled(B=3, q_len=2, H=16, seq_lens_override=(10, 300, 1))
    inp = W.make_inputs(w)
    _, flops, kv = bench.algorithmic_work(inp, window=100)
    # request 1: query 0 sees [199, 299), query 1 [200, 300): the union is [199, 300)
    assert kv == (10 + 101 + 1) * 576
    assert flops == 2.0 * 16 * (576 + 512) * (9 + 10 + 100 + 100 + 0 + 1)


def test_code_hash_ignores_comments_only():
    a = "int f(int x) {  // the input\n  return x + 1; /* one\n more */\n}\n"
    b = "// header\nint f(int x) {\n\n  return x + 1;\n}\n"
    c = "int f(int x) {\n  return x + 2;\n}\n"
    assert bench._code_tokens(a) == bench._code_tokens(b)
    assert bench._code_tokens(a) != bench._code_tokens(c)
    assert len(bench.kernel_source_sha()) == 16


def test_roofline_takes_the_binding_resource_of_each_format():
    """bf16 at q_len 1 does 2*128*(576+512) flops per 1152 cache bytes (242 flops/byte), under
    the ridge of the measured peaks, so it is HBM-bound; FP8 (576 bytes per token) and NVFP4
    verify (324 bytes per token, four queries) are tensor-bound.  The fraction is the achieved
    rate over the peak of that bound, and the roofline time the larger of the two times."""
    peaks = {"hbm": 6775.3, "bf16": 1933.3, "source": "measured"}
    tokens, H = 131072, 128
    per_token_flops = 2.0 * H * (576 + 512)
    for bpt, q_len, bound in ((1152, 1, "hbm"), (576, 1, "tensor"), (324, 4, "tensor")):
        nbytes, flops = tokens * bpt, tokens * q_len * per_token_flops
        t_mem, t_mma = nbytes / (peaks["hbm"] * 1e9), flops / (peaks["bf16"] * 1e12)
        t = 2.5 * max(t_mem, t_mma)
        roof = bench._roofline(nbytes, flops, t, peaks)
        assert roof["bound"] == bound
        assert roof["unit"] == ("GB/s" if bound == "hbm" else "TFLOP/s")
        assert abs(roof["frac"] - 0.4) < 1e-12
        assert abs(roof["roofline_us"] - 1e6 * max(t_mem, t_mma)) < 1e-9
        assert roof["peak"] == (peaks["hbm"] if bound == "hbm" else peaks["bf16"])
