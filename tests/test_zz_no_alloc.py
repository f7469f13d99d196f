"""mla_decode_no_alloc: the decode for callers that cannot allocate device memory (code run
inside another runtime that owns all device allocations, or a process whose device
footprint must stay fixed).  Its scratch is a static buffer inside the library, so these
tests check, through the C ABI, that two calls in a row give the same results as
mla_decode with a caller-allocated workspace, and that shapes needing more scratch than
the buffer holds are refused.  Collected last on purpose (file name)."""
import ctypes

import numpy as np
import pytest
import torch

from mla_latent_kv_split_gb300 import binding as mb
from mla_latent_kv_split_gb300 import workloads as W

from gpu_util import ATOL, LSE_ATOL, RTOL, ensure_built, run_decode, to_device

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 48 << 20


def _call_c(L, dev, inp, out, lse, num_splits):
    w = inp["workload"]
    scratch = ctypes.c_void_p(0)
    code = L.mla_decode_no_alloc(
        dev["q_nope"].data_ptr(), dev["q_pe"].data_ptr(), dev["cache"].data_ptr(), dev["block_table"].data_ptr(),
        int(inp["block_table"].shape[1]), dev["seq_lens"].data_ptr(), w.B, w.q_len, w.H, int(inp["num_pages"]),
        w.page_size, float(w.sm_scale), mb.KV_DTYPE[w.kv_dtype], float(inp["kv_scale"]), int(num_splits),
        out.data_ptr(), lse.data_ptr(), torch.cuda.current_stream().cuda_stream, ctypes.byref(scratch))
    return code, scratch.value


@pytest.mark.parametrize("kv_dtype,num_splits", [("bf16", 0), ("fp8", 3), ("nvfp4", 0)])
def test_no_alloc_matches_mla_decode_on_two_calls(kv_dtype, num_splits):
    L = ensure_built()
    w = W.WORKLOADS["paged_bf16_ragged"].scaled(B=6, q_len=2 if kv_dtype == "nvfp4" else 1, kv_dtype=kv_dtype,
                                                seq_lens_override=(1500, 64, 1, 3000, 700, 129))
    inp = W.make_inputs(w)
    dev = to_device(inp)
    ref_out, ref_lse, ref_status, _ = run_decode(inp, dev, num_splits=num_splits)
    # q_len 2 with a 1-token request reports SEQ_LT_QLEN on both entry points
    assert ref_status == (0x4 if w.q_len == 2 else 0)
    fin = np.isfinite(ref_lse)
    for call in range(2):
        out = torch.full((w.B, w.q_len, w.H, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.full((w.B, w.q_len, w.H), float("nan"), dtype=torch.float32, device="cuda")
        code, scratch = _call_c(L, dev, inp, out, lse, num_splits)
        assert code == 0, L.mla_status_string(code).decode()
        assert scratch and scratch % 256 == 0
        assert mb.mla_decode_read_status(scratch) == ref_status
        o = out.float().cpu().double().numpy()
        l = lse.cpu().double().numpy()
        assert np.all(np.abs(o - ref_out) <= ATOL + RTOL * np.abs(ref_out)), f"call {call}: output differs"
        assert np.array_equal(np.isfinite(l), fin)
        assert np.all(np.abs(l[fin] - ref_lse[fin]) <= LSE_ATOL), f"call {call}: lse differs"


def test_no_alloc_refuses_shapes_beyond_its_scratch():
    L = ensure_built()
    # 512 (b, i) units x 4 forced splits x 128 heads of partials is far above 48 MiB
    need = mb.mla_decode_workspace_size(256, 2, 128, 4)
    assert need > SCRATCH_BYTES
    w = W.WORKLOADS["paged_bf16_uniform"].scaled(B=256, q_len=2, seq_len=64)
    inp = W.make_inputs(w)
    dev = to_device(inp)
    out = torch.empty((w.B, w.q_len, w.H, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((w.B, w.q_len, w.H), dtype=torch.float32, device="cuda")
    code, _ = _call_c(L, dev, inp, out, lse, 4)
    assert code == 3  # MLA_ERR_WORKSPACE_TOO_SMALL, nothing enqueued
