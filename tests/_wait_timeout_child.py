"""Child process of tests/test_gpu_wait_timeout.py (run in a fresh process so that the
test build of the library never shares a process with the tests' own).

It loads the fault-injection build of the library (same sources; every bounded wait gives
up after 20 ms; one CTA can be told to leave one tile unloaded), runs one decode in which
CTA 0 skips the loads of its third tile, then the same decode with nothing skipped, then
the same decode through the shipped library, and prints one JSON line with what it saw."""
import ctypes
import json
import os
import sys
import time

import numpy as np
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))
sys.path.insert(0, HERE)

from mla_latent_kv_split_gb300 import binding as mb  # noqa: E402
from mla_latent_kv_split_gb300 import build  # noqa: E402
from mla_latent_kv_split_gb300 import workloads as W  # noqa: E402

from gpu_util import assert_close, oracle_ref, to_device  # noqa: E402


def main():
    F = ctypes.CDLL(build.build(fault_injection=True))
    P, I, Fl, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    F.mla_decode.restype = I
    F.mla_decode.argtypes = [P, P, P, P, I, P, I, I, I, I, I, Fl, I, Fl, I, P, Z, P, P, P]
    F.mla_decode_read_status.restype = I
    F.mla_decode_read_status.argtypes = [P, ctypes.POINTER(ctypes.c_uint32), P]
    F.mla_fault_injection_drop_tile.restype = I
    F.mla_fault_injection_drop_tile.argtypes = [I, I]

    # one request of 16 full tiles, forced into one part: the first 2-CTA worker takes it all
    w = W.WORKLOADS["paged_bf16_uniform"].scaled(B=1, seq_len=1024, num_splits=1)
    inp = W.make_inputs(w)
    dev = to_device(inp)
    ws = mb.alloc_workspace(w.B, w.q_len, w.H, w.num_splits)
    out = torch.empty((w.B, w.q_len, w.H, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((w.B, w.q_len, w.H), dtype=torch.float32, device="cuda")

    def call():
        rc = F.mla_decode(dev["q_nope"].data_ptr(), dev["q_pe"].data_ptr(), dev["cache"].data_ptr(),
                          dev["block_table"].data_ptr(), dev["block_table"].shape[1], dev["seq_lens"].data_ptr(),
                          w.B, w.q_len, w.H, inp["num_pages"], w.page_size, w.sm_scale, mb.KV_DTYPE[w.kv_dtype],
                          inp["kv_scale"], w.num_splits, ws.data_ptr(), ws.numel(), out.data_ptr(), lse.data_ptr(),
                          None)
        torch.cuda.synchronize()
        st = ctypes.c_uint32(0)
        F.mla_decode_read_status(ws.data_ptr(), ctypes.byref(st), None)
        return rc, int(st.value)

    res = {}
    assert F.mla_fault_injection_drop_tile(0, 2) == 0
    t0 = time.perf_counter()
    res["dropped_rc"], res["dropped_status"] = call()
    res["dropped_seconds"] = time.perf_counter() - t0
    assert F.mla_fault_injection_drop_tile(-1, -1) == 0
    res["next_rc"], res["next_status"] = call()
    ref_out, ref_lse = oracle_ref(inp)
    try:
        assert_close(out.float().cpu().double().numpy(), lse.cpu().double().numpy(), ref_out, ref_lse,
                     what="after the abort, test build")
        res["next_matches_oracle"] = True
    except AssertionError as e:
        res["next_matches_oracle"] = str(e)
    o, l = mb.mla_decode(dev["q_nope"], dev["q_pe"], dev["cache"], dev["block_table"], dev["seq_lens"],
                         w.sm_scale, w.kv_dtype, inp["kv_scale"], w.num_splits, page_size=w.page_size,
                         num_pages=inp["num_pages"], workspace=ws)
    res["shipped_status"] = mb.mla_decode_read_status(ws)
    try:
        assert_close(o.float().cpu().double().numpy(), l.cpu().double().numpy(), ref_out, ref_lse,
                     what="after the abort, shipped library")
        res["shipped_matches_oracle"] = True
    except AssertionError as e:
        res["shipped_matches_oracle"] = str(e)
    print("RESULT " + json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
