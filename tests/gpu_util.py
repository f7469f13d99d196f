"""Helpers for the GPU parity tests: upload seeded inputs, call the library through the
C ABI binding, and compare with the float64 oracle at the stated tolerance."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from mla_latent_kv_split_gb300 import binding as mb

# Tolerance of the decode: |out - ref| <= ATOL + RTOL*|ref| on the bf16 output and
# |lse - ref| <= LSE_ATOL on the fp32 log-sum-exp.  Relative L2 error of the output is
# also gated (REL_L2) to catch kernels that are wrong but inside the elementwise bound.
ATOL, RTOL, LSE_ATOL, REL_L2 = 1e-2, 1e-2, 1e-3, 5e-3


def ensure_built():
    from mla_latent_kv_split_gb300 import build
    build.build()
    return mb.lib()


def to_device(inp: dict, device="cuda"):
    w = inp["workload"]
    d = {}
    d["q_nope"] = torch.from_numpy(inp["q_nope"].view(np.int16)).view(torch.bfloat16).to(device)
    d["q_pe"] = torch.from_numpy(inp["q_pe"].view(np.int16)).view(torch.bfloat16).to(device)
    cache = inp["cache"]
    if cache.dtype == np.uint16:
        d["cache"] = torch.from_numpy(cache.view(np.int16)).view(torch.bfloat16).to(device)
    else:
        d["cache"] = torch.from_numpy(cache).to(device)
    d["block_table"] = torch.from_numpy(inp["block_table"]).to(device)
    d["seq_lens"] = torch.from_numpy(inp["seq_lens"]).to(device)
    return d


def run_decode(inp: dict, dev: dict | None = None, num_splits=None, workspace=None, out=None, lse=None,
               window: int = 0, sinks=None):
    w = inp["workload"]
    dev = dev or to_device(inp)
    ns = w.num_splits if num_splits is None else num_splits
    if workspace is None:
        workspace = mb.alloc_workspace(w.B, w.q_len, w.H, ns)
    d_sinks = None if sinks is None else torch.from_numpy(np.asarray(sinks, np.float32)).cuda()
    out, lse = mb.mla_decode(dev["q_nope"], dev["q_pe"], dev["cache"], dev["block_table"], dev["seq_lens"],
                             w.sm_scale, w.kv_dtype, inp["kv_scale"], ns, page_size=w.page_size,
                             num_pages=inp["num_pages"], workspace=workspace, out=out, lse=lse,
                             window=window, sinks=d_sinks)
    status = mb.mla_decode_read_status(workspace)
    torch.cuda.synchronize()
    o = out.float().cpu().double().numpy()
    l = lse.cpu().double().numpy()
    return o, l, status, workspace


def oracle_ref(inp: dict, rows=None, window: int = 0, sinks=None):
    w = inp["workload"]
    return oracle.mla_decode_ref(inp["q_nope"], inp["q_pe"], inp["cache"], inp["block_table"], inp["seq_lens"],
                                 w.sm_scale, kv_dtype=w.kv_dtype, kv_scale=inp["kv_scale"],
                                 page_size=w.page_size, rows=rows, window=window,
                                 sinks=None if sinks is None else np.asarray(sinks, np.float64))


def assert_close(out, lse, ref_out, ref_lse, rows=None, what=""):
    if rows is not None:
        idx = tuple(np.array(rows).T)
        out, lse, ref_out, ref_lse = out[idx], lse[idx], ref_out[idx], ref_lse[idx]
    fin = np.isfinite(ref_lse)
    assert np.array_equal(fin, np.isfinite(lse)), f"{what}: -inf pattern of lse differs"
    assert np.all(np.isfinite(out)), f"{what}: non-finite output"
    err = np.abs(out - ref_out)
    bound = ATOL + RTOL * np.abs(ref_out)
    worst = np.unravel_index(np.argmax(err - bound), err.shape)
    assert np.all(err <= bound), f"{what}: out err {err[worst]:.3g} > {bound[worst]:.3g} at {worst}"
    if fin.any():
        le = np.abs(lse[fin] - ref_lse[fin]).max()
        assert le <= LSE_ATOL, f"{what}: lse err {le:.3g}"
    assert np.all(out[~fin] == 0), f"{what}: empty rows must be 0"
    empty = np.all(ref_out == 0, axis=-1)  # nothing visible (a finite sink still sets lse)
    assert np.all(out[empty] == 0), f"{what}: rows with nothing visible must be 0"
    den = np.linalg.norm(ref_out)
    if den > 0:
        rel = np.linalg.norm(out - ref_out) / den
        assert rel <= REL_L2, f"{what}: rel L2 {rel:.3g}"
