"""Repeated calls on the same inputs: every call must report a clean device status and give
bit-identical results (the schedule, the MMA order and the split-K combine are all fixed),
so a race between the kernel's roles, or a wait that gave up, shows here even when it is
rare.  The cases give each scheduling worker one or many work items, with and without
split partials."""
import numpy as np
import pytest
import torch

from mla_latent_kv_split_gb300 import binding as mb
from mla_latent_kv_split_gb300 import workloads as W

from gpu_util import ensure_built, to_device

pytestmark = pytest.mark.gpu

CASES = {
    # one or two items per worker, every unit split (the bench workload)
    "uniform_full": ("paged_bf16_uniform", dict(), 0, 40),
    # many short items per worker, tails in most tiles
    "ragged_many_items": ("paged_bf16_ragged", dict(B=256, ragged=(1, 700)), 0, 25),
    # forced splits: partials for every unit
    "forced_splits": ("paged_bf16_uniform", dict(B=8, seq_len=3000), 3, 25),
    "fp8": ("paged_fp8", dict(B=32, seq_len=4000), 0, 15),
    "nvfp4_verify": ("paged_nvfp4_verify4", dict(B=2, seq_len=20000), 0, 10),
}


@pytest.mark.parametrize("key", list(CASES))
def test_repeated_calls_identical_and_clean(key):
    ensure_built()
    name, kw, ns, reps = CASES[key]
    w = W.WORKLOADS[name].scaled(**kw)
    inp = W.make_inputs(w)
    dev = to_device(inp)
    ws = mb.alloc_workspace(w.B, w.q_len, w.H, ns)
    first = None
    for k in range(reps):
        out, lse = mb.mla_decode(dev["q_nope"], dev["q_pe"], dev["cache"], dev["block_table"], dev["seq_lens"],
                                 w.sm_scale, w.kv_dtype, inp["kv_scale"], ns, page_size=w.page_size,
                                 num_pages=inp["num_pages"], workspace=ws)
        status = mb.mla_decode_read_status(ws)
        assert status == 0, f"call {k}: device status {status:#x}"
        if first is None:
            first = (out.clone(), lse.clone())
            assert torch.isfinite(out.float()).all()
        else:
            assert torch.equal(out.view(torch.int16), first[0].view(torch.int16)), f"call {k}: output differs"
            assert np.array_equal(lse.cpu().numpy().view(np.int32), first[1].cpu().numpy().view(np.int32)), \
                f"call {k}: lse differs"
