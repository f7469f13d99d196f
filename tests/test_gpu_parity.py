"""GPU parity: the CUDA path through the C ABI against the float64 oracle, element by element,
on seeded inputs of the five workloads' shapes (scaled so the oracle takes seconds, still
spanning several tiles and ragged tails) and the edge cases."""
import numpy as np
import pytest
import torch

import oracle
from mla_latent_kv_split_gb300 import binding as mb
from mla_latent_kv_split_gb300 import workloads as W

from gpu_util import assert_close, ensure_built, oracle_ref, run_decode, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()


def _case(name, **kw):
    return W.make_inputs(W.WORKLOADS[name].scaled(**kw))


SMALL = {
    "tiny_contig_bf16": dict(),
    "uniform_bf16": ("paged_bf16_uniform", dict(B=4, seq_len=1000)),
    "ragged_bf16": ("paged_bf16_ragged", dict(B=8, seq_lens_override=(1, 63, 64, 65, 2000, 3333, 127, 129))),
    "fp8": ("paged_fp8", dict(B=3, seq_lens_override=(700, 64, 1500))),
    "nvfp4_verify4": ("paged_nvfp4_verify4", dict(B=2, seq_lens_override=(300, 5))),
    "nvfp4_q1": ("paged_nvfp4_verify4", dict(B=3, q_len=1, seq_lens_override=(1000, 33, 64))),
    "fp8_verify2": ("paged_fp8", dict(B=2, q_len=2, seq_lens_override=(513, 2))),
}


@pytest.mark.parametrize("key", list(SMALL))
def test_parity_small(key):
    spec = SMALL[key]
    inp = W.make_inputs(W.WORKLOADS[key]) if key == "tiny_contig_bf16" else _case(spec[0], **spec[1])
    out, lse, status, _ = run_decode(inp)
    ref_out, ref_lse = oracle_ref(inp)
    assert status == 0, hex(status)
    assert_close(out, lse, ref_out, ref_lse, what=key)


@pytest.mark.parametrize("H", [16, 32, 64, 128])
@pytest.mark.parametrize("ps", [32, 64])
@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8", "nvfp4"])
def test_parity_heads_pages_dtypes(H, ps, kv_dtype):
    inp = _case("paged_bf16_ragged", B=3, H=H, page_size=ps, kv_dtype=kv_dtype, seq_lens_override=(97, 320, 1))
    out, lse, status, _ = run_decode(inp)
    assert status == 0
    assert_close(out, lse, *oracle_ref(inp), what=f"H{H} ps{ps} {kv_dtype}")


@pytest.mark.parametrize("n", [1, 2, 3, 5, 8])
def test_forced_splits_and_partials(n):
    inp = _case("paged_bf16_uniform", B=2, H=32, seq_lens_override=(450, 130))
    out, lse, status, ws = run_decode(inp, num_splits=n)
    assert status == 0
    assert_close(out, lse, *oracle_ref(inp), what=f"splits={n}")
    # the partials in the workspace match the oracle's split model
    w = inp["workload"]
    pl = mb.mla_decode_plan_host(inp["seq_lens"], 1, inp["block_table"].shape[1], 64, n, mb.mla_decode_num_workers())
    _, _, parts = oracle.mla_decode_split_ref(
        inp["q_nope"], inp["q_pe"], inp["cache"], inp["block_table"], inp["seq_lens"], w.sm_scale,
        lambda b, i, nv: oracle.forced_split_ranges(nv, n), page_size=64)
    wsn = ws.cpu().numpy()
    slots_cap = (wsn.size - 32768) // (w.H * 513 * 4)
    # partial outputs are bf16, stored column-octet-major: [slot][64 octets][H][8]
    bits = wsn[32768:32768 + slots_cap * w.H * 512 * 2].view(np.uint16).reshape(slots_cap, 64, w.H, 8)
    po = oracle.decode_bf16(bits.transpose(0, 2, 1, 3).reshape(slots_cap, w.H, 512))
    pls = wsn[32768 + slots_cap * w.H * 512 * 4:][: slots_cap * w.H * 4].view(np.float32).reshape(slots_cap, w.H)
    for b in range(2):
        if pl["parts"][b] > 1:
            o_ref, l_ref = parts[(b, 0)]
            s0 = pl["slot"][b]
            got_o = po[s0:s0 + pl["parts"][b]].astype(np.float64)
            got_l = pls[s0:s0 + pl["parts"][b]].astype(np.float64)
            assert np.max(np.abs(got_l - l_ref)) < 1e-3
            assert np.max(np.abs(got_o - o_ref) - (1e-2 + 1e-2 * np.abs(o_ref))) <= 0


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8", "nvfp4"])
def test_poisoned_tails_and_unused_pages(kv_dtype):
    inp = _case("paged_bf16_ragged", B=4, H=64, kv_dtype=kv_dtype, seq_lens_override=(65, 1, 130, 191),
                extra_pages=3)
    W.poison_unused(inp)
    out, lse, status, _ = run_decode(inp)
    assert status == 0
    assert_close(out, lse, *oracle_ref(inp), what="poisoned")


def test_empty_and_short_sequences():
    inp = _case("paged_bf16_uniform", B=3, H=16, q_len=3, seq_lens_override=(0, 2, 70))
    out, lse, status, _ = run_decode(inp)
    assert status & 0x4  # seq_len < q_len reported
    ref = oracle_ref(inp)
    assert_close(out, lse, *ref, what="empty/short")


def test_device_status_bits_and_skipped_pages():
    inp = _case("paged_bf16_uniform", B=2, H=16, seq_lens_override=(200, 100))
    bad = inp["block_table"].copy()
    bad[0, 1] = inp["num_pages"] + 7  # out of range, the table itself is valid memory
    inp2 = dict(inp, block_table=bad)
    out, lse, status, _ = run_decode(inp2)
    assert status & 0x1
    # request 1 is untouched and still exact
    ref_out, ref_lse = oracle_ref(inp, rows=[(1, 0)])
    assert_close(out, lse, ref_out, ref_lse, rows=[(1, 0)], what="good row")
    # seq_len beyond the table's capacity: clamped and reported
    sl = inp["seq_lens"].copy()
    sl[1] = inp["block_table"].shape[1] * 64 + 5
    out, lse, status, _ = run_decode(dict(inp, seq_lens=sl))
    assert status & 0x2
    assert np.all(np.isfinite(out))


def test_repeat_calls_are_deterministic_and_need_no_zeroed_workspace():
    inp = _case("paged_bf16_ragged", B=5, seq_lens_override=(900, 17, 3000, 64, 5000))
    dev = to_device(inp)
    w = inp["workload"]
    ws = mb.alloc_workspace(w.B, w.q_len, w.H, 0)
    ws.fill_(0xAB)  # garbage
    o1, l1, s1, _ = run_decode(inp, dev, workspace=ws)
    o2, l2, s2, _ = run_decode(inp, dev, workspace=ws)
    assert s1 == 0 and s2 == 0
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    assert_close(o1, l1, *oracle_ref(inp), what="garbage workspace")


def test_workspace_size_and_too_small():
    C = mb.mla_decode_num_workers()
    assert C >= 1
    n = mb.mla_decode_workspace_size(32, 1, 128, 0)
    assert n == 32768 + 2 * C * 128 * 513 * 4
    assert mb.mla_decode_workspace_size(4, 2, 64, 3) == 32768 + 4 * 2 * 3 * 64 * 513 * 4
    inp = _case("paged_bf16_uniform", B=2, H=16, seq_len=100)
    dev = to_device(inp)
    ws = torch.empty(n // 1000, dtype=torch.uint8, device="cuda")
    with pytest.raises(mb.MLAError) as e:
        run_decode(inp, dev, workspace=ws)
    assert e.value.code == 3


def test_standalone_reduce_matches():
    inp = _case("paged_bf16_uniform", B=2, H=32, seq_lens_override=(640, 300))
    dev = to_device(inp)
    out, lse, status, ws = run_decode(inp, dev, num_splits=4)
    out2 = torch.zeros((2, 1, 32, 512), dtype=torch.bfloat16, device="cuda")
    lse2 = torch.zeros((2, 1, 32), dtype=torch.float32, device="cuda")
    mb.mla_splitk_reduce(ws, 2, 1, 32, out2, lse2)
    torch.cuda.synchronize()
    # every unit of this case is split, so the stand-alone reduce rewrites all of them
    assert np.array_equal(out2.float().cpu().double().numpy(), out)
    assert np.array_equal(lse2.cpu().double().numpy(), lse)


# ------------------------------------------------------------------ full-size workloads
FULL = ["paged_bf16_uniform", "paged_bf16_ragged", "paged_fp8", "paged_nvfp4_verify4"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_every_row(name):
    # Every (b, i) of the workload at its full size, in the bench's launch configuration
    # (the library's own schedule), against the oracle: the split boundaries between
    # workers and the combine of the split rows all fall somewhere in these rows.
    inp = W.make_inputs(W.WORKLOADS[name])
    out, lse, status, _ = run_decode(inp)
    assert status == 0
    ref_out, ref_lse = oracle_ref(inp)
    assert_close(out, lse, ref_out, ref_lse, what=name)
    assert np.all(np.isfinite(out)) and np.all(np.isfinite(lse))
