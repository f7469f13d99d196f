"""GPU parity of the CUDA-core decode kernel that small bf16 calls take (the tensor-core
kernel's pipeline set-up outlasts their whole work) against the float64 oracle: heads,
page sizes, ragged tails inside and across tiles, causal verify, the library's split
(one range per (b, i) here) and forced splits with their workspace partials (TileGym
mla_decoding_split_kv.py: partial outputs and log-sum-exps combined by splitk_reduce),
sliding windows and per-head sinks, poisoned unused cache rows, out-of-range pages and
empty requests.  Every case runs with the small-call limit raised so the CUDA-core kernel
takes it (every case fits in one wave of CTAs, as that path requires), and one case checks
from the workspace plan that it did."""
import numpy as np
import pytest

import oracle
from mla_latent_kv_split_gb300 import binding as mb
from mla_latent_kv_split_gb300 import workloads as W

from gpu_util import assert_close, ensure_built, oracle_ref, run_decode, small_call_limit

pytestmark = pytest.mark.gpu

BIG = 1 << 40  # every bf16 call within the CTA bound takes the CUDA-core kernel


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()


def _case(name, **kw):
    return W.make_inputs(W.WORKLOADS[name].scaled(**kw))


def _one_wave(ctas):
    """The CUDA-core path takes a call only when its CTAs fit in one wave."""
    if ctas > 2 * mb.mla_decode_num_workers():
        pytest.skip("the case needs more SMs than this device has")


def _plan(ws, U):
    """The workspace plan: {parts, first partial slot} per (b, i)."""
    w = ws.cpu().numpy()
    return w[256:256 + 8 * U].view(np.int32).reshape(U, 2)


def test_small_call_takes_the_cuda_core_kernel():
    inp = _case("paged_bf16_uniform", B=1, H=16, seq_len=1024)
    with small_call_limit(BIG):
        out, lse, status, ws = run_decode(inp, num_splits=0)
    assert status == 0
    assert_close(out, lse, *oracle_ref(inp), what="small, heuristic")
    # one range per (b, i): the tensor-core kernel's schedule would cut these 16 tiles
    # across many workers
    assert _plan(ws, 1)[0, 0] == 1
    with small_call_limit(0):
        out2, lse2, status2, ws2 = run_decode(inp, num_splits=0)
    assert status2 == 0 and _plan(ws2, 1)[0, 0] > 1
    assert_close(out2, lse2, *oracle_ref(inp), what="same call, tensor cores")


def test_default_limit_routes_the_tiny_workload():
    inp = W.make_inputs(W.WORKLOADS["tiny_contig_bf16"])
    with small_call_limit(mb.MLA_SMALL_CALL_DEFAULT):
        out, lse, status, ws = run_decode(inp)
    assert status == 0
    assert_close(out, lse, *oracle_ref(inp), what="tiny, default limit")


@pytest.mark.parametrize("H,lens", [(16, (97, 320, 1, 64)), (64, (97, 1)), (128, (320,))])
@pytest.mark.parametrize("ps", [32, 64])
def test_small_parity_heads_pages(H, lens, ps):
    _one_wave(len(lens) * H)
    inp = _case("paged_bf16_ragged", B=len(lens), H=H, page_size=ps, seq_lens_override=lens)
    with small_call_limit(BIG):
        out, lse, status, _ = run_decode(inp, num_splits=0)
    assert status == 0
    assert_close(out, lse, *oracle_ref(inp), what=f"small H{H} ps{ps}")


@pytest.mark.parametrize("q_len", [2, 4])
def test_small_causal_verify(q_len):
    _one_wave(2 * q_len * 16)
    inp = _case("paged_bf16_uniform", B=2, H=16, q_len=q_len, seq_lens_override=(130, 65))
    with small_call_limit(BIG):
        out, lse, status, _ = run_decode(inp, num_splits=0)
    assert status == 0
    assert_close(out, lse, *oracle_ref(inp), what=f"small q_len {q_len}")


@pytest.mark.parametrize("n", [1, 2, 3, 4])
def test_small_forced_splits_and_partials(n):
    _one_wave(2 * n * 16)
    inp = _case("paged_bf16_uniform", B=2, H=16, seq_lens_override=(450, 130))
    with small_call_limit(BIG):
        out, lse, status, ws = run_decode(inp, num_splits=n)
    assert status == 0
    assert_close(out, lse, *oracle_ref(inp), what=f"small splits={n}")
    w = inp["workload"]
    pl = mb.mla_decode_plan_host(inp["seq_lens"], 1, inp["block_table"].shape[1], 64, n, mb.mla_decode_num_workers())
    got_plan = _plan(ws, 2)
    assert np.array_equal(got_plan[:, 0], pl["parts"])
    _, _, parts = oracle.mla_decode_split_ref(
        inp["q_nope"], inp["q_pe"], inp["cache"], inp["block_table"], inp["seq_lens"], w.sm_scale,
        lambda b, i, nv: oracle.forced_split_ranges(nv, n), page_size=64)
    wsn = ws.cpu().numpy()
    slots_cap = (wsn.size - 32768) // (w.H * 513 * 4)
    bits = wsn[32768:32768 + slots_cap * w.H * 512 * 2].view(np.uint16).reshape(slots_cap, 64, w.H, 8)
    po = oracle.decode_bf16(bits.transpose(0, 2, 1, 3).reshape(slots_cap, w.H, 512))
    pls = wsn[32768 + slots_cap * w.H * 512 * 4:][: slots_cap * w.H * 4].view(np.float32).reshape(slots_cap, w.H)
    for b in range(2):
        if pl["parts"][b] > 1:
            assert got_plan[b, 1] == pl["slot"][b]
            o_ref, l_ref = parts[(b, 0)]
            s0 = pl["slot"][b]
            got_o = po[s0:s0 + pl["parts"][b]].astype(np.float64)
            got_l = pls[s0:s0 + pl["parts"][b]].astype(np.float64)
            assert np.max(np.abs(got_l - l_ref)) < 1e-3
            assert np.max(np.abs(got_o - o_ref) - (1e-2 + 1e-2 * np.abs(o_ref))) <= 0


LENS = {0: (0, 1, 63, 64, 65, 700, 129), 3: (0, 65, 700)}


@pytest.mark.parametrize("num_splits", [0, 3])
@pytest.mark.parametrize("window", [1, 64, 65, 640])
def test_small_window_and_sinks(window, num_splits):
    lens = LENS[num_splits]
    _one_wave(len(lens) * max(num_splits, 1) * 16)
    w = W.WORKLOADS["paged_bf16_ragged"].scaled(B=len(lens), H=16, seq_lens_override=lens)
    inp = W.make_inputs(w)
    sinks = W.draw_sinks(16, seed=window)
    sinks[3] = -np.inf
    with small_call_limit(BIG):
        out, lse, status, _ = run_decode(inp, num_splits=num_splits, window=window, sinks=sinks)
    assert status == 0x4  # the seq_len 0 request is reported (shorter than q_len)
    assert_close(out, lse, *oracle_ref(inp, window=window, sinks=sinks), what=f"small W{window} n{num_splits}")


def test_small_poisoned_tails_bad_pages_and_empty_requests():
    inp = _case("paged_bf16_ragged", B=4, H=32, seq_lens_override=(65, 1, 130, 191), extra_pages=3)
    W.poison_unused(inp)
    with small_call_limit(BIG):
        out, lse, status, _ = run_decode(inp, num_splits=0)
    assert status == 0
    assert_close(out, lse, *oracle_ref(inp), what="small poisoned")
    # an out-of-range page: reported, and the other requests stay exact
    inp = _case("paged_bf16_uniform", B=2, H=16, seq_lens_override=(200, 100))
    bad = inp["block_table"].copy()
    bad[0, 1] = inp["num_pages"] + 7
    with small_call_limit(BIG):
        out, lse, status, _ = run_decode(dict(inp, block_table=bad), num_splits=2)
    assert status & 0x1
    ref_out, ref_lse = oracle_ref(inp, rows=[(1, 0)])
    assert_close(out, lse, ref_out, ref_lse, rows=[(1, 0)], what="small good row")
    # empty and shorter-than-q_len requests
    inp = _case("paged_bf16_uniform", B=3, H=16, q_len=3, seq_lens_override=(0, 2, 70))
    with small_call_limit(BIG):
        out, lse, status, _ = run_decode(inp, num_splits=0)
    assert status & 0x4
    assert_close(out, lse, *oracle_ref(inp), what="small empty/short")


def test_small_call_captured_in_a_graph():
    """The CUDA-core decode and the combine inside a CUDA graph: replays equal an eager call
    bit for bit, also after the queries and sequence lengths change in place."""
    import torch
    from gpu_util import to_device
    w = W.WORKLOADS["paged_bf16_ragged"].scaled(B=4, H=16, seq_lens_override=(100, 250, 7, 64))
    inp = W.make_inputs(w)
    dev = to_device(inp)
    ws = mb.alloc_workspace(w.B, w.q_len, w.H, 2)

    def call(out=None, lse=None, stream=None):
        return mb.mla_decode(dev["q_nope"], dev["q_pe"], dev["cache"], dev["block_table"], dev["seq_lens"],
                             w.sm_scale, w.kv_dtype, inp["kv_scale"], 2, page_size=w.page_size,
                             num_pages=inp["num_pages"], workspace=ws, out=out, lse=lse, stream=stream)

    with small_call_limit(BIG):
        ref_out, ref_lse = call()
        torch.cuda.synchronize()
        ref_out, ref_lse = ref_out.clone(), ref_lse.clone()
        assert _plan(ws, 4)[1, 0] == 2  # forced splits: the partials and the combine are used
        out, lse = torch.empty_like(ref_out), torch.empty_like(ref_lse)
        graph = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            with torch.cuda.graph(graph, stream=side):
                call(out, lse, side)
        torch.cuda.current_stream().wait_stream(side)
        for _ in range(3):
            out.fill_(float("nan"))
            lse.fill_(float("nan"))
            graph.replay()
            torch.cuda.synchronize()
            assert mb.mla_decode_read_status(ws) == 0
            assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))
            assert torch.equal(lse.view(torch.int32), ref_lse.view(torch.int32))
        g = torch.Generator().manual_seed(7)
        dev["q_nope"].copy_(torch.randn(dev["q_nope"].shape, generator=g).to(torch.bfloat16))
        new_lens = np.array([60, 200, 3, 64], dtype=np.int32)
        dev["seq_lens"].copy_(torch.from_numpy(new_lens))
        graph.replay()
        torch.cuda.synchronize()
        ref2_out, ref2_lse = call()
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), ref2_out.view(torch.int16))
        assert torch.equal(lse.view(torch.int32), ref2_lse.view(torch.int32))
    inp2 = dict(inp)
    inp2["q_nope"] = dev["q_nope"].cpu().view(torch.int16).numpy().view(np.uint16)
    inp2["seq_lens"] = new_lens
    assert_close(out.float().cpu().double().numpy(), lse.cpu().double().numpy(), *oracle_ref(inp2),
                 what="small call, graph replay")
