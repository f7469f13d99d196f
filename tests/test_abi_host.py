"""CPU-side checks of the C ABI: the library loads and exports every declared symbol, host
validation rejects bad arguments before touching the GPU, and the split schedule the
kernels evaluate (mirrored on the host) covers every KV tile exactly once."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
from mla_latent_kv_split_gb300 import binding as mb

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ITEM_COST = 4  # placeholder slots per work item in the library's balanced split


@pytest.fixture(scope="module")
def L():
    if not os.path.exists(mb.LIB_PATH):
        from mla_latent_kv_split_gb300 import build
        build.build()
    return mb.lib()


def _declared_functions():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", fn)).read()
            txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(mla_[a-z0-9_]+)\s*\(", txt, flags=re.M)
    return sorted(set(names))


def test_library_exports_every_declared_symbol(L):
    declared = _declared_functions()
    assert len(declared) >= 8, declared
    for name in declared:
        assert hasattr(L, name), name
    assert set(mb.EXPORTED) <= set(declared)
    assert L.mla_decode_abi_version() == 3
    for code in range(6):
        assert L.mla_status_string(code).decode().startswith("MLA_")


def _call(L, **over):
    a = dict(q_nope=16, q_pe=16, kv=128, bt=16, max_pages=4, sl=16, B=1, q_len=1, H=16, num_pages=4,
             page_size=64, sm_scale=0.1, kv_dtype=0, kv_scale=1.0, num_splits=0, ws=256, ws_bytes=1 << 30,
             out=16, lse=16, stream=None)
    a.update(over)
    return L.mla_decode(a["q_nope"], a["q_pe"], a["kv"], a["bt"], a["max_pages"], a["sl"], a["B"], a["q_len"],
                        a["H"], a["num_pages"], a["page_size"], a["sm_scale"], a["kv_dtype"], a["kv_scale"],
                        a["num_splits"], a["ws"], a["ws_bytes"], a["out"], a["lse"], a["stream"])


@pytest.mark.parametrize("over,code", [
    (dict(H=24), 2), (dict(H=0), 1), (dict(H=256), 2), (dict(page_size=16), 2), (dict(page_size=128), 2),
    (dict(q_len=0), 1), (dict(q_len=9), 2), (dict(B=-1), 1), (dict(B=1025), 2), (dict(kv_dtype=7), 1),
    (dict(sm_scale=float("nan")), 1), (dict(kv_dtype=1, kv_scale=0.0), 1), (dict(kv_dtype=1, kv_scale=float("inf")), 1),
    (dict(num_splits=-1), 1), (dict(max_pages=0), 1), (dict(num_pages=0), 1),
    (dict(q_nope=None), 1), (dict(kv=None), 1), (dict(ws=None), 1), (dict(out=None), 1),
    (dict(q_nope=18), 1), (dict(kv=144), 1), (dict(ws=128), 1), (dict(max_pages=1 << 30), 2),
])
def test_host_validation_rejects_before_launch(L, over, code):
    assert _call(L, **over) == code


def test_empty_batch_is_a_noop(L):
    assert _call(L, B=0, q_nope=None, q_pe=None, kv=None, bt=None, sl=None, ws=None, out=None, lse=None) == 0


def _check_plan(seq_lens, q_len, ps, num_splits, C, max_pages=None, window=0):
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    if max_pages is None:
        max_pages = max(1, int(-(-max(int(seq_lens.max()), 1) // ps)))
    pl = mb.mla_decode_plan_host(seq_lens, q_len, max_pages, ps, num_splits, C, window=window)
    U = len(seq_lens) * q_len
    vis = np.array([oracle.visible_len(min(max(int(seq_lens[u // q_len]), 0), max_pages * ps), q_len, u % q_len)
                    for u in range(U)])
    # 64-token tiles from the one holding the window's first position to the last visible one
    first = np.array([oracle.window_range(int(v), window)[0] for v in vis])
    tiles = np.where(vis > 0, -(-vis // 64) - first // 64, 0)
    assert np.array_equal(pl["tiles"], tiles)
    # schedule order: query-major for a verify batch in the heuristic mode (position
    # k = i * B + b holds unit (b, i)), else the unit order
    B = len(seq_lens)
    order = [(k % B) * q_len + k // B for k in range(U)] if (q_len > 1 and num_splits == 0) else list(range(U))
    assert sorted(order) == list(range(U))
    # slots: contiguous, disjoint, only for split units, in schedule order
    used = 0
    for u in order:
        if pl["parts"][u] > 1:
            assert pl["slot"][u] == used
            used += pl["parts"][u]
        else:
            assert pl["slot"][u] == -1
        assert pl["parts"][u] == 0 if tiles[u] == 0 else pl["parts"][u] >= 1
    assert used == pl["slots_used"]
    if num_splits > 0:
        for u in range(U):
            if tiles[u] and window == 0:
                assert pl["parts"][u] == len(oracle.forced_split_ranges(int(vis[u]), num_splits))
            elif tiles[u]:  # ranges of cdiv(tiles, num_splits) tiles: never more than num_splits
                span = -(-int(tiles[u]) // num_splits)
                assert pl["parts"][u] == -(-int(tiles[u]) // span) <= num_splits
    else:
        assert used <= 2 * C
        # brute force: every unit with tiles is ITEM_COST placeholder slots then its tiles;
        # the slots are dealt to workers by the balanced rule and a unit's parts are the
        # workers holding any of its tiles
        slots_u = np.where(tiles > 0, tiles + ITEM_COST, 0)
        N = int(slots_u.sum())
        Ca = min(C, N)
        owner = np.empty(N, dtype=np.int64)
        for c in range(Ca):
            owner[c * N // Ca:(c + 1) * N // Ca] = c
        t0 = 0
        for u in order:
            if tiles[u]:
                assert pl["tile_begin"][u] == t0
                real = owner[t0 + ITEM_COST:t0 + ITEM_COST + tiles[u]]
                assert pl["parts"][u] == len(set(real.tolist()))
            t0 += slots_u[u]
        # balance: every active worker gets floor or ceil of N / Ca slots
        if N:
            counts = np.bincount(owner, minlength=Ca)
            assert counts.max() - counts.min() <= 1
    return pl


@pytest.mark.parametrize("C", [1, 2, 5, 76, 300])
def test_plan_heuristic_covers_and_balances(L, C):
    rng = np.random.default_rng(C)
    for trial in range(5):
        B = int(rng.integers(1, 40))
        q_len = int(rng.integers(1, 5))
        seq = rng.integers(0, 5000, size=B)
        _check_plan(seq, q_len, 64, 0, C)


@pytest.mark.parametrize("C", [76, 74, 64, 7])
def test_plan_on_the_full_size_workloads(L, C):
    """The schedule of every workload at its full size (the request lengths the bench and the
    full-size parity tests use, drawn without the caches), checked by brute force with the
    GB300's 76 workers and other worker counts (coverage, balance, contiguous partial slots,
    at most 2C of them: the bound the heuristic-mode workspace is sized for)."""
    import torch
    from mla_latent_kv_split_gb300 import workloads as W
    for w in W.WORKLOADS.values():
        seq = W.draw_seq_lens(w, torch.Generator().manual_seed(w.seed))
        _check_plan(seq, w.q_len, w.page_size, w.num_splits, C)


@pytest.mark.parametrize("n", [1, 2, 3, 7])
def test_plan_forced_splits(L, n):
    _check_plan([256, 1, 0, 700, 64, 65], 1, 64, n, 76)
    _check_plan([256, 9, 300], 4, 32, n, 3)


def test_plan_tiny_contiguous_two_splits(L):
    pl = _check_plan([256], 1, 64, 2, 76)
    assert pl["parts"][0] == 2 and pl["slots_used"] == 2


def test_plan_clamps_and_negative_lengths(L):
    pl = _check_plan([-5, 10 ** 6, 3], 2, 64, 0, 4, max_pages=2)
    assert pl["tiles"][0] == 0 and pl["tiles"][1] == 0  # seq_len -5 -> nothing visible
    assert pl["tiles"][2] == 2 and pl["tiles"][3] == 2  # clamped to 128: 127 and 128 visible


@pytest.mark.parametrize("window", [1, 63, 64, 65, 200, 5000])
@pytest.mark.parametrize("num_splits", [0, 2, 3])
def test_plan_with_sliding_window(L, window, num_splits):
    rng = np.random.default_rng(window + num_splits)
    for trial in range(4):
        B = int(rng.integers(1, 20))
        q_len = int(rng.integers(1, 4))
        seq = rng.integers(0, 3000, size=B)
        _check_plan(seq, q_len, 64 if trial % 2 else 32, num_splits, int(rng.integers(1, 80)), window=window)


def test_window_and_sink_arguments_validated(L):
    args = [16, 16, 128, 16, 4, 16, 1, 1, 16, 4, 64, 0.1, 0, 1.0, 0]
    assert L.mla_decode_ex(*args, -1, None, 256, 1 << 30, 16, 16, None) == 1  # negative window
    assert L.mla_decode_ex(*args, 0, 18, 256, 1 << 30, 16, 16, None) == 1  # misaligned sinks
    assert L.mla_decode_ex(*args[:6], 0, *args[7:], 5, None, None, 0, None, None, None) == 0  # B = 0
    i32 = ctypes.POINTER(ctypes.c_int32)
    z = (ctypes.c_int32 * 1)()
    sl = (ctypes.c_int32 * 1)(10)
    assert L.mla_decode_plan_host(sl, 1, 1, 1, 64, 0, -3, 4, z, z, z, z, z) == 1


def test_kv_append_arguments_validated(L):
    P = 1 << 20  # any 128-byte aligned non-null value: nothing is launched on these paths
    ok = dict(lat=P, ls=576, rope=P + 1024, rs=576, slots=P, T=4, cache=P, num_pages=2, ps=64, kd=0, scale=1.0,
              status=None)

    def call(**over):
        a = dict(ok)
        a.update(over)
        return L.mla_kv_append(a["lat"], a["ls"], a["rope"], a["rs"], a["slots"], a["T"], a["cache"], a["num_pages"],
                               a["ps"], a["kd"], a["scale"], a["status"], None)

    for over, code in [(dict(T=-1), 1), (dict(num_pages=0), 1), (dict(ps=16), 2), (dict(kd=5), 1),
                       (dict(kd=1, scale=0.0), 1), (dict(kd=1, scale=float("nan")), 1), (dict(lat=None), 1),
                       (dict(slots=None), 1), (dict(ls=511), 1), (dict(rs=60), 1), (dict(ls=580), 1),
                       (dict(lat=P + 2), 1), (dict(rope=P + 8), 1), (dict(slots=P + 4), 1), (dict(cache=P + 64), 1),
                       (dict(status=P + 2), 1)]:
        assert call(**over) == code, over
    assert call(T=0, lat=None, rope=None, slots=None, cache=None) == 0


def test_batched_gemv_arguments_validated(L):
    P = 1 << 20
    ok = dict(x=P, xt=128 * 192, xh=192, w=P, out=P, ot=128 * 512, oh=512, T=4, H=128, N=512, K=128, status=None)

    def call(**over):
        a = dict(ok)
        a.update(over)
        return L.mla_batched_gemv(a["x"], a["xt"], a["xh"], a["w"], a["out"], a["ot"], a["oh"], a["T"], a["H"],
                                  a["N"], a["K"], a["status"], None)

    for over, code in [(dict(T=-1), 1), (dict(H=0), 1), (dict(N=0), 1), (dict(K=4), 1), (dict(K=100), 1),
                       (dict(x=None), 1), (dict(w=None), 1), (dict(out=None), 1), (dict(x=P + 8), 1),
                       (dict(w=P + 2), 1), (dict(out=P + 4), 1), (dict(xh=120), 1), (dict(xh=196), 1),
                       (dict(xt=100), 1), (dict(oh=500), 1), (dict(H=70000), 2), (dict(status=P + 1), 1)]:
        assert call(**over) == code, over
    assert call(T=0, x=None, w=None, out=None) == 0


def test_binding_shape_checks_raise_before_the_library_is_called(L):
    import torch
    x = torch.empty((4, 2, 128), dtype=torch.bfloat16)
    w = torch.empty((2, 64, 96), dtype=torch.bfloat16)  # K mismatch
    with pytest.raises(ValueError):
        mb.mla_batched_gemv(x, w, out=torch.empty((4, 2, 64), dtype=torch.bfloat16))
    w = torch.empty((2, 64, 128), dtype=torch.bfloat16)
    with pytest.raises(ValueError):  # out not [T, H, N]
        mb.mla_batched_gemv(x, w, out=torch.empty((4, 2, 65), dtype=torch.bfloat16))
    tok = torch.empty((3, 576), dtype=torch.bfloat16)
    with pytest.raises(ValueError):  # rope view of the wrong width
        mb.mla_kv_append(tok[:, :512], tok[:, 500:], torch.zeros(3, dtype=torch.int64),
                         torch.empty((1, 64, 576), dtype=torch.bfloat16))
    with pytest.raises(ValueError):  # slots and rows disagree
        mb.mla_kv_append(tok[:, :512], tok[:, 512:], torch.zeros(2, dtype=torch.int64),
                         torch.empty((1, 64, 576), dtype=torch.bfloat16))


def test_binding_reports_library_errors_with_their_code(L):
    # T > 0 with a null cache is rejected by the library's validation: MLAError(code 1)
    import torch
    tok = torch.empty((3, 576), dtype=torch.bfloat16)
    with pytest.raises(mb.MLAError) as e:
        mb.mla_kv_append(tok[:, :512], tok[:, 512:], torch.zeros(3, dtype=torch.int64), 0,
                         page_size=64, num_pages=1, stream=0)
    assert e.value.code == 1


@pytest.mark.parametrize("B,q_len,H,n", [(32, 1, 128, 5), (1, 1, 16, 2), (8, 4, 128, 3), (4, 2, 64, 3),
                                         (1024, 1, 128, 1), (2, 8, 16, 4096)])
def test_forced_workspace_size_is_header_plus_tokenspeed_formula(L, B, q_len, H, n):
    # forced splits: at most n partials per (b, i), each H*(512+1) fp32 values -- the
    # tokenspeed decode workspace formula -- after the 32 KB plan / status header
    assert mb.mla_decode_workspace_size(B, q_len, H, n) == 32768 + oracle.workspace_bytes_formula(B, H, q_len, n)


def test_verify_batch_schedule_aligns_the_queries_of_a_request(L):
    # The NVFP4 verify workload's shape: 8 requests x 4 queries of 131,072 positions on 76
    # workers.  In query-major order the workers serving query i of a request cover the same
    # tiles as those serving query 0, 19 workers further on, so that a page read for one
    # query is still in L2 when the others read it.
    B, q_len, C, S = 8, 4, 76, 131072
    seq = np.full(B, S, dtype=np.int32)
    pl = _check_plan(seq, q_len, 64, 0, C)
    tiles = pl["tiles"]
    slots = np.where(tiles > 0, tiles + ITEM_COST, 0)
    order = [(k % B) * q_len + k // B for k in range(B * q_len)]
    N = int(slots.sum())
    ranges = {}
    for c in range(C):
        lo, hi = c * N // C, (c + 1) * N // C
        for u in order:
            r0 = pl["tile_begin"][u] + ITEM_COST
            a, b = max(lo, r0), min(hi, r0 + tiles[u])
            if a < b:
                ranges.setdefault(c, []).append((u // q_len, u % q_len, a - r0, b - r0))
    per = C // q_len
    for c in range(per):
        for i in range(1, q_len):
            mine, theirs = ranges[c], ranges[c + i * per]
            assert len(mine) == len(theirs)
            for (b0, i0, a0, e0), (b1, i1, a1, e1) in zip(mine, theirs):
                assert b0 == b1 and i0 == 0 and i1 == i
                assert abs(a0 - a1) <= 1 and abs(e0 - e1) <= 1


def test_small_call_limit_setter_and_default():
    """The small-call limit is a plain value: the setter returns the previous one, and the
    binding's default mirrors the header's."""
    import re
    hdr = open(os.path.join(ROOT, "include", "mla_decode.h")).read()
    m = re.search(r"#define MLA_SMALL_CALL_DEFAULT (\d+)u", hdr)
    assert m and int(m.group(1)) == mb.MLA_SMALL_CALL_DEFAULT
    old = mb.mla_decode_set_small_call_limit(123)
    try:
        assert mb.mla_decode_set_small_call_limit(456) == 123
    finally:
        assert mb.mla_decode_set_small_call_limit(old) == 456
