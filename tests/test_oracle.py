"""Pins for the float64 oracle, against things other than itself: OCP spec tables, torch's
own fp8/bf16 conversions, torch's scaled_dot_product_attention in float64, pure-Python
brute force on tiny inputs, closed forms and invariants of softmax attention."""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import mla_ref
from mla_latent_kv_split_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    rows = []
    for line in open(os.path.join(GOLDEN, name)):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        c, v = line.split()
        rows.append((int(c, 0), float(v)))
    return rows


# ---------------------------------------------------------------------- number formats

def test_e4m3_table_matches_torch_for_every_code():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = oracle.decode_e4m3(np.arange(256, dtype=np.uint8))
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(ref[~nan], got[~nan])
    assert np.array_equal(np.signbit(ref[~nan]), np.signbit(got[~nan]))


def test_e4m3_spec_values():
    for code, val in _golden("ocp_e4m3_specials.txt"):
        got = oracle.decode_e4m3(np.array([code], dtype=np.uint8))[0]
        if math.isnan(val):
            assert math.isnan(got)
        else:
            assert got == val and math.copysign(1, got) == math.copysign(1, val), hex(code)


def test_e2m1_table_matches_ocp_mx_spec():
    for code, val in _golden("ocp_e2m1_values.txt"):
        got = oracle.decode_e2m1(np.array([code], dtype=np.uint8))[0]
        assert got == val and math.copysign(1, got) == math.copysign(1, val), code


def test_e2m1_values_are_a_subset_of_e4m3_codes():
    # every E2M1 value is exactly an E4M3 value; torch's RNE cast must reproduce it
    vals = torch.tensor(oracle.E2M1_TABLE, dtype=torch.float32)
    back = vals.to(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(back, oracle.E2M1_TABLE)


def test_bf16_decode_matches_torch():
    rng = np.random.default_rng(0)
    bits = rng.integers(0, 1 << 16, size=4096, dtype=np.uint16)
    bits = bits[(bits & 0x7F80) != 0x7F80]  # finite patterns only
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(oracle.decode_bf16(bits), ref)


def test_fp8_cache_decode_matches_torch_times_scale():
    x = torch.randn(3, 64, 576, generator=torch.Generator().manual_seed(3)) * 50
    codes = W.quantize_e4m3_rne(x)
    scale = 0.0371
    got = oracle.dequant_pages(codes, "fp8", 64, scale, np.arange(3))
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy() * np.float64(np.float32(scale))
    assert np.array_equal(got, ref)


def test_nvfp4_page_layout_hand_built():
    # Build one 2-token page by hand from the documented layout and check every element.
    ps = 2
    nb = oracle.nvfp4_page_bytes(ps)
    assert nb == ps * 288 + ps * 36
    page = np.zeros((1, nb), dtype=np.uint8)
    rng = np.random.default_rng(7)
    codes = rng.integers(0, 16, size=(ps, 576), dtype=np.uint8)
    # E4M3 scale codes: 0x38 = 1.0, 0x40 = 2.0, 0x30 = 0.5 ; pick per group
    scode = rng.choice(np.array([0x38, 0x40, 0x30, 0x3C], dtype=np.uint8), size=(ps, 36))
    sval = {0x38: 1.0, 0x40: 2.0, 0x30: 0.5, 0x3C: 1.5}
    e2m1 = {c: v for c, v in _golden("ocp_e2m1_values.txt")}
    for t in range(ps):
        for j in range(288):
            page[0, t * 288 + j] = int(codes[t, 2 * j]) | (int(codes[t, 2 * j + 1]) << 4)
        for gi in range(36):
            page[0, ps * 288 + t * 36 + gi] = scode[t, gi]
    got = oracle.dequant_pages(page, "nvfp4", ps, 1.0, np.array([0]))[0]
    for t in range(ps):
        for e in range(576):
            assert got[t, e] == e2m1[int(codes[t, e])] * sval[int(scode[t, e // 16])]


def test_nvfp4_quantiser_roundtrip_half_step():
    x = torch.randn(4, 64, 576, generator=torch.Generator().manual_seed(5))
    pages = W.quantize_nvfp4_pages(x)
    deq = oracle.dequant_pages(pages, "nvfp4", 64, 1.0, np.arange(4))
    xs = x.double().numpy().reshape(4, 64, 36, 16)
    amax = np.abs(xs).max(-1, keepdims=True)
    s = torch.from_numpy((amax / 6.0).astype(np.float32)).to(torch.float8_e4m3fn).double().numpy()
    err = np.abs(deq.reshape(xs.shape) - xs)
    # within half of the widest E2M1 step (2.0 between 4 and 6) times the block scale,
    # plus the clamp at 6*s when the scale rounded down
    bound = s * 1.0 + np.maximum(0, amax - 6 * s) + 1e-12
    assert np.all(err <= bound)
    # values exactly on the grid come back exactly
    grid = torch.tensor([0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -6.0, -0.5, 0.0, 3.0, -1.5, 2.0, 4.0, 1.0, 6.0])
    xg = (grid * 0.25).repeat(36).reshape(1, 1, 576)
    back = oracle.dequant_pages(W.quantize_nvfp4_pages(xg), "nvfp4", 1, 1.0, np.array([0]))
    assert np.array_equal(back.reshape(-1), xg.double().numpy().reshape(-1))


# ---------------------------------------------------------------------- the decode

def _rand_bits(shape, seed):
    return W._bf16_bits(torch.randn(shape, generator=torch.Generator().manual_seed(seed)))


def _contig_case(H=4, n=10, seed=0):
    qn = _rand_bits((1, 1, H, 512), seed)
    qp = _rand_bits((1, 1, H, 64), seed + 1)
    cache = _rand_bits((1, max(n, 1), 576), seed + 2)  # one page of n tokens
    return qn, qp, cache


def test_decode_matches_torch_sdpa_float64():
    H, n = 6, 37
    qn, qp, cache = _contig_case(H, n, seed=11)
    scale = 1 / math.sqrt(192)
    out, lse = oracle.mla_decode_ref(qn, qp, cache, np.array([[0]]), np.array([n]), scale, page_size=n)
    q = torch.from_numpy(np.concatenate([oracle.decode_bf16(qn[0, 0]), oracle.decode_bf16(qp[0, 0])], -1))
    k = torch.from_numpy(oracle.decode_bf16(cache[0]))
    ref = torch.nn.functional.scaled_dot_product_attention(
        q[None, :, None, :], k[None, None].expand(1, H, n, 576), k[None, None, :, :512].expand(1, H, n, 512),
        scale=scale)[0, :, 0]
    assert np.max(np.abs(out[0, 0] - ref.numpy())) < 1e-12
    lse_ref = torch.logsumexp(scale * (q @ k.T), dim=-1).numpy()
    assert np.max(np.abs(lse[0, 0] - lse_ref)) < 1e-12


def test_decode_matches_pure_python_brute_force():
    H, n = 3, 5
    qn, qp, cache = _contig_case(H, n, seed=21)
    scale = 0.3
    out, lse = oracle.mla_decode_ref(qn, qp, cache, np.array([[0]]), np.array([n]), scale, page_size=n)
    qf = [[float(v) for v in oracle.decode_bf16(qn[0, 0, h])] + [float(v) for v in oracle.decode_bf16(qp[0, 0, h])]
          for h in range(H)]
    kf = [[float(v) for v in oracle.decode_bf16(cache[0, t])] for t in range(n)]
    for h in range(H):
        xs = [scale * math.fsum(qf[h][c] * kf[t][c] for c in range(576)) for t in range(n)]
        m = max(xs)
        z = math.fsum(math.exp(x - m) for x in xs)
        assert abs(lse[0, 0, h] - (m + math.log(z))) < 1e-12
        for c in range(0, 512, 37):
            o = math.fsum(math.exp(xs[t] - m) / z * kf[t][c] for t in range(n))
            assert abs(out[0, 0, h, c] - o) < 1e-12


def test_single_token_kv_returns_that_row():
    qn, qp, cache = _contig_case(5, 1, seed=31)
    out, lse = oracle.mla_decode_ref(qn, qp, cache, np.array([[0]]), np.array([1]), 0.07, page_size=1)
    row = oracle.decode_bf16(cache[0, 0])
    assert np.array_equal(out[0, 0], np.broadcast_to(row[:512], (5, 512)))
    q = np.concatenate([oracle.decode_bf16(qn[0, 0]), oracle.decode_bf16(qp[0, 0])], -1)
    assert np.allclose(lse[0, 0], 0.07 * (q @ row), rtol=0, atol=1e-12)


def test_equal_scores_give_mean_of_v():
    # q_nope = 0 and identical k_pe for every token -> every score equal
    H, n = 4, 23
    qn = np.zeros((1, 1, H, 512), dtype=np.uint16)
    qp = _rand_bits((1, 1, H, 64), 41)
    cache = _rand_bits((1, n, 576), 42)
    cache[0, :, 512:] = cache[0, 0, 512:]
    out, lse = oracle.mla_decode_ref(qn, qp, cache, np.array([[0]]), np.array([n]), 0.1, page_size=n)
    v = oracle.decode_bf16(cache[0, :, :512])
    assert np.max(np.abs(out[0, 0] - v.mean(0)[None])) < 1e-12
    x = 0.1 * (oracle.decode_bf16(qp[0, 0]) @ oracle.decode_bf16(cache[0, 0, 512:]))
    assert np.max(np.abs(lse[0, 0] - (x + math.log(n)))) < 1e-12


def test_one_hot_score_selects_row():
    H, n = 2, 9
    qn, qp, cache = _contig_case(H, n, seed=51)
    k = oracle.decode_bf16(cache[0])
    # make the query a huge multiple of token 4's key -> softmax is one-hot on token 4
    qn = W._bf16_bits(torch.from_numpy(np.tile(k[4, :512] * 40, (1, 1, H, 1)).astype(np.float32)))
    qp = W._bf16_bits(torch.from_numpy(np.tile(k[4, 512:] * 40, (1, 1, H, 1)).astype(np.float32)))
    out, _ = oracle.mla_decode_ref(qn, qp, cache, np.array([[0]]), np.array([n]), 1.0, page_size=n)
    assert np.max(np.abs(out[0, 0] - k[4, :512][None])) < 1e-9


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8", "nvfp4"])
def test_split_count_invariance(kv_dtype):
    w = W.WORKLOADS["paged_bf16_uniform"].scaled(B=2, H=8, seq_lens_override=(300, 77), kv_dtype=kv_dtype)
    inp = W.make_inputs(w)
    args = (inp["q_nope"], inp["q_pe"], inp["cache"], inp["block_table"], inp["seq_lens"], w.sm_scale)
    kw = dict(kv_dtype=kv_dtype, kv_scale=inp["kv_scale"], page_size=64)
    ref_out, ref_lse = oracle.mla_decode_ref(*args, **kw)
    for n in (1, 2, 3, 5):
        out, lse, parts = oracle.mla_decode_split_ref(
            *args, lambda b, i, nv: oracle.forced_split_ranges(nv, n), **kw)
        assert np.max(np.abs(out - ref_out)) < 1e-12
        assert np.max(np.abs(lse - ref_lse)) < 1e-12
    # ragged, uneven hand-picked splits including an empty one
    out, lse, _ = oracle.mla_decode_split_ref(
        *args, lambda b, i, nv: [(0, 13), (13, 13), (13, 200), (200, 10**6)], **kw)
    assert np.max(np.abs(out - ref_out)) < 1e-12 and np.max(np.abs(lse - ref_lse)) < 1e-12


def test_combine_all_empty():
    out, lse = oracle.combine_ref(np.zeros((3, 2, 512)), np.full((3, 2), -np.inf))
    assert np.all(out == 0) and np.all(np.isneginf(lse))


def test_page_permutation_and_head_permutation_invariance():
    w = W.WORKLOADS["paged_bf16_uniform"].scaled(B=2, H=8, seq_lens_override=(200, 129))
    inp = W.make_inputs(w)
    args = dict(sm_scale=w.sm_scale, page_size=64)
    out, lse = oracle.mla_decode_ref(inp["q_nope"], inp["q_pe"], inp["cache"], inp["block_table"], inp["seq_lens"], **args)
    # move every page to a new physical slot
    P = inp["cache"].shape[0]
    perm = np.random.default_rng(0).permutation(P)
    cache2 = np.empty_like(inp["cache"])
    cache2[perm] = inp["cache"]
    table2 = perm[inp["block_table"]].astype(np.int32)
    out2, lse2 = oracle.mla_decode_ref(inp["q_nope"], inp["q_pe"], cache2, table2, inp["seq_lens"], **args)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)
    hp = np.random.default_rng(1).permutation(8)
    out3, lse3 = oracle.mla_decode_ref(inp["q_nope"][:, :, hp], inp["q_pe"][:, :, hp], inp["cache"],
                                       inp["block_table"], inp["seq_lens"], **args)
    assert np.max(np.abs(out3 - out[:, :, hp])) < 1e-12 and np.max(np.abs(lse3 - lse[:, :, hp])) < 1e-12


def test_causal_verify_equals_separate_decodes_and_sdpa_mask():
    q_len = 4
    w = W.WORKLOADS["paged_nvfp4_verify4"].scaled(B=2, H=4, seq_lens_override=(70, 5), kv_dtype="bf16")
    inp = W.make_inputs(w)
    out, lse = oracle.mla_decode_ref(inp["q_nope"], inp["q_pe"], inp["cache"], inp["block_table"],
                                     inp["seq_lens"], w.sm_scale, page_size=64)
    for b in range(2):
        L = int(inp["seq_lens"][b])
        for i in range(q_len):
            o1, l1 = oracle.mla_decode_ref(inp["q_nope"][b:b + 1, i:i + 1], inp["q_pe"][b:b + 1, i:i + 1],
                                           inp["cache"], inp["block_table"][b:b + 1],
                                           np.array([L - q_len + 1 + i]), w.sm_scale, page_size=64)
            assert np.max(np.abs(o1[0, 0] - out[b, i])) < 1e-12 and np.max(np.abs(l1[0, 0] - lse[b, i])) < 1e-12
        # the same via torch SDPA with an explicit boolean mask
        keys = torch.from_numpy(oracle.gather_tokens(inp["cache"], inp["block_table"][b], L, "bf16", 64))
        q = torch.from_numpy(np.concatenate([oracle.decode_bf16(inp["q_nope"][b]), oracle.decode_bf16(inp["q_pe"][b])], -1))
        mask = torch.arange(L)[None, :] <= (L - q_len + torch.arange(q_len))[:, None]
        ref = torch.nn.functional.scaled_dot_product_attention(
            q.permute(1, 0, 2), keys[None].expand(4, L, 576), keys[None, :, :512].expand(4, L, 512),
            attn_mask=mask[None].expand(4, q_len, L), scale=w.sm_scale).permute(1, 0, 2)
        assert np.max(np.abs(ref.numpy() - out[b])) < 1e-12


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8", "nvfp4"])
def test_poisoned_tails_do_not_change_output(kv_dtype):
    w = W.WORKLOADS["paged_bf16_uniform"].scaled(B=3, H=4, seq_lens_override=(65, 1, 130), kv_dtype=kv_dtype,
                                                 extra_pages=2)
    inp = W.make_inputs(w)
    args = lambda c: oracle.mla_decode_ref(inp["q_nope"], inp["q_pe"], c, inp["block_table"], inp["seq_lens"],
                                           w.sm_scale, kv_dtype=kv_dtype, kv_scale=inp["kv_scale"], page_size=64)
    out, lse = args(inp["cache"])
    W.poison_unused(inp)
    out2, lse2 = args(inp["cache"])
    assert np.all(np.isfinite(out2)) and np.array_equal(out, out2) and np.array_equal(lse, lse2)


def test_empty_sequence_and_query():
    w = W.WORKLOADS["paged_bf16_uniform"].scaled(B=2, H=2, q_len=2, seq_lens_override=(0, 1))
    inp = W.make_inputs(w)
    out, lse = oracle.mla_decode_ref(inp["q_nope"], inp["q_pe"], inp["cache"], inp["block_table"],
                                     inp["seq_lens"], 0.1, page_size=64)
    assert np.all(out[0] == 0) and np.all(np.isneginf(lse[0]))
    assert np.all(out[1, 0] == 0) and np.all(np.isneginf(lse[1, 0]))  # query 0 sees nothing
    row = oracle.decode_bf16(inp["cache"][inp["block_table"][1, 0], 0, :512])
    assert np.array_equal(out[1, 1], np.broadcast_to(row, (2, 512)))


# ---------------------------------------------------------------------- host integer helpers

def test_tilegym_integer_helpers():
    assert [oracle.next_power_of_2(n) for n in (-3, 0, 1, 2, 3, 5, 128, 129)] == [1, 1, 1, 2, 4, 8, 128, 256]
    assert [oracle.cdiv(a, 64) for a in (0, 1, 64, 65, 4096)] == [0, 1, 1, 2, 64]
    # 148 SMs, B=1, S=256: estimate 148 -> 256//148=1 -> pow2 1 -> at least 128 -> 2 splits
    assert oracle.tilegym_split_heuristic(148, 1, 256) == (128, 2)
    assert oracle.tilegym_split_heuristic(152, 32, 4096) == (1024, 4)


def test_forced_split_ranges():
    assert oracle.forced_split_ranges(256, 2) == [(0, 128), (128, 256)]
    assert oracle.forced_split_ranges(300, 2) == [(0, 192), (192, 300)]
    assert oracle.forced_split_ranges(10, 4) == [(0, 10)]
    assert oracle.forced_split_ranges(0, 3) == [(0, 0)]


# ---------------------------------------------------------------------- sliding window and sinks

def _windowed(inp, w, window, sinks=None):
    return oracle.mla_decode_ref(inp["q_nope"], inp["q_pe"], inp["cache"], inp["block_table"], inp["seq_lens"],
                                 w.sm_scale, kv_dtype=w.kv_dtype, kv_scale=inp["kv_scale"], page_size=w.page_size,
                                 window=window, sinks=sinks)


def test_window_range_cases():
    assert oracle.window_range(10, 0) == (0, 10)
    assert oracle.window_range(10, 3) == (7, 10)
    assert oracle.window_range(10, 10) == (0, 10)
    assert oracle.window_range(10, 11) == (0, 10)
    assert oracle.window_range(0, 4) == (0, 0)
    assert oracle.window_range(1, 1) == (0, 1)


def test_window_at_least_visible_length_is_no_window():
    w = W.WORKLOADS["paged_bf16_ragged"].scaled(B=3, H=4, q_len=2, seq_lens_override=(5, 130, 64))
    inp = W.make_inputs(w)
    o0, l0 = _windowed(inp, w, 0)
    o1, l1 = _windowed(inp, w, 130)
    assert np.array_equal(o0, o1) and np.array_equal(l0, l1)


def test_window_one_returns_the_last_visible_row():
    w = W.WORKLOADS["paged_bf16_ragged"].scaled(B=2, H=3, q_len=2, seq_lens_override=(77, 2))
    inp = W.make_inputs(w)
    out, lse = _windowed(inp, w, 1)
    for b in range(2):
        L = int(inp["seq_lens"][b])
        keys = oracle.gather_tokens(inp["cache"], inp["block_table"][b], L, "bf16", 64)
        for i in range(2):
            t = L - 2 + i  # the newest position query i sees
            assert np.array_equal(out[b, i], np.broadcast_to(keys[t, :512], (3, 512)))
            q = np.concatenate([oracle.decode_bf16(inp["q_nope"][b, i]), oracle.decode_bf16(inp["q_pe"][b, i])], -1)
            assert np.max(np.abs(lse[b, i] - w.sm_scale * (q @ keys[t]))) < 1e-12


@pytest.mark.parametrize("window", [1, 40, 64, 65, 100])
def test_window_equals_sdpa_with_a_band_mask(window):
    q_len = 3
    w = W.WORKLOADS["paged_fp8"].scaled(B=2, H=4, q_len=q_len, page_size=32, seq_lens_override=(150, 70))
    inp = W.make_inputs(w)
    out, lse = _windowed(inp, w, window)
    for b in range(2):
        L = int(inp["seq_lens"][b])
        keys = torch.from_numpy(oracle.gather_tokens(inp["cache"], inp["block_table"][b], L, "fp8", 32,
                                                     inp["kv_scale"]))
        q = torch.from_numpy(np.concatenate([oracle.decode_bf16(inp["q_nope"][b]),
                                             oracle.decode_bf16(inp["q_pe"][b])], -1))  # [q_len, H, 576]
        t = torch.arange(L)[None, :]
        newest = (L - q_len + torch.arange(q_len))[:, None]  # last position query i sees
        mask = (t <= newest) & (t > newest - window)
        ref = torch.nn.functional.scaled_dot_product_attention(
            q.permute(1, 0, 2), keys[None].expand(4, L, 576), keys[None, :, :512].expand(4, L, 512),
            attn_mask=mask[None].expand(4, q_len, L), scale=w.sm_scale).permute(1, 0, 2)
        assert np.max(np.abs(ref.numpy() - out[b])) < 1e-12
        x = w.sm_scale * torch.einsum("ihc,tc->iht", q, keys)
        lref = torch.logsumexp(x.masked_fill(~mask[:, None, :], -math.inf), dim=-1)
        assert np.max(np.abs(lref.numpy() - lse[b])) < 1e-12


def test_window_equals_a_request_holding_only_the_window():
    # the last W positions copied into a fresh request of length W give the same result
    W_ = 70
    w = W.WORKLOADS["paged_bf16_uniform"].scaled(B=1, H=4, page_size=64, seq_lens_override=(200,))
    inp = W.make_inputs(w)
    out, lse = _windowed(inp, w, W_)
    keys_bits = np.concatenate([inp["cache"][p] for p in inp["block_table"][0, :4]])[:200]
    short = np.zeros((2, 64, 576), dtype=np.uint16)
    short.reshape(128, 576)[:W_] = keys_bits[200 - W_:]
    o2, l2 = oracle.mla_decode_ref(inp["q_nope"], inp["q_pe"], short, np.array([[0, 1]], dtype=np.int32),
                                   np.array([W_]), w.sm_scale)
    assert np.array_equal(out, o2) and np.array_equal(lse, l2)


def test_sink_minus_infinity_is_no_sink():
    w = W.WORKLOADS["paged_bf16_ragged"].scaled(B=2, H=4, seq_lens_override=(90, 0))
    inp = W.make_inputs(w)
    o0, l0 = _windowed(inp, w, 0)
    o1, l1 = _windowed(inp, w, 0, sinks=np.full(4, -np.inf))
    # exp(-inf) adds an exact 0 to the normaliser; only the summation order may differ
    assert np.array_equal(np.isneginf(l0), np.isneginf(l1)) and np.all(o1[1] == 0)
    fin = np.isfinite(l0)
    assert np.max(np.abs(o0 - o1)) < 1e-14 and np.max(np.abs(l0[fin] - l1[fin])) < 1e-13


def test_sink_equal_to_the_single_score_halves_the_row():
    qn, qp, cache = _contig_case(3, 1, seed=61)
    q = np.concatenate([oracle.decode_bf16(qn[0, 0]), oracle.decode_bf16(qp[0, 0])], -1)
    row = oracle.decode_bf16(cache[0, 0])
    x = 0.05 * (q @ row)
    out, lse = oracle.mla_decode_ref(qn, qp, cache, np.array([[0]]), np.array([1]), 0.05, page_size=1, sinks=x)
    assert np.max(np.abs(out[0, 0] - 0.5 * row[None, :512])) < 1e-12
    assert np.max(np.abs(lse[0, 0] - (x + math.log(2.0)))) < 1e-12


def test_sink_with_nothing_visible():
    w = W.WORKLOADS["paged_bf16_ragged"].scaled(B=1, H=3, q_len=2, seq_lens_override=(1,))
    inp = W.make_inputs(w)
    s = np.array([0.5, -2.0, -np.inf])
    out, lse = _windowed(inp, w, 0, sinks=s)
    assert np.all(out[0, 0] == 0) and np.array_equal(lse[0, 0], s)  # query 0 sees no position


def test_sink_is_a_zero_value_token():
    # A token whose latent part is 0 contributes nothing to the output; with its rope part
    # solved so that each head's score equals that head's sink, attending it as an extra
    # token must equal the sink.
    H, n = 16, 29
    rng = np.random.default_rng(71)
    q = rng.standard_normal((H, 576))
    keys = rng.standard_normal((n, 576))
    scale = 0.09
    sinks = rng.uniform(-1.0, 6.0, H)
    k_pe = np.linalg.lstsq(q[:, 512:], sinks / scale, rcond=None)[0]
    assert np.max(np.abs(scale * (q[:, 512:] @ k_pe) - sinks)) < 1e-12
    extra = np.concatenate([np.zeros(512), k_pe])[None]
    o_tok, l_tok = mla_ref.mla_decode_one(q, np.concatenate([keys, extra]), scale)
    o_snk, l_snk = mla_ref.mla_decode_one(q, keys, scale, sink=sinks)
    assert np.max(np.abs(o_tok - o_snk)) < 1e-11 and np.max(np.abs(l_tok - l_snk)) < 1e-11


def test_window_and_sink_pure_python():
    H, n, W_ = 2, 9, 4
    qn, qp, cache = _contig_case(H, n, seed=81)
    sinks = np.array([1.5, -0.25])
    out, lse = oracle.mla_decode_ref(qn, qp, cache, np.array([[0]]), np.array([n]), 0.2, page_size=n,
                                     window=W_, sinks=sinks)
    qf = np.concatenate([oracle.decode_bf16(qn[0, 0]), oracle.decode_bf16(qp[0, 0])], -1).tolist()
    kf = oracle.decode_bf16(cache[0]).tolist()
    for h in range(H):
        xs = [0.2 * math.fsum(qf[h][c] * kf[t][c] for c in range(576)) for t in range(n - W_, n)]
        z = math.fsum([math.exp(x) for x in xs] + [math.exp(sinks[h])])
        assert abs(lse[0, 0, h] - math.log(z)) < 1e-12
        for c in range(0, 512, 41):
            o = math.fsum(math.exp(x) / z * kf[n - W_ + j][c] for j, x in enumerate(xs))
            assert abs(out[0, 0, h, c] - o) < 1e-12


def _workspace_golden():
    rows, bounds = [], []
    with open(os.path.join(GOLDEN, "workspace_bytes.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].split()
            if not line:
                continue
            if line[0] == "bound":
                bounds.append(tuple(int(x) for x in line[1:]))
            else:
                rows.append(tuple(int(x) for x in line))
    return rows, bounds


def test_workspace_bytes_formula_matches_hand_worked_sizes():
    # tokenspeed tokenspeed_mla.py, the CuteDSL decode workspace notes: B*H*q_len*split_kv*(D+1)*acc_bytes
    rows, bounds = _workspace_golden()
    assert len(rows) >= 4 and bounds
    for B, H, q_len, splits, D, acc, want in rows:
        assert oracle.workspace_bytes_formula(B, H, q_len, splits, D=D, acc_bytes=acc) == want
    # the per-device bound of the same notes, num_SMs*H*q_len*(D+1)*4, holds whenever
    # B*split_kv <= num_SMs, and is reached at B*split_kv == num_SMs
    for sms, H, q_len, D, want in bounds:
        for B in (1, 2, 5, 19, 32, 76, 152):
            for splits in range(1, sms // B + 1):
                assert oracle.workspace_bytes_formula(B, H, q_len, splits, D=D) <= want
        assert oracle.workspace_bytes_formula(sms, H, q_len, 1, D=D) == want
        assert oracle.workspace_bytes_formula(8, H, q_len, sms // 8, D=D) == want
    # one partial of one head is the 512 output values plus its log-sum-exp
    assert oracle.workspace_bytes_formula(1, 1, 1, 1) == (512 + 1) * 4
