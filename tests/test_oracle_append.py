"""Pins for the KV-append oracle (quantise-on-write), against things other than itself:
torch's float8_e4m3fn cast, the OCP value tables and hand-derived E2M1 rounding cases
(tests/golden), brute-force nearest-value search, the seeded input generator's own
torch-based quantisers (a separate implementation of the same recipe), and round trips
through the decode oracle within the formats' half-step bound."""
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import kv_append_ref as KA
from mla_latent_kv_split_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_e4m3_encoder_matches_torch_cast():
    pos = oracle.E4M3_TABLE[:0x7F]
    mids = (pos[:-1] + pos[1:]) / 2  # every tie between neighbouring codes
    rng = np.random.default_rng(1)
    xs = np.concatenate([pos, mids, np.nextafter(mids.astype(np.float32), np.float32(np.inf)),
                         np.nextafter(mids.astype(np.float32), np.float32(-np.inf)),
                         rng.uniform(-448, 448, 200000), rng.standard_normal(50000) * 1e-3,
                         np.float32(2.0) ** -np.arange(5, 30, dtype=np.float32)]).astype(np.float32)
    xs = np.concatenate([xs, -xs])
    ref = torch.from_numpy(xs).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(KA.encode_e4m3(xs), ref)


def test_e4m3_encoder_saturates():
    assert KA.encode_e4m3(np.array([448.0, 464.0, 480.0, 1e9], np.float32)).tolist() == [0x7E] * 4
    assert KA.encode_e4m3(np.array([-464.0, -1e30], np.float32)).tolist() == [0xFE] * 2
    assert KA.encode_e4m3(np.array([0.0, -0.0, -1e-30], np.float32)).tolist() == [0x00, 0x80, 0x80]


def test_e2m1_encoder_golden_rounding():
    rows = []
    for line in open(os.path.join(GOLDEN, "e2m1_rounding.txt")):
        line = line.strip()
        if line and not line.startswith("#"):
            v, c = line.split()
            rows.append((float(v), int(c)))
    xs = np.array([v for v, _ in rows], np.float32)
    assert KA.encode_e2m1(xs).tolist() == [c for _, c in rows]


def test_e2m1_encoder_every_code_and_brute_force():
    assert KA.encode_e2m1(oracle.E2M1_TABLE.astype(np.float32)).tolist() == list(range(16))
    rng = np.random.default_rng(2)
    xs = rng.uniform(-8, 8, 20000).astype(np.float32)
    codes = KA.encode_e2m1(xs)
    vals = oracle.E2M1_TABLE[:8]
    for x, c in zip(xs[:4000], codes[:4000]):
        d = np.abs(vals - min(abs(float(x)), 6.0))
        best = np.flatnonzero(d == d.min())
        want = best[0] if len(best) == 1 else best[best % 2 == 0][0]
        assert c == (want | (8 if x < 0 else 0))


def _rows(T, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn((T, 576), generator=g) * 3
    bits = x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    return bits[:, :512].copy(), bits[:, 512:].copy(), bits


def test_fp8_append_matches_generator_quantiser():
    lat, rope, bits = _rows(40, 3)
    x = torch.from_numpy(oracle.decode_bf16(bits).astype(np.float32))
    scale = float(np.float32(x.abs().max().item() / 448.0))
    cache = np.zeros((2, 32, 576), np.uint8)
    out = KA.kv_append_ref(cache, lat, rope, np.arange(40) + 10, "fp8", 32, scale)
    ref = W.quantize_e4m3_rne(x / torch.tensor(scale, dtype=torch.float32))
    assert np.array_equal(out.reshape(64, 576)[10:50], ref)
    assert np.all(out.reshape(64, 576)[:10] == 0) and np.all(out.reshape(64, 576)[50:] == 0)


@pytest.mark.parametrize("ps", [32, 64])
def test_nvfp4_append_matches_generator_quantiser(ps):
    T = ps + 5
    lat, rope, bits = _rows(T, 4)
    x = torch.from_numpy(oracle.decode_bf16(bits).astype(np.float32))
    x[3, :16] = 0  # an all-zero group
    bits[3, :16] = 0
    lat[3, :16] = 0
    cache = np.zeros((2, oracle.nvfp4_page_bytes(ps)), np.uint8)
    out = KA.kv_append_ref(cache, lat, rope, np.arange(T), "nvfp4", ps)
    pad = torch.zeros((2 * ps, 576))
    pad[:T] = x
    ref = W.quantize_nvfp4_pages(pad.reshape(2, ps, 576))
    data = ps * 288
    assert np.array_equal(out[0], ref[0])
    assert np.array_equal(out[1, :5 * 288], ref[1, :5 * 288])
    assert np.array_equal(out[1, data:data + 5 * 36], ref[1, data:data + 5 * 36])
    assert np.all(out[1, 5 * 288:data] == 0) and np.all(out[1, data + 5 * 36:] == 0)


def test_append_round_trip_within_half_step():
    lat, rope, bits = _rows(64, 5)
    x = oracle.decode_bf16(bits)
    slots = np.random.default_rng(6).permutation(64)
    # bf16: exact
    c = KA.kv_append_ref(np.zeros((1, 64, 576), np.uint16), lat, rope, slots, "bf16", 64)
    assert np.array_equal(oracle.dequant_pages(c, "bf16", 64, 1.0, [0])[0][slots], x)
    # fp8: |x/s - e4m3| <= half the spacing of E4M3 at that magnitude (3 mantissa bits)
    s = float(np.float32(np.abs(x).max() / 448.0))
    c = KA.kv_append_ref(np.zeros((1, 64, 576), np.uint8), lat, rope, slots, "fp8", 64, s)
    y = oracle.dequant_pages(c, "fp8", 64, s, [0])[0][slots] / s
    q = x / s
    ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(q), 2.0 ** -6))) - 3)
    assert np.all(np.abs(y - q) <= ulp / 2 * (1 + 1e-6))
    # nvfp4: per group |x - v| <= scale * (half the E2M1 spacing at that magnitude), the
    # spacing being 0.5 below 2, 1 in [2, 4), 2 above
    c = KA.kv_append_ref(np.zeros((1, oracle.nvfp4_page_bytes(64)), np.uint8), lat, rope, slots, "nvfp4", 64)
    y = oracle.dequant_pages(c, "nvfp4", 64, 1.0, [0])[0][slots]
    data = 64 * 288
    sc = oracle.decode_e4m3(c[0, data:].reshape(64, 36))[slots]
    sc16 = np.repeat(sc, 16, axis=1)
    r = np.abs(x) / sc16
    step = np.where(r < 2, 0.5, np.where(r < 4, 1.0, 2.0))
    within = r <= 6
    assert np.all(np.abs(y - x)[within] <= (sc16 * step / 2)[within] * (1 + 1e-9))
    assert np.all(np.abs(y[~within]) == 6 * sc16[~within])  # saturated (scale rounded down)


def test_append_skips_padding_and_out_of_range_slots():
    lat, rope, bits = _rows(4, 7)
    cache = np.full((2, 32, 576), 0x1234, np.uint16)
    out = KA.kv_append_ref(cache, lat, rope, np.array([-1, 5, 64, 63]), "bf16", 32)
    flat = out.reshape(64, 576)
    assert np.array_equal(flat[5], bits[1]) and np.array_equal(flat[63], bits[3])
    keep = np.ones(64, bool)
    keep[[5, 63]] = False
    assert np.all(flat[keep] == 0x1234)
