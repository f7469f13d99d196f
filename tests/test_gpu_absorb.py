"""GPU parity of the per-head batched projection (metrale mla_batched_gemv) against the
float64 oracle: the Q absorption and V up-projection shapes of DeepSeek-style MLA (H
heads, nope 128, latent 512, v 128) for decode-sized and larger token counts (several
token tiles, ragged tails), strided inputs (q_nope read straight out of [T, H, 192] raw
query rows), ragged N and K (out-of-range rows and columns read as zeros), and the chain
absorb -> decode -> up-project against the oracle chain."""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import absorb_ref as AB
from mla_latent_kv_split_gb300 import binding as mb
from mla_latent_kv_split_gb300 import workloads as W

from gpu_util import ATOL, RTOL, ensure_built, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()


def _bf16(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * scale).to(torch.bfloat16)


def _bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _check(out, ref, what):
    out = out.float().cpu().double().numpy()
    err = np.abs(out - ref)
    bound = ATOL + RTOL * np.abs(ref)
    worst = np.unravel_index(np.argmax(err - bound), err.shape)
    assert np.all(err <= bound), f"{what}: err {err[worst]:.3g} > {bound[worst]:.3g} at {worst}"
    rel = np.linalg.norm(out - ref) / max(np.linalg.norm(ref), 1e-30)
    assert rel <= 5e-3, f"{what}: rel L2 {rel:.3g}"


@pytest.mark.parametrize("T", [1, 32, 300])
@pytest.mark.parametrize("H", [16, 128])
def test_q_absorption(T, H):
    raw = _bf16((T, H, 192), 1 + T)             # [q_nope 128 | q_pe 64] per head
    w_ukT = _bf16((H, 512, 128), 2, 1 / math.sqrt(128))  # W_UK^T per head
    x = raw[:, :, :128]
    ref = AB.batched_gemv_ref(_bits(x), _bits(w_ukT))
    out = mb.mla_batched_gemv(x.cuda(), w_ukT.cuda())
    torch.cuda.synchronize()
    _check(out, ref, f"absorb T{T} H{H}")


@pytest.mark.parametrize("T", [1, 32, 257])
def test_v_up_projection(T):
    H = 128
    o_lat = _bf16((T, H, 512), 3 + T, 0.2)
    w_uv = _bf16((H, 128, 512), 4, 1 / math.sqrt(512))
    ref = AB.batched_gemv_ref(_bits(o_lat), _bits(w_uv))
    out = torch.full((T, H, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    mb.mla_batched_gemv(o_lat.cuda(), w_uv.cuda(), out=out)
    torch.cuda.synchronize()
    _check(out, ref, f"v-up T{T}")


def test_ragged_n_and_k_and_strided_out():
    T, H, N, K = 19, 3, 200, 72
    x = _bf16((T, H, K), 5)
    w = _bf16((H, N, K), 6, 0.1)
    ref = AB.batched_gemv_ref(_bits(x), _bits(w))
    big = torch.zeros((T, H, N + 40), dtype=torch.bfloat16, device="cuda")
    out = big[:, :, 16:16 + N]
    mb.mla_batched_gemv(x.cuda(), w.cuda(), out=out)
    torch.cuda.synchronize()
    _check(out, ref, "ragged")
    assert torch.count_nonzero(big[:, :, :16]) == 0 and torch.count_nonzero(big[:, :, 16 + N:]) == 0


def test_absorb_decode_up_chain():
    # q_nope (raw) -> absorbed q -> split-KV decode -> V up-projection, against the oracle
    # chain in float64 (the GPU chain rounds the absorbed q and the latent output to bf16)
    w = W.WORKLOADS["paged_bf16_ragged"].scaled(B=3, H=32, seq_lens_override=(700, 65, 2000))
    inp = W.make_inputs(w)
    T, H = w.B * w.q_len, w.H
    q_raw = _bf16((T, H, 128), 7)
    w_ukT = _bf16((H, 512, 128), 8, 1 / math.sqrt(128))
    w_uv = _bf16((H, 128, 512), 9, 1 / math.sqrt(512))
    dev = to_device(inp)
    q_lat = torch.empty((w.B, w.q_len, H, 512), dtype=torch.bfloat16, device="cuda")
    mb.mla_batched_gemv(q_raw.cuda(), w_ukT.cuda(), out=q_lat.view(T, H, 512))
    out_lat, lse = mb.mla_decode(q_lat, dev["q_pe"], dev["cache"], dev["block_table"], dev["seq_lens"], w.sm_scale,
                                 w.kv_dtype, inp["kv_scale"], page_size=w.page_size, num_pages=inp["num_pages"])
    o = mb.mla_batched_gemv(out_lat.view(T, H, 512), w_uv.cuda())
    torch.cuda.synchronize()

    q_lat_ref = AB.batched_gemv_ref(_bits(q_raw), _bits(w_ukT))  # [T, H, 512] float64
    ref = np.empty((T, H, 128))
    for b in range(w.B):
        L = int(inp["seq_lens"][b])
        keys = oracle.gather_tokens(inp["cache"], inp["block_table"][b], L, w.kv_dtype, w.page_size)
        q = np.concatenate([q_lat_ref[b], oracle.decode_bf16(inp["q_pe"][b, 0])], -1)
        o_lat, _ = oracle.mla_decode_one(q, keys, w.sm_scale)
        ref[b] = AB.batched_gemv_ref(o_lat[None], _bits(w_uv))[0]
    _check(o, ref, "absorb-decode-up")
