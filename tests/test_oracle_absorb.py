"""Pins for the per-head projection oracle (metrale mla_batched_gemv) against things other
than itself: pure-Python brute force, identity / permutation weights, and the identity that
makes the absorbed form exact (absorbed Q + latent decode + V up-projection equals ordinary
attention over up-projected keys and values, evaluated with torch SDPA)."""
import math

import numpy as np
import torch

import oracle
from oracle import absorb_ref as AB
from mla_latent_kv_split_gb300 import workloads as W


def _bits(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * scale).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_batched_gemv_brute_force():
    x, w = _bits((2, 3, 5), 1), _bits((3, 4, 5), 2)
    out = AB.batched_gemv_ref(x, w)
    xv, wv = oracle.decode_bf16(x).tolist(), oracle.decode_bf16(w).tolist()
    for t in range(2):
        for h in range(3):
            for n in range(4):
                assert abs(out[t, h, n] - math.fsum(wv[h][n][k] * xv[t][h][k] for k in range(5))) < 1e-14


def test_batched_gemv_identity_and_permutation():
    T, H, K = 3, 4, 64
    x = _bits((T, H, K), 3)
    eye = np.zeros((H, 128, K), np.float64)
    for h in range(H):
        eye[h, :K, :K] = np.eye(K)[np.random.default_rng(h).permutation(K)]
    out = AB.batched_gemv_ref(x, eye)
    xv = oracle.decode_bf16(x)
    for h in range(H):
        perm = np.random.default_rng(h).permutation(K)
        assert np.array_equal(out[:, h, :K], xv[:, h, perm])
        assert np.all(out[:, h, K:] == 0)


def test_absorbed_decode_equals_attention_over_up_projected_kv():
    # DeepSeek-style shapes, scaled: H heads, nope 128, rope 64, latent 512, v 128
    H, n, dn, dv = 4, 37, 128, 128
    rng = np.random.default_rng(9)
    c = rng.standard_normal((n, 512))
    k_pe = rng.standard_normal((n, 64))
    q_nope = rng.standard_normal((1, H, dn))
    q_pe = rng.standard_normal((H, 64))
    w_uk = rng.standard_normal((H, dn, 512)) / math.sqrt(512)
    w_uv = rng.standard_normal((H, dv, 512)) / math.sqrt(512)
    scale = 1 / math.sqrt(dn + 64)
    # absorbed path: q_lat = W_UK^T q_nope per head, latent decode, o = W_UV o_lat
    q_lat = AB.batched_gemv_ref(q_nope, np.transpose(w_uk, (0, 2, 1)))[0]  # [H, 512]
    o_lat, lse = oracle.mla_decode_one(np.concatenate([q_lat, q_pe], -1), np.concatenate([c, k_pe], -1), scale)
    o = AB.batched_gemv_ref(o_lat[None], w_uv)[0]  # [H, dv]
    # ordinary attention: K_h = [W_UK c | k_pe], V_h = W_UV c
    k = torch.from_numpy(np.concatenate([np.einsum("hdc,tc->htd", w_uk, c), np.broadcast_to(k_pe, (H, n, 64))], -1))
    v = torch.from_numpy(np.einsum("hdc,tc->htd", w_uv, c))
    q = torch.from_numpy(np.concatenate([q_nope[0], q_pe], -1))[:, None]
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, scale=scale)[:, 0].numpy()
    assert np.max(np.abs(o - ref)) < 1e-12
    lref = torch.logsumexp(scale * (q @ k.transpose(1, 2))[:, 0], dim=-1).numpy()
    assert np.max(np.abs(lse - lref)) < 1e-12
