"""GPU parity of the KV-cache append with quantise-on-write against the append oracle:
the stored bytes must be identical (every rounding decision is taken on the same fp32
quotients on both sides), for the three formats and both page sizes, with padding and
out-of-range locations, strided [T, 576] inputs, values that round to signed zero or
saturate, and all-zero groups.  Then the path it feeds: append this step's tokens and
decode, against the decode oracle on the oracle-appended cache."""
import numpy as np
import pytest
import torch

import oracle
from oracle import kv_append_ref as KA
from mla_latent_kv_split_gb300 import binding as mb
from mla_latent_kv_split_gb300 import workloads as W

from gpu_util import assert_close, ensure_built, oracle_ref, run_decode, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()


def _tokens(T, seed, specials=True):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn((T, 576), generator=g) * 2
    if specials and T > 3:
        x[1, :16] = 0  # all-zero group
        x[2, 16:32] = torch.tensor([1e-30, -1e-30] * 8)  # rounds to signed zeros
        x[3, 40] = 3e4  # large outlier in a group
        x[3, 41] = -3e4
    return x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _empty_cache(kv_dtype, num_pages, ps, fill):
    if kv_dtype == "bf16":
        return np.full((num_pages, ps, 576), fill, np.uint16)
    if kv_dtype == "fp8":
        return np.full((num_pages, ps, 576), fill & 0xFF, np.uint8)
    return np.full((num_pages, oracle.nvfp4_page_bytes(ps)), fill & 0xFF, np.uint8)


def _to_dev_cache(cache):
    if cache.dtype == np.uint16:
        return torch.from_numpy(cache.view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(cache).cuda()


def _from_dev_cache(dcache, like):
    if like.dtype == np.uint16:
        return dcache.view(torch.int16).cpu().numpy().view(np.uint16)
    return dcache.cpu().numpy()


@pytest.mark.parametrize("T", [1, 7, 100])
@pytest.mark.parametrize("ps", [32, 64])
@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8", "nvfp4"])
def test_append_bytes_equal_oracle(kv_dtype, ps, T):
    num_pages = 5
    bits = _tokens(T, seed=T + ps)
    rng = np.random.default_rng(T * 7 + ps)
    slots = rng.permutation(num_pages * ps)[:T].astype(np.int64)
    if T > 4:
        slots[0] = -1  # padding
        slots[4] = num_pages * ps + 3  # past the cache
    kv_scale = 0.05 if kv_dtype == "fp8" else 1.0  # 3e4 / 0.05 saturates E4M3
    cache = _empty_cache(kv_dtype, num_pages, ps, 0x5A5A)
    ref = KA.kv_append_ref(cache, bits[:, :512], bits[:, 512:], slots, kv_dtype, ps, kv_scale)

    x = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()  # [T, 576]
    dcache = _to_dev_cache(cache)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mb.mla_kv_append(x[:, :512], x[:, 512:], torch.from_numpy(slots).cuda(), dcache, page_size=ps,
                     kv_dtype=kv_dtype, kv_scale=kv_scale, num_pages=num_pages, device_status=status)
    torch.cuda.synchronize()
    got = _from_dev_cache(dcache, cache)
    assert np.array_equal(got, ref), f"{np.count_nonzero(got != ref)} bytes differ"
    assert int(status.item()) == (0x40 if T > 4 else 0)


def test_append_empty_batch_is_a_noop():
    cache = torch.zeros((1, 64, 576), dtype=torch.bfloat16, device="cuda")
    e = torch.empty((0, 576), dtype=torch.bfloat16, device="cuda")
    mb.mla_kv_append(e[:, :512], e[:, 512:], torch.empty(0, dtype=torch.int64, device="cuda"), cache)
    torch.cuda.synchronize()
    assert torch.count_nonzero(cache) == 0


@pytest.mark.parametrize("num_splits", [0, 3])
@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8", "nvfp4"])
def test_append_then_decode(kv_dtype, num_splits):
    # q_len = 2 new tokens per request are written at positions seq_len-2, seq_len-1 (their
    # pages already in the block table), then decoded
    q_len = 2
    w = W.WORKLOADS["paged_fp8"].scaled(B=4, q_len=q_len, H=32, kv_dtype=kv_dtype,
                                        seq_lens_override=(2, 65, 700, 129))
    inp = W.make_inputs(w)
    ps = w.page_size
    T = w.B * q_len
    bits = _tokens(T, seed=11, specials=False)  # scores in the workloads' range
    slots = np.empty(T, np.int64)
    for b in range(w.B):
        L = int(inp["seq_lens"][b])
        for i in range(q_len):
            pos = L - q_len + i
            slots[b * q_len + i] = int(inp["block_table"][b, pos // ps]) * ps + pos % ps
    kv_scale = inp["kv_scale"]
    new_cache = KA.kv_append_ref(inp["cache"], bits[:, :512], bits[:, 512:], slots, kv_dtype, ps, kv_scale)

    dev = to_device(inp)
    x = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()
    mb.mla_kv_append(x[:, :512], x[:, 512:], torch.from_numpy(slots).cuda(), dev["cache"], page_size=ps,
                     kv_dtype=kv_dtype, kv_scale=kv_scale, num_pages=inp["num_pages"])
    got = _from_dev_cache(dev["cache"], inp["cache"])
    assert np.array_equal(got, new_cache)
    out, lse, status, _ = run_decode(inp, dev=dev, num_splits=num_splits)
    assert status == 0, hex(status)
    inp2 = dict(inp)
    inp2["cache"] = new_cache
    assert_close(out, lse, *oracle_ref(inp2), what=f"append+decode {kv_dtype}")


def _every_finite_bf16(shuffle_seed=None):
    """All 65,280 finite bf16 bit patterns (both zeros, subnormals, up to +-max), as
    [T, 576] token rows, padded with zeros."""
    b = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    b = b[(b & 0x7F80) != 0x7F80]
    if shuffle_seed is not None:
        b = np.random.default_rng(shuffle_seed).permutation(b)
    T = -(-b.size // 576)
    out = np.zeros(T * 576, np.uint16)
    out[:b.size] = b
    return out.reshape(T, 576)


def _append_both(kv_dtype, bits, kv_scale, ps=64):
    T = bits.shape[0]
    num_pages = -(-T // ps)
    slots = np.arange(T, dtype=np.int64)
    cache = _empty_cache(kv_dtype, num_pages, ps, 0)
    ref = KA.kv_append_ref(cache, bits[:, :512], bits[:, 512:], slots, kv_dtype, ps, kv_scale)
    x = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()
    dcache = _to_dev_cache(cache)
    mb.mla_kv_append(x[:, :512], x[:, 512:], torch.from_numpy(slots).cuda(), dcache, page_size=ps,
                     kv_dtype=kv_dtype, kv_scale=kv_scale, num_pages=num_pages)
    torch.cuda.synchronize()
    return _from_dev_cache(dcache, cache), ref


@pytest.mark.parametrize("kv_scale", [1.0, 0.05, 1.0 / 3.0, 0.0123456789, 2.0 ** -7, 3.7, 448.0 / 3.0, 1e-30, 1e30])
def test_fp8_append_every_bf16_value(kv_scale):
    # every finite bf16 value divided by the scale and rounded to E4M3: the quotient the
    # kernel forms (reciprocal and one correction step) must be the correctly rounded one
    # wherever that decides the code, so every stored byte equals the oracle's
    got, ref = _append_both("fp8", _every_finite_bf16(), np.float32(kv_scale).item())
    assert np.array_equal(got, ref), f"{np.count_nonzero(got != ref)} bytes differ"


@pytest.mark.parametrize("seed", [0, 1])
def test_nvfp4_append_every_bf16_value(seed):
    # every finite bf16 value, sorted by magnitude into groups of 15 neighbours, each group
    # completed by a 16th value that sets its block scale at 1 to 12 times the group's
    # largest (so x / scale covers every E2M1 code): the scale E4M3(amax / 6) and each code
    # E2M1(x / scale) as the oracle's
    b = _every_finite_bf16().reshape(-1)
    v = torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).float().numpy()
    v = v[np.argsort(np.abs(v), kind="stable")]
    rng = np.random.default_rng(seed)
    n = -(-v.size // 15)
    vals = np.zeros(n * 15, np.float32)
    vals[:v.size] = v * np.where(rng.random(v.size) < 0.5, -1.0, 1.0)
    groups = np.zeros((n, 16), np.float32)
    groups[:, 1:] = vals.reshape(n, 15)
    factors = np.array([1.0, 1.3, 1.7, 2.3, 3.0, 4.0, 5.5, 7.5, 12.0], np.float32)
    with np.errstate(over="ignore"):
        setter = np.abs(groups[:, 1:]).max(axis=1) * factors[rng.integers(0, factors.size, n)]
    groups[:, 0] = np.minimum(setter, np.float32(3.3895314e38))  # the largest finite bf16
    x = torch.from_numpy(groups.reshape(-1))
    T = -(-x.numel() // 576)
    flat = torch.zeros(T * 576)
    flat[:x.numel()] = x
    bits = flat.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).reshape(T, 576)
    got, ref = _append_both("nvfp4", bits, 1.0)
    assert np.array_equal(got, ref), f"{np.count_nonzero(got != ref)} bytes differ"
