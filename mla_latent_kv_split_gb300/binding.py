"""Python binding of ``libmla_decode.so`` (the C ABI in ``include/mla_decode.h``).

Argument marshalling only: shapes and raw device pointers are read from torch tensors
(torch is used for device memory and streams) and passed to the C entry points of the
same names.  Every step of the decode runs in the library's CUDA kernels; there is no
fallback of any kind, and a missing library raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "lib", "libmla_decode.so")

MLA_KV_BF16, MLA_KV_FP8_E4M3, MLA_KV_NVFP4 = 0, 1, 2
MLA_SMALL_CALL_DEFAULT = 256  # include/mla_decode.h
KV_DTYPE = {"bf16": MLA_KV_BF16, "fp8": MLA_KV_FP8_E4M3, "nvfp4": MLA_KV_NVFP4}
STATUS_BITS = {
    0x1: "PAGE_OUT_OF_RANGE", 0x2: "SEQ_TOO_LONG", 0x4: "SEQ_LT_QLEN", 0x8: "NEG_SEQ_LEN",
    0x10: "WAIT_TIMEOUT", 0x20: "Q_RANGE", 0x40: "SLOT_OUT_OF_RANGE",
}
EXPORTED = (
    "mla_decode_abi_version", "mla_status_string", "mla_decode_workspace_size", "mla_decode",
    "mla_splitk_reduce", "mla_decode_read_status", "mla_decode_num_workers", "mla_decode_plan_host",
    "mla_decode_no_alloc", "mla_decode_ex", "mla_kv_append", "mla_batched_gemv",
    "mla_decode_set_small_call_limit",
)


class MLAError(RuntimeError):
    def __init__(self, fn: str, code: int, msg: str):
        super().__init__(f"{fn} failed: {msg} ({code})")
        self.code = code


_lock = threading.Lock()
_handle = None


def lib() -> ctypes.CDLL:
    """The loaded library (opened once).  Raises if it has not been built."""
    global _handle
    with _lock:
        if _handle is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                                   "or python mla_latent_kv_split_gb300/build.py")
            h = ctypes.CDLL(LIB_PATH)
            P, I, F, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
            h.mla_decode_abi_version.restype = I
            h.mla_status_string.restype = ctypes.c_char_p
            h.mla_status_string.argtypes = [I]
            h.mla_decode_workspace_size.restype = I
            h.mla_decode_workspace_size.argtypes = [I, I, I, I, ctypes.POINTER(Z)]
            h.mla_decode.restype = I
            h.mla_decode.argtypes = [P, P, P, P, I, P, I, I, I, I, I, F, I, F, I, P, Z, P, P, P]
            h.mla_decode_ex.restype = I
            h.mla_decode_ex.argtypes = [P, P, P, P, I, P, I, I, I, I, I, F, I, F, I, I, P, P, Z, P, P, P]
            h.mla_splitk_reduce.restype = I
            h.mla_splitk_reduce.argtypes = [P, Z, I, I, I, P, P, P, P]
            h.mla_decode_read_status.restype = I
            h.mla_decode_read_status.argtypes = [P, ctypes.POINTER(ctypes.c_uint32), P]
            h.mla_decode_num_workers.restype = I
            h.mla_decode_num_workers.argtypes = [ctypes.POINTER(I)]
            i32p = ctypes.POINTER(ctypes.c_int32)
            h.mla_decode_plan_host.restype = I
            h.mla_decode_plan_host.argtypes = [i32p, I, I, I, I, I, I, I, i32p, i32p, i32p, i32p, i32p]
            L64 = ctypes.c_int64
            h.mla_kv_append.restype = I
            h.mla_kv_append.argtypes = [P, L64, P, L64, P, I, P, I, I, I, F, P, P]
            h.mla_batched_gemv.restype = I
            h.mla_batched_gemv.argtypes = [P, L64, L64, P, P, L64, L64, I, I, I, I, P, P]
            h.mla_decode_set_small_call_limit.restype = Z
            h.mla_decode_set_small_call_limit.argtypes = [Z]
            h.mla_decode_no_alloc.restype = I
            h.mla_decode_no_alloc.argtypes = [P, P, P, P, I, P, I, I, I, I, I, F, I, F, I, P, P, P,
                                              ctypes.POINTER(P)]
            _handle = h
        return _handle


def _check(fn: str, code: int) -> None:
    if code != 0:
        raise MLAError(fn, code, lib().mla_status_string(code).decode())


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream_ptr(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def mla_decode_workspace_size(B: int, q_len: int, H: int, num_splits: int = 0) -> int:
    n = ctypes.c_size_t(0)
    _check("mla_decode_workspace_size", lib().mla_decode_workspace_size(B, q_len, H, num_splits, ctypes.byref(n)))
    return n.value


def mla_decode_set_small_call_limit(limit: int) -> int:
    """Sets the small-call limit (bf16 calls whose key ranges span at most this many cache
    positions run on the CUDA-core decode kernel; 0: never); returns the previous limit."""
    return int(lib().mla_decode_set_small_call_limit(int(limit)))


def mla_decode_num_workers() -> int:
    w = ctypes.c_int(0)
    _check("mla_decode_num_workers", lib().mla_decode_num_workers(ctypes.byref(w)))
    return w.value


def alloc_workspace(B: int, q_len: int, H: int, num_splits: int = 0, device=None):
    """A torch uint8 device buffer of the size mla_decode needs (plumbing only)."""
    import torch
    n = mla_decode_workspace_size(B, q_len, H, num_splits)
    return torch.empty(n, dtype=torch.uint8, device=device or "cuda")


def mla_decode(q_nope, q_pe, kv_cache, block_table, seq_lens, sm_scale: float, kv_dtype="bf16",
               kv_scale: float = 1.0, num_splits: int = 0, page_size: int | None = None,
               num_pages: int | None = None, workspace=None, out=None, lse=None, stream=None,
               window: int = 0, sinks=None):
    """Calls ``mla_decode`` (or ``mla_decode_ex`` when ``window`` or ``sinks`` is given).
    Tensors: ``q_nope [B,q_len,H,512]`` / ``q_pe [B,q_len,H,64]`` bf16, ``kv_cache``
    (``[P,ps,576]`` bf16 / uint8, or ``[P, ps*324]`` uint8 for NVFP4 with ``page_size``
    given), ``block_table [B,max_pages]`` int32, ``seq_lens [B]`` int32, ``sinks [H]`` fp32,
    all on the device.  Returns ``(out, lse)`` (allocated with torch when not given)."""
    import torch
    B, q_len, H, _ = q_nope.shape
    kd = KV_DTYPE[kv_dtype] if isinstance(kv_dtype, str) else int(kv_dtype)
    if page_size is None:
        page_size = kv_cache.shape[1]
    if num_pages is None:
        num_pages = kv_cache.shape[0]
    if workspace is None:
        workspace = alloc_workspace(B, q_len, H, num_splits, q_nope.device)
    if out is None:
        out = torch.empty((B, q_len, H, 512), dtype=torch.bfloat16, device=q_nope.device)
    if lse is None:
        lse = torch.empty((B, q_len, H), dtype=torch.float32, device=q_nope.device)
    nbytes = workspace.numel() * workspace.element_size() if not isinstance(workspace, int) else 1 << 62
    head = (_ptr(q_nope), _ptr(q_pe), _ptr(kv_cache), _ptr(block_table), int(block_table.shape[1]),
            _ptr(seq_lens), B, q_len, H, int(num_pages), int(page_size), float(sm_scale), kd,
            float(kv_scale), int(num_splits))
    tail = (_ptr(workspace), nbytes, _ptr(out), _ptr(lse), _stream_ptr(stream))
    if window or sinks is not None:
        _check("mla_decode_ex", lib().mla_decode_ex(*head, int(window), _ptr(sinks), *tail))
    else:
        _check("mla_decode", lib().mla_decode(*head, *tail))
    return out, lse


def mla_splitk_reduce(workspace, B: int, q_len: int, H: int, out, lse=None, stream=None, sinks=None):
    _check("mla_splitk_reduce", lib().mla_splitk_reduce(
        _ptr(workspace), workspace.numel() * workspace.element_size(), B, q_len, H, _ptr(sinks), _ptr(out),
        _ptr(lse), _stream_ptr(stream)))
    return out, lse


def mla_decode_read_status(workspace, stream=None) -> int:
    """The device status word of the last decode on ``workspace`` (synchronises)."""
    v = ctypes.c_uint32(0)
    code = lib().mla_decode_read_status(_ptr(workspace), ctypes.byref(v), _stream_ptr(stream))
    if code not in (0, 5):
        _check("mla_decode_read_status", code)
    return v.value


def mla_decode_plan_host(seq_lens, q_len: int, max_pages: int, page_size: int, num_splits: int = 0,
                         workers: int = 0, window: int = 0):
    """The schedule as the kernels evaluate it, computed on the host (for tests)."""
    sl = np.ascontiguousarray(np.asarray(seq_lens, dtype=np.int32))
    B = sl.shape[0]
    U = B * q_len
    arrs = [np.zeros(U, dtype=np.int32) for _ in range(4)]
    used = ctypes.c_int32(0)
    i32p = ctypes.POINTER(ctypes.c_int32)
    _check("mla_decode_plan_host", lib().mla_decode_plan_host(
        sl.ctypes.data_as(i32p), B, q_len, max_pages, page_size, num_splits, int(window), workers,
        *[a.ctypes.data_as(i32p) for a in arrs], ctypes.byref(used)))
    return dict(tile_begin=arrs[0], tiles=arrs[1], parts=arrs[2], slot=arrs[3], slots_used=used.value)


def mla_decode_no_alloc(q_nope, q_pe, kv_cache, block_table, seq_lens, sm_scale: float, kv_dtype="bf16",
                        kv_scale: float = 1.0, num_splits: int = 0, page_size: int | None = None,
                        num_pages: int | None = None, out=None, lse=None, stream=None):
    """Calls ``mla_decode_no_alloc`` (scratch in the library's static device buffer; for
    callers that cannot allocate).  Returns ``(out, lse, scratch_address)``; ``out``/``lse``
    are allocated with torch here only when not given."""
    import torch
    B, q_len, H, _ = q_nope.shape
    kd = KV_DTYPE[kv_dtype] if isinstance(kv_dtype, str) else int(kv_dtype)
    if page_size is None:
        page_size = kv_cache.shape[1]
    if num_pages is None:
        num_pages = kv_cache.shape[0]
    if out is None:
        out = torch.empty((B, q_len, H, 512), dtype=torch.bfloat16, device=q_nope.device)
    if lse is None:
        lse = torch.empty((B, q_len, H), dtype=torch.float32, device=q_nope.device)
    scratch = ctypes.c_void_p(0)
    _check("mla_decode_no_alloc", lib().mla_decode_no_alloc(
        _ptr(q_nope), _ptr(q_pe), _ptr(kv_cache), _ptr(block_table), int(block_table.shape[1]),
        _ptr(seq_lens), B, q_len, H, int(num_pages), int(page_size), float(sm_scale), kd,
        float(kv_scale), int(num_splits), _ptr(out), _ptr(lse), _stream_ptr(stream), ctypes.byref(scratch)))
    return out, lse, scratch.value


def mla_kv_append(latent, rope, slots, kv_cache, page_size: int | None = None, kv_dtype="bf16",
                  kv_scale: float = 1.0, num_pages: int | None = None, device_status=None, stream=None):
    """Calls ``mla_kv_append``: ``latent [T, 512]`` / ``rope [T, 64]`` bf16 row views (any
    row stride that is a multiple of 8 elements, unit stride inside a row), ``slots [T]``
    int64, all on the device; ``kv_cache`` as for :func:`mla_decode`; ``device_status`` an
    optional int32/uint32 device tensor of one element that out-of-range slots OR a bit into."""
    T = int(slots.shape[0])
    kd = KV_DTYPE[kv_dtype] if isinstance(kv_dtype, str) else int(kv_dtype)
    if page_size is None:
        page_size = kv_cache.shape[1]
    if num_pages is None:
        num_pages = kv_cache.shape[0]
    for t, w in ((latent, 512), (rope, 64)):
        if T and (t.dim() != 2 or t.shape[0] != T or t.shape[1] != w or t.stride(1) != 1):
            raise ValueError(f"expected a [{T}, {w}] row view with unit column stride, got {tuple(t.shape)}")
    _check("mla_kv_append", lib().mla_kv_append(
        _ptr(latent), int(latent.stride(0)) if T else 512, _ptr(rope), int(rope.stride(0)) if T else 64,
        _ptr(slots), T, _ptr(kv_cache), int(num_pages), int(page_size), kd, float(kv_scale),
        _ptr(device_status), _stream_ptr(stream)))
    return kv_cache


def mla_batched_gemv(x, weight, out=None, device_status=None, stream=None):
    """Calls ``mla_batched_gemv``: ``x [T, H, K]`` bf16 (any token / head strides that are
    multiples of 8 elements, unit stride along K), ``weight [H, N, K]`` bf16 contiguous,
    ``out [T, H, N]`` bf16 (allocated with torch when not given; unit stride along N).
    Returns ``out`` with ``out[t, h, n] = sum_k weight[h, n, k] * x[t, h, k]``."""
    import torch
    T, H, K = x.shape
    H2, N, K2 = weight.shape
    if (H2, K2) != (H, K) or x.stride(2) != 1 or not weight.is_contiguous():
        raise ValueError(f"shapes x {tuple(x.shape)} / weight {tuple(weight.shape)} do not match")
    if out is None:
        out = torch.empty((T, H, N), dtype=torch.bfloat16, device=x.device)
    if tuple(out.shape) != (T, H, N) or out.stride(2) != 1:
        raise ValueError(f"out must be a [{T}, {H}, {N}] view with unit stride along N")
    _check("mla_batched_gemv", lib().mla_batched_gemv(
        _ptr(x), int(x.stride(0)), int(x.stride(1)), _ptr(weight), _ptr(out), int(out.stride(0)), int(out.stride(1)),
        T, H, N, K, _ptr(device_status), _stream_ptr(stream)))
    return out
