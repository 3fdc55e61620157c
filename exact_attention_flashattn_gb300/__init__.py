"""Exact scaled-dot-product attention on GB300: Python binding of ``libbwattn``.

Every function here only checks and marshals arguments (shapes, dtypes, device pointers,
the current CUDA stream) and calls the C-ABI in ``libbwattn.so``; all arithmetic runs in the
library's CUDA kernels. PyTorch supplies device memory and streams. There is no fallback:
if the library is missing or a call fails, a ``RuntimeError`` is raised.

Calls (see ``include/bwattn.h`` for the full contract):

* ``attn_fwd(q, k, v, causal, scale, window=0)``: prefill / cross attention, q [B, Hq, Nq, d],
  k, v [B, Hkv, Nk, d]; bf16 (tcgen05 kernel) or fp32 (fp32 FMA kernel); ``window`` > 0 adds a
  causal sliding window.
* ``attn_fwd_host(...)``: the same prefill from host tensors, with the copies overlapping the
  kernels (workspace from ``fwd_host_workspace_size``).
* ``attn_decode(q, kcache, vcache, nk, num_splits)``: single-query split-K decode,
  q [B, Hq, d], caches [B, Hkv, cap, d] bf16, nk [B] int32 on the device;
  ``attn_decode_paged`` over a paged cache and a block table; ``attn_decode_fp8`` /
  ``attn_decode_paged_fp8`` over E4M3 caches with per-channel scales.
* ``attn_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k, causal)``:
  packed sequences, q [total_q, Hq, d], k, v [total_k, Hkv, d] bf16.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

__all__ = [
    "attn_fwd", "attn_fwd_host", "attn_decode", "attn_decode_paged", "attn_decode_fp8", "attn_decode_paged_fp8",
    "attn_varlen", "fwd_host_workspace_size", "decode_workspace_size", "varlen_workspace_size",
    "get_status", "clear_status", "set_wait_timeout_ns", "test_wait_timeout", "launch_count", "lib",
    "status_string", "BwattnError", "OK", "ERR_INVALID_ARG", "ERR_UNSUPPORTED", "ERR_CUDA", "ERR_TIMEOUT",
]

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT = 0, 1, 2, 3, 4
DTYPE_FP32, DTYPE_BF16 = 0, 1

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libbwattn.so")
_lock = threading.Lock()
_lib = None


class BwattnError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} (status {status})")


def lib() -> ctypes.CDLL:
    """The loaded C library; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"libbwattn.so not found at {LIB_PATH}; build it with "
                "`python -m exact_attention_flashattn_gb300.build` (needs nvcc for sm_103a)")
        L = ctypes.CDLL(LIB_PATH)
        vp, ci, cf, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        L.attn_fwd.argtypes = [vp, vp, vp, vp, vp] + [ci] * 7 + [cf, ci, vp]
        L.attn_fwd.restype = ci
        L.attn_fwd_window.argtypes = [vp, vp, vp, vp, vp] + [ci] * 7 + [cf, ci, vp]
        L.attn_fwd_window.restype = ci
        L.attn_fwd_host.argtypes = [vp, vp, vp, vp, vp] + [ci] * 7 + [cf, ci, vp, sz, vp]
        L.attn_fwd_host.restype = ci
        L.attn_fwd_host_workspace_size.argtypes = [ci] * 7
        L.attn_fwd_host_workspace_size.restype = sz
        L.attn_decode_workspace_size.argtypes = [ci, ci, ci, ci]
        L.attn_decode_workspace_size.restype = sz
        L.attn_decode.argtypes = [vp, vp, vp, vp, vp] + [ci] * 6 + [cf, vp, vp, sz, vp]
        L.attn_decode.restype = ci
        L.attn_decode_paged.argtypes = [vp] * 6 + [ci] * 8 + [cf, vp, vp, sz, vp]
        L.attn_decode_fp8.argtypes = [vp] * 7 + [ci] * 6 + [cf, vp, vp, sz, vp]
        L.attn_decode_paged_fp8.argtypes = [vp] * 8 + [ci] * 8 + [cf, vp, vp, sz, vp]
        L.attn_decode_paged.restype = ci
        L.attn_varlen_workspace_size.argtypes = [ci] * 5
        L.attn_varlen_workspace_size.restype = sz
        L.attn_varlen.argtypes = [vp] * 7 + [ci] * 9 + [cf, vp, sz, vp]
        L.attn_varlen.restype = ci
        L.attn_varlen_window.argtypes = [vp] * 7 + [ci] * 9 + [cf, vp, sz, vp]
        L.attn_varlen_window.restype = ci
        L.bwattn_last_cuda_error.argtypes = []
        L.bwattn_last_cuda_error.restype = ci
        L.bwattn_status_string.argtypes = [ci]
        L.bwattn_status_string.restype = ctypes.c_char_p
        L.bwattn_get_status.argtypes = [vp]
        L.bwattn_get_status.restype = ci
        L.bwattn_clear_status.argtypes = [vp]
        L.bwattn_clear_status.restype = ci
        L.bwattn_set_wait_timeout_ns.argtypes = [ctypes.c_uint64]
        L.bwattn_set_wait_timeout_ns.restype = None
        L.bwattn_test_wait_timeout.argtypes = [vp]
        L.bwattn_test_wait_timeout.restype = ci
        L.bwattn_launch_count.argtypes = []
        L.bwattn_launch_count.restype = ctypes.c_uint64
        L.bwattn_version.argtypes = []
        L.bwattn_version.restype = ci
        _lib = L
        return L


def status_string(status: int) -> str:
    try:
        return lib().bwattn_status_string(int(status)).decode()
    except Exception:  # pragma: no cover - only when the library itself is missing
        return "unknown"


def _check(rc: int, what: str):
    if rc != OK:
        if rc == ERR_CUDA:
            err = lib().bwattn_last_cuda_error()
            raise BwattnError(rc, f"{what} (cudaError {err})")
        raise BwattnError(rc, what)


def _stream(stream=None) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def _ptr(t) -> int | None:
    return None if t is None else int(t.data_ptr())


def _cuda(t: torch.Tensor, name: str, dtype=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")


def _scale(scale, d):
    return (1.0 / math.sqrt(d)) if scale is None else float(scale)


def attn_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, causal: bool = True, scale: float | None = None,
             out: torch.Tensor | None = None, lse: torch.Tensor | bool | None = True, stream=None, window: int = 0):
    """Prefill / cross attention. q [B, Hq, Nq, d]; k, v [B, Hkv, Nk, d] -> (o, lse or None).

    ``window`` > 0 (causal only): sliding window of that many keys ending at each query's limit."""
    if window and not causal:
        raise ValueError("a sliding window needs causal=True")
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be 4-D [B, H, N, d]")
    B, Hq, Nq, d = q.shape
    Bk, Hkv, Nk, dk = k.shape
    if Bk != B or dk != d or tuple(v.shape) != tuple(k.shape):
        raise ValueError("k and v must be [B, Hkv, Nk, d] with q's B and d")
    if q.dtype == torch.bfloat16:
        dt = DTYPE_BF16
    elif q.dtype == torch.float32:
        dt = DTYPE_FP32
    else:
        raise ValueError(f"unsupported dtype {q.dtype}")
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _cuda(t, n, q.dtype)
    if out is None:
        out = torch.empty_like(q)
    _cuda(out, "out", q.dtype)
    lse_t = None
    if lse is True:
        lse_t = torch.empty((B, Hq, Nq), dtype=torch.float32, device=q.device)
    elif isinstance(lse, torch.Tensor):
        lse_t = lse
        _cuda(lse_t, "lse", torch.float32)
    if window:
        rc = lib().attn_fwd_window(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse_t), B, Hq, Hkv, Nq, Nk, d,
                                   int(window), _scale(scale, d), dt, _stream(stream))
        _check(rc, "attn_fwd_window")
        return out, lse_t
    rc = lib().attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse_t), B, Hq, Hkv, Nq, Nk, d, int(bool(causal)),
                        _scale(scale, d), dt, _stream(stream))
    _check(rc, "attn_fwd")
    return out, lse_t


def fwd_host_workspace_size(B: int, Hq: int, Hkv: int, Nq: int, Nk: int, d: int, dtype=torch.bfloat16) -> int:
    dt = DTYPE_BF16 if dtype == torch.bfloat16 else DTYPE_FP32
    return int(lib().attn_fwd_host_workspace_size(B, Hq, Hkv, Nq, Nk, d, dt))


def attn_fwd_host(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, causal: bool = True, scale: float | None = None,
                  out: torch.Tensor | None = None, lse: torch.Tensor | bool | None = True,
                  workspace: torch.Tensor | None = None, stream=None, device=None):
    """attn_fwd on host (CPU) tensors, copies included; pinned memory lets them overlap the kernels.
    The call is asynchronous on ``stream`` (the current stream of ``device`` by default): read
    ``out`` after synchronising it."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        if not isinstance(t, torch.Tensor) or t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous host tensor")
    if q.dim() != 4 or k.dim() != 4 or tuple(v.shape) != tuple(k.shape):
        raise ValueError("q [B, Hq, Nq, d]; k, v [B, Hkv, Nk, d]")
    B, Hq, Nq, d = q.shape
    _, Hkv, Nk, _ = k.shape
    if q.dtype not in (torch.bfloat16, torch.float32) or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("q, k, v must all be bf16 or all fp32")
    dt = DTYPE_BF16 if q.dtype == torch.bfloat16 else DTYPE_FP32
    if out is None:
        out = torch.empty_like(q, pin_memory=q.is_pinned())
    if out.is_cuda or out.dtype != q.dtype or tuple(out.shape) != tuple(q.shape) or not out.is_contiguous():
        raise ValueError("out must be a contiguous host tensor like q")
    lse_t = None
    if lse is True:
        lse_t = torch.empty((B, Hq, Nq), dtype=torch.float32, pin_memory=q.is_pinned())
    elif isinstance(lse, torch.Tensor):
        lse_t = lse
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    need = int(lib().attn_fwd_host_workspace_size(B, Hq, Hkv, Nq, Nk, d, dt))
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    _cuda(workspace, "workspace")
    with torch.cuda.device(dev):
        rc = lib().attn_fwd_host(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse_t), B, Hq, Hkv, Nq, Nk, d,
                                 int(bool(causal)), _scale(scale, d), dt, _ptr(workspace),
                                 workspace.numel() * workspace.element_size(), _stream(stream))
    _check(rc, "attn_fwd_host")
    return out, lse_t


def decode_workspace_size(B: int, Hq: int, d: int, num_splits: int) -> int:
    return int(lib().attn_decode_workspace_size(B, Hq, d, num_splits))


def attn_decode(q: torch.Tensor, kcache: torch.Tensor, vcache: torch.Tensor, nk: torch.Tensor, num_splits: int,
                scale: float | None = None, workspace: torch.Tensor | None = None, out: torch.Tensor | None = None,
                lse: torch.Tensor | bool | None = True, stream=None):
    """Single-query decode. q [B, Hq, d]; caches [B, Hkv, cap, d]; nk [B] int32 (device)."""
    if q.dim() != 3 or kcache.dim() != 4:
        raise ValueError("q must be [B, Hq, d] and caches [B, Hkv, cap, d]")
    B, Hq, d = q.shape
    Bk, Hkv, cap, dk = kcache.shape
    if Bk != B or dk != d or tuple(vcache.shape) != tuple(kcache.shape):
        raise ValueError("kcache and vcache must be [B, Hkv, cap, d] with q's B and d")
    for t, n in ((q, "q"), (kcache, "kcache"), (vcache, "vcache")):
        _cuda(t, n, torch.bfloat16)
    _cuda(nk, "nk", torch.int32)
    if out is None:
        out = torch.empty_like(q)
    _cuda(out, "out", torch.bfloat16)
    lse_t = None
    if lse is True:
        lse_t = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    elif isinstance(lse, torch.Tensor):
        lse_t = lse
        _cuda(lse_t, "lse", torch.float32)
    need = decode_workspace_size(B, Hq, d, num_splits)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    _cuda(workspace, "workspace")
    rc = lib().attn_decode(_ptr(q), _ptr(kcache), _ptr(vcache), _ptr(out), _ptr(nk), B, Hq, Hkv, cap, d,
                           int(num_splits), _scale(scale, d), _ptr(lse_t), _ptr(workspace),
                           workspace.numel() * workspace.element_size(), _stream(stream))
    _check(rc, "attn_decode")
    return out, lse_t


def attn_decode_paged(q: torch.Tensor, k_pages: torch.Tensor, v_pages: torch.Tensor, block_table: torch.Tensor,
                      nk: torch.Tensor, num_splits: int, scale: float | None = None,
                      workspace: torch.Tensor | None = None, out: torch.Tensor | None = None,
                      lse: torch.Tensor | bool | None = True, stream=None):
    """Paged decode. q [B, Hq, d]; pages [num_pages, page_size, Hkv, d]; block_table [B, max_pages]
    int32 and nk [B] int32 on the device."""
    if q.dim() != 3 or k_pages.dim() != 4 or block_table.dim() != 2:
        raise ValueError("q must be [B, Hq, d], pages [num_pages, page_size, Hkv, d], block_table [B, max_pages]")
    B, Hq, d = q.shape
    num_pages, page_size, Hkv, dk = k_pages.shape
    if dk != d or tuple(v_pages.shape) != tuple(k_pages.shape) or block_table.shape[0] != B:
        raise ValueError("k_pages and v_pages must be [num_pages, page_size, Hkv, d]; block_table [B, max_pages]")
    for t, n in ((q, "q"), (k_pages, "k_pages"), (v_pages, "v_pages")):
        _cuda(t, n, torch.bfloat16)
    _cuda(block_table, "block_table", torch.int32)
    _cuda(nk, "nk", torch.int32)
    if out is None:
        out = torch.empty_like(q)
    _cuda(out, "out", torch.bfloat16)
    lse_t = None
    if lse is True:
        lse_t = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    elif isinstance(lse, torch.Tensor):
        lse_t = lse
        _cuda(lse_t, "lse", torch.float32)
    need = decode_workspace_size(B, Hq, d, num_splits)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    _cuda(workspace, "workspace")
    rc = lib().attn_decode_paged(_ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(out), _ptr(block_table), _ptr(nk), B, Hq,
                                 Hkv, page_size, num_pages, block_table.shape[1], d, int(num_splits), _scale(scale, d),
                                 _ptr(lse_t), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                 _stream(stream))
    _check(rc, "attn_decode_paged")
    return out, lse_t


_FP8_CODES = (torch.uint8, torch.float8_e4m3fn)


def _fp8_cache(k, v, k_scale, v_scale, Hkv, d, names):
    for t, n in ((k, names[0]), (v, names[1])):
        _cuda(t, n)
        if t.dtype not in _FP8_CODES:
            raise ValueError(f"{n} must hold E4M3 codes (uint8 or float8_e4m3fn), got {t.dtype}")
    for t, n in ((k_scale, "k_scale"), (v_scale, "v_scale")):
        _cuda(t, n, torch.float32)
        if tuple(t.shape) != (Hkv, d):
            raise ValueError(f"{n} must be [Hkv, d] = [{Hkv}, {d}]")


def _decode_outputs(q, B, Hq, d, num_splits, out, lse, workspace):
    if out is None:
        out = torch.empty_like(q)
    _cuda(out, "out", torch.bfloat16)
    lse_t = None
    if lse is True:
        lse_t = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    elif isinstance(lse, torch.Tensor):
        lse_t = lse
        _cuda(lse_t, "lse", torch.float32)
    need = decode_workspace_size(B, Hq, d, num_splits)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    _cuda(workspace, "workspace")
    return out, lse_t, workspace


def attn_decode_fp8(q: torch.Tensor, kcache: torch.Tensor, vcache: torch.Tensor, k_scale: torch.Tensor,
                    v_scale: torch.Tensor, nk: torch.Tensor, num_splits: int, scale: float | None = None,
                    workspace: torch.Tensor | None = None, out: torch.Tensor | None = None,
                    lse: torch.Tensor | bool | None = True, stream=None):
    """Decode against an FP8 cache. q [B, Hq, d] bf16; caches [B, Hkv, cap, d] of E4M3 codes;
    k_scale, v_scale [Hkv, d] fp32 (value = e4m3(code) * scale[head, channel]); nk [B] int32."""
    if q.dim() != 3 or kcache.dim() != 4:
        raise ValueError("q must be [B, Hq, d] and caches [B, Hkv, cap, d]")
    B, Hq, d = q.shape
    Bk, Hkv, cap, dk = kcache.shape
    if Bk != B or dk != d or tuple(vcache.shape) != tuple(kcache.shape):
        raise ValueError("kcache and vcache must be [B, Hkv, cap, d] with q's B and d")
    _cuda(q, "q", torch.bfloat16)
    _fp8_cache(kcache, vcache, k_scale, v_scale, Hkv, d, ("kcache", "vcache"))
    _cuda(nk, "nk", torch.int32)
    out, lse_t, workspace = _decode_outputs(q, B, Hq, d, num_splits, out, lse, workspace)
    rc = lib().attn_decode_fp8(_ptr(q), _ptr(kcache), _ptr(vcache), _ptr(k_scale), _ptr(v_scale), _ptr(out), _ptr(nk),
                               B, Hq, Hkv, cap, d, int(num_splits), _scale(scale, d), _ptr(lse_t), _ptr(workspace),
                               workspace.numel() * workspace.element_size(), _stream(stream))
    _check(rc, "attn_decode_fp8")
    return out, lse_t


def attn_decode_paged_fp8(q: torch.Tensor, k_pages: torch.Tensor, v_pages: torch.Tensor, k_scale: torch.Tensor,
                          v_scale: torch.Tensor, block_table: torch.Tensor, nk: torch.Tensor, num_splits: int,
                          scale: float | None = None, workspace: torch.Tensor | None = None,
                          out: torch.Tensor | None = None, lse: torch.Tensor | bool | None = True, stream=None):
    """Paged decode against FP8 pages [num_pages, page_size, Hkv, d] of E4M3 codes."""
    if q.dim() != 3 or k_pages.dim() != 4 or block_table.dim() != 2:
        raise ValueError("q must be [B, Hq, d], pages [num_pages, page_size, Hkv, d], block_table [B, max_pages]")
    B, Hq, d = q.shape
    num_pages, page_size, Hkv, dk = k_pages.shape
    if dk != d or tuple(v_pages.shape) != tuple(k_pages.shape) or block_table.shape[0] != B:
        raise ValueError("k_pages and v_pages must be [num_pages, page_size, Hkv, d]; block_table [B, max_pages]")
    _cuda(q, "q", torch.bfloat16)
    _fp8_cache(k_pages, v_pages, k_scale, v_scale, Hkv, d, ("k_pages", "v_pages"))
    _cuda(block_table, "block_table", torch.int32)
    _cuda(nk, "nk", torch.int32)
    out, lse_t, workspace = _decode_outputs(q, B, Hq, d, num_splits, out, lse, workspace)
    rc = lib().attn_decode_paged_fp8(_ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(k_scale), _ptr(v_scale), _ptr(out),
                                     _ptr(block_table), _ptr(nk), B, Hq, Hkv, page_size, num_pages,
                                     block_table.shape[1], d, int(num_splits), _scale(scale, d), _ptr(lse_t),
                                     _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream))
    _check(rc, "attn_decode_paged_fp8")
    return out, lse_t


def varlen_workspace_size(num_seqs: int, max_seqlen_k: int, Hq: int, Hkv: int, d: int) -> int:
    return int(lib().attn_varlen_workspace_size(num_seqs, max_seqlen_k, Hq, Hkv, d))


def attn_varlen(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, cu_seqlens_q: torch.Tensor,
                cu_seqlens_k: torch.Tensor, max_seqlen_q: int, max_seqlen_k: int, causal: bool = True,
                scale: float | None = None, workspace: torch.Tensor | None = None, out: torch.Tensor | None = None,
                lse: torch.Tensor | bool | None = True, stream=None, window: int = 0):
    """Packed varlen. q [total_q, Hq, d]; k, v [total_k, Hkv, d]; cu_seqlens int32 [num_seqs + 1] (device).

    ``window`` > 0 (causal only): sliding window of that many keys ending at each query's limit."""
    if window and not causal:
        raise ValueError("a sliding window needs causal=True")
    if q.dim() != 3 or k.dim() != 3:
        raise ValueError("q must be [total_q, Hq, d] and k, v [total_k, Hkv, d]")
    tq, Hq, d = q.shape
    tk, Hkv, dk = k.shape
    if dk != d or tuple(v.shape) != tuple(k.shape):
        raise ValueError("k and v must be [total_k, Hkv, d] with q's d")
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _cuda(t, n, torch.bfloat16)
    _cuda(cu_seqlens_q, "cu_seqlens_q", torch.int32)
    _cuda(cu_seqlens_k, "cu_seqlens_k", torch.int32)
    num_seqs = cu_seqlens_q.numel() - 1
    if cu_seqlens_k.numel() != num_seqs + 1:
        raise ValueError("cu_seqlens_q and cu_seqlens_k must have the same length")
    if out is None:
        out = torch.empty_like(q)
    _cuda(out, "out", torch.bfloat16)
    lse_t = None
    if lse is True:
        lse_t = torch.empty((tq, Hq), dtype=torch.float32, device=q.device)
    elif isinstance(lse, torch.Tensor):
        lse_t = lse
        _cuda(lse_t, "lse", torch.float32)
    need = varlen_workspace_size(num_seqs, int(max_seqlen_k), Hq, Hkv, d)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    _cuda(workspace, "workspace")
    if window:
        fn, mode, what = lib().attn_varlen_window, int(window), "attn_varlen_window"
    else:
        fn, mode, what = lib().attn_varlen, int(bool(causal)), "attn_varlen"
    rc = fn(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse_t), _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), num_seqs, tq,
            tk, int(max_seqlen_q), int(max_seqlen_k), Hq, Hkv, d, mode, _scale(scale, d), _ptr(workspace),
            workspace.numel() * workspace.element_size(), _stream(stream))
    _check(rc, what)
    return out, lse_t


def get_status(stream=None) -> int:
    """Synchronises the stream; BWATTN_ERR_TIMEOUT if a kernel gave up a wait, else OK."""
    return int(lib().bwattn_get_status(_stream(stream)))


def clear_status(stream=None) -> None:
    _check(lib().bwattn_clear_status(_stream(stream)), "bwattn_clear_status")


def set_wait_timeout_ns(ns: int) -> None:
    lib().bwattn_set_wait_timeout_ns(int(ns))


def test_wait_timeout(stream=None) -> None:
    _check(lib().bwattn_test_wait_timeout(_stream(stream)), "bwattn_test_wait_timeout")


def launch_count() -> int:
    return int(lib().bwattn_launch_count())
