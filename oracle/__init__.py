"""Exact-attention oracle: a plain, slow fp64 CPU implementation.

TEST INFRASTRUCTURE ONLY. The product path (``exact_attention_flashattn_gb300`` and its
CUDA library) never imports, links or calls anything here; only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` do.

The arithmetic lives in ``attention_oracle.cpp`` (IEEE double, no fast-math); this module
compiles it with the host C++ compiler and wraps it with ctypes. Every function takes and
returns numpy float64 arrays. Sources, by page title and section:

* naive: "Attention kernels" (llm-inference-explained), Concept, Algorithm 0; "Attention
  Computation in Practice", section 4 (naive form); safe softmax from "Attention from the
  kernel's side", The online softmax.
* tiled: the online-softmax recurrence, "Attention from the kernel's side", The online
  softmax; "Attention kernels", Maths (first display).
* split-K + merge: "Attention kernels", Maths (second display) and Concept (Split-K);
  "Attention from the kernel's side", Flash-decoding.
* GQA by index: "Attention Computation in Practice", GQA in the kernel.
* varlen: "Attention Computation in Practice", the four attention kernels (APPEND / MIXED).
* FP8 KV cache: E4M3 codes times a per-(KV head, channel) scale, decoded from the format's
  definition ("Attention from the kernel's side", Why a quantised cache needs a fused kernel).

Parity pins for every function live in ``tests/test_oracle_pins.py``; none is unpinned.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attention_oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

METHOD_NAIVE = 0
METHOD_TILED = 1
METHOD_SPLITK = 2


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/liboracle.so`` (host code, no GPU)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    cxx = os.environ.get("CXX", "g++")
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = [cxx, "-O2", "-std=c++17", "-fPIC", "-shared", "-pthread", "-fno-fast-math",
           "-ffp-contract=off", _SRC, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB)
        D = ctypes.POINTER(ctypes.c_double)
        I32 = ctypes.POINTER(ctypes.c_int32)
        c_int, c_double = ctypes.c_int, ctypes.c_double
        lib.oracle_attention.argtypes = [D, D, D, D, D] + [c_int] * 7 + [c_double] + [c_int] * 4
        lib.oracle_decode.argtypes = [D, D, D, I32, D, D] + [c_int] * 5 + [c_double] + [c_int] * 3
        lib.oracle_varlen.argtypes = [D, D, D, I32, I32, D, D] + [c_int] * 5 + [c_double] + [c_int] * 4
        lib.oracle_probs.argtypes = [D, D, D, c_int, c_int, c_int, c_int, c_double]
        lib.oracle_partials.argtypes = [D, D, D, c_int, c_int, c_double, c_int, D, D, D]
        lib.oracle_merge.argtypes = [c_double, c_double, D, c_double, c_double, D, c_int, D, D, D]
        lib.oracle_hardware_threads.argtypes = []
        lib.oracle_e4m3_decode.argtypes = [ctypes.c_void_p, ctypes.c_int64, D]
        for f in ("oracle_attention", "oracle_decode", "oracle_varlen", "oracle_probs",
                  "oracle_partials", "oracle_merge", "oracle_hardware_threads", "oracle_e4m3_decode"):
            getattr(lib, f).restype = c_int
        _lib = lib
        return lib


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _dp(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _ip(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


def _method(method: str, block: int | None, workers: int | None) -> tuple[int, int]:
    if method == "naive":
        return METHOD_NAIVE, 0
    if method == "tiled":
        return METHOD_TILED, int(block if block is not None else 128)
    if method == "splitk":
        return METHOD_SPLITK, int(workers if workers is not None else 1)
    raise ValueError(f"unknown oracle method {method!r}")


def hardware_threads() -> int:
    return int(_load().oracle_hardware_threads())


def attention(q, k, v, causal: bool, scale: float | None = None, method: str = "tiled",
              block: int | None = None, workers: int | None = None, nthreads: int = 0, window: int = 0):
    """Dense layout: q [B, Hq, Nq, d]; k, v [B, Hkv, Nk, d] -> (o [B, Hq, Nq, d], lse [B, Hq, Nq]).

    Causal masking is aligned to the end of the key sequence when Nq != Nk. ``window`` > 0 adds a
    sliding window ("Attention Computation in Practice", Masking variants): query i sees keys
    i' - window < j <= i' with i' = i + (Nk - Nq).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, Hq, Nq, d = q.shape
    _, Hkv, Nk, _ = k.shape
    if scale is None:
        scale = 1.0 / float(np.sqrt(d))
    o = np.zeros((B, Hq, Nq, d), dtype=np.float64)
    lse = np.zeros((B, Hq, Nq), dtype=np.float64)
    m, p = _method(method, block, workers)
    rc = _load().oracle_attention(_dp(q), _dp(k), _dp(v), _dp(o), _dp(lse), B, Hq, Hkv, Nq, Nk, d,
                                  int(bool(causal)), float(scale), m, p, int(nthreads), int(window))
    if rc != 0:
        raise ValueError(f"oracle_attention rejected its arguments (rc={rc})")
    return o, lse


def decode(q, kcache, vcache, nk, scale: float | None = None, method: str = "splitk",
           workers: int | None = None, block: int | None = None, nthreads: int = 0):
    """q [B, Hq, d]; caches [B, Hkv, cap, d]; nk [B] -> (o [B, Hq, d], lse [B, Hq])."""
    q, kc, vc, nk = _f64(q), _f64(kcache), _f64(vcache), _i32(nk)
    B, Hq, d = q.shape
    _, Hkv, cap, _ = kc.shape
    if scale is None:
        scale = 1.0 / float(np.sqrt(d))
    o = np.zeros((B, Hq, d), dtype=np.float64)
    lse = np.zeros((B, Hq), dtype=np.float64)
    m, p = _method(method, block, workers)
    rc = _load().oracle_decode(_dp(q), _dp(kc), _dp(vc), _ip(nk), _dp(o), _dp(lse), B, Hq, Hkv, cap, d,
                               float(scale), m, p, int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle_decode rejected its arguments (rc={rc})")
    return o, lse


def decode_paged(q, k_pages, v_pages, block_table, nk, scale: float | None = None, method: str = "splitk",
                 workers: int | None = None, block: int | None = None, nthreads: int = 0):
    """Paged decode ("Attention Computation in Practice", PagedAttention's kernel difference):
    pages [num_pages, page_size, Hkv, d], block_table [B, max_pages]. Key j of sequence b is row
    j % page_size of page block_table[b][j // page_size]; the keys are gathered into contiguous
    caches [B, Hkv, max_pages * page_size, d] (data movement only) and passed to ``decode``."""
    kp, vp = _f64(k_pages), _f64(v_pages)
    table = np.asarray(block_table, dtype=np.int64)
    num_pages, ps, Hkv, d = kp.shape
    B, mp = table.shape
    kc = kp[table].reshape(B, mp * ps, Hkv, d).transpose(0, 2, 1, 3)
    vc = vp[table].reshape(B, mp * ps, Hkv, d).transpose(0, 2, 1, 3)
    return decode(q, kc, vc, nk, scale=scale, method=method, workers=workers, block=block, nthreads=nthreads)


def e4m3_decode(codes) -> np.ndarray:
    """FP8 E4M3 codes (uint8, any shape) -> float64 values of the same shape."""
    x = np.ascontiguousarray(np.asarray(codes, dtype=np.uint8))
    out = np.empty(x.shape, dtype=np.float64)
    rc = _load().oracle_e4m3_decode(x.ctypes.data_as(ctypes.c_void_p), int(x.size), _dp(out))
    if rc != 0:
        raise ValueError("oracle_e4m3_decode rejected its arguments")
    return out


def decode_fp8(q, k_codes, v_codes, k_scale, v_scale, nk, scale: float | None = None, method: str = "splitk",
               workers: int | None = None, block: int | None = None, nthreads: int = 0):
    """Decode against an FP8 KV cache: caches [B, Hkv, cap, d] of E4M3 codes (uint8), scales
    [Hkv, d]; the cached value is e4m3(code) * scale[head, channel] ("Attention from the
    kernel's side", Why a quantised cache needs a fused kernel). The caches are decoded to
    float64 and passed to ``decode``."""
    kq, vq = np.asarray(k_codes, dtype=np.uint8), np.asarray(v_codes, dtype=np.uint8)
    ks, vs = _f64(k_scale), _f64(v_scale)
    B, Hkv, cap, d = kq.shape
    if ks.shape != (Hkv, d) or vs.shape != (Hkv, d) or vq.shape != kq.shape:
        raise ValueError("k/v codes [B, Hkv, cap, d] and scales [Hkv, d] expected")
    kc = e4m3_decode(kq) * ks[None, :, None, :]
    vc = e4m3_decode(vq) * vs[None, :, None, :]
    return decode(q, kc, vc, nk, scale=scale, method=method, workers=workers, block=block, nthreads=nthreads)


def varlen(q, k, v, cu_q, cu_k, causal: bool, scale: float | None = None, method: str = "tiled",
           block: int | None = None, workers: int | None = None, nthreads: int = 0, window: int = 0):
    """Packed: q [total_q, Hq, d]; k, v [total_k, Hkv, d] -> (o [total_q, Hq, d], lse [total_q, Hq])."""
    q, k, v, cu_q, cu_k = _f64(q), _f64(k), _f64(v), _i32(cu_q), _i32(cu_k)
    tq, Hq, d = q.shape
    _, Hkv, _ = k.shape
    if scale is None:
        scale = 1.0 / float(np.sqrt(d))
    o = np.zeros((tq, Hq, d), dtype=np.float64)
    lse = np.zeros((tq, Hq), dtype=np.float64)
    m, p = _method(method, block, workers)
    rc = _load().oracle_varlen(_dp(q), _dp(k), _dp(v), _ip(cu_q), _ip(cu_k), _dp(o), _dp(lse),
                               len(cu_q) - 1, Hq, Hkv, d, int(bool(causal)), float(scale), m, p,
                               int(nthreads), int(window))
    if rc != 0:
        raise ValueError(f"oracle_varlen rejected its arguments (rc={rc})")
    return o, lse


def probs(q, k, causal: bool, scale: float | None = None) -> np.ndarray:
    """Softmax matrix of the naive path for one head: q [Nq, d], k [Nk, d] -> P [Nq, Nk]."""
    q, k = _f64(q), _f64(k)
    Nq, d = q.shape
    Nk = k.shape[0]
    if scale is None:
        scale = 1.0 / float(np.sqrt(d))
    p = np.zeros((Nq, Nk), dtype=np.float64)
    rc = _load().oracle_probs(_dp(q), _dp(k), _dp(p), Nq, Nk, d, int(bool(causal)), float(scale))
    if rc != 0:
        raise ValueError("oracle_probs rejected its arguments")
    return p


def partials(q, k, v, workers: int, scale: float | None = None):
    """Split-K partial states of one query q [d] over keys k, v [n, d]: (m [W], l [W], o [W, d])."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    n, d = k.shape
    if scale is None:
        scale = 1.0 / float(np.sqrt(d))
    m = np.zeros(workers)
    l = np.zeros(workers)
    o = np.zeros((workers, d))
    rc = _load().oracle_partials(_dp(q), _dp(k), _dp(v), n, d, float(scale), int(workers), _dp(m), _dp(l),
                                 _dp(o))
    if rc != 0:
        raise ValueError("oracle_partials rejected its arguments")
    return m, l, o


def merge(ma: float, la: float, oa, mb: float, lb: float, ob):
    """Two-state merge of partial (m, l, o) states -> (m, l, o)."""
    oa, ob = _f64(oa), _f64(ob)
    d = oa.shape[0]
    m = ctypes.c_double()
    l = ctypes.c_double()
    o = np.zeros(d)
    rc = _load().oracle_merge(float(ma), float(la), _dp(oa), float(mb), float(lb), _dp(ob), d,
                              ctypes.byref(m), ctypes.byref(l), _dp(o))
    if rc != 0:
        raise ValueError("oracle_merge rejected its arguments")
    return m.value, l.value, o
