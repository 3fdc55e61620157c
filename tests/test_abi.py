"""The C-ABI library loads, exports every symbol include/bwattn.h declares, and rejects bad
arguments on the host before any CUDA call (so these run without a GPU)."""
import ctypes
import os
import re

import pytest

import exact_attention_flashattn_gb300 as bw
from exact_attention_flashattn_gb300 import build as bw_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "bwattn.h")


@pytest.fixture(scope="module")
def L():
    bw_build.build()
    return bw.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:[A-Za-z_][\w\s\*]*?)\b([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "defined")))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("attn_fwd", "attn_fwd_window", "attn_fwd_host", "attn_fwd_host_workspace_size", "attn_decode", "attn_decode_paged", "attn_decode_fp8",
              "attn_decode_paged_fp8", "attn_varlen", "attn_varlen_window",
              "attn_decode_workspace_size", "attn_varlen_workspace_size",
              "bwattn_get_status", "bwattn_clear_status", "bwattn_last_cuda_error", "bwattn_status_string",
              "bwattn_set_wait_timeout_ns", "bwattn_test_wait_timeout", "bwattn_launch_count", "bwattn_version"):
        assert n in names


def test_every_declared_symbol_is_exported(L):
    for n in declared_functions():
        assert hasattr(L, n), n


def test_version_and_strings(L):
    assert L.bwattn_version() >= 100
    assert bw.status_string(bw.OK) == "ok"
    assert "invalid" in bw.status_string(bw.ERR_INVALID_ARG)


FAKE = 0x10000  # 16-byte aligned, never dereferenced: validation fails before any CUDA call


def fwd(L, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=None, B=1, Hq=2, Hkv=1, Nq=8, Nk=8, d=128, causal=1, scale=0.1,
             dtype=bw.DTYPE_BF16, stream=None)
    a.update(kw)
    return L.attn_fwd(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["Hq"], a["Hkv"], a["Nq"], a["Nk"], a["d"],
                      a["causal"], a["scale"], a["dtype"], a["stream"])


def test_fwd_argument_errors(L):
    assert fwd(L, q=None) == bw.ERR_INVALID_ARG
    assert fwd(L, o=None) == bw.ERR_INVALID_ARG
    assert fwd(L, Hq=3, Hkv=2) == bw.ERR_INVALID_ARG
    assert fwd(L, Nq=-1) == bw.ERR_INVALID_ARG
    assert fwd(L, scale=0.0) == bw.ERR_INVALID_ARG
    assert fwd(L, scale=float("nan")) == bw.ERR_INVALID_ARG
    assert fwd(L, causal=2) == bw.ERR_INVALID_ARG
    assert fwd(L, q=FAKE + 8) == bw.ERR_INVALID_ARG  # misaligned
    assert fwd(L, lse=FAKE + 2) == bw.ERR_INVALID_ARG
    assert fwd(L, d=96) == bw.ERR_UNSUPPORTED
    assert fwd(L, dtype=7) == bw.ERR_UNSUPPORTED
    assert fwd(L, d=256, B=0) == bw.OK  # bf16 at d = 256: the tcgen05 kernel's d = 256 instance
    assert fwd(L, d=256, dtype=bw.DTYPE_FP32) == bw.ERR_UNSUPPORTED  # the fp32 FMA kernel stops at 128
    # empty work is a valid no-op that touches nothing
    assert fwd(L, B=0, q=None, k=None, v=None, o=None) == bw.OK
    assert fwd(L, Nq=0, q=None, k=None, v=None, o=None) == bw.OK


def dec(L, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, nk=FAKE, B=2, Hq=8, Hkv=2, cap=64, d=128, S=4, scale=0.1, lse=None,
             ws=FAKE, wsb=1 << 30, stream=None)
    a.update(kw)
    return L.attn_decode(a["q"], a["k"], a["v"], a["o"], a["nk"], a["B"], a["Hq"], a["Hkv"], a["cap"], a["d"], a["S"],
                         a["scale"], a["lse"], a["ws"], a["wsb"], a["stream"])


def test_decode_argument_errors(L):
    need = L.attn_decode_workspace_size(2, 8, 128, 4)
    assert need >= 2 * 8 * 4 * 130 * 4
    assert dec(L, nk=None) == bw.ERR_INVALID_ARG
    assert dec(L, ws=None) == bw.ERR_INVALID_ARG
    assert dec(L, wsb=need - 1) == bw.ERR_INVALID_ARG
    assert dec(L, S=0) == bw.ERR_INVALID_ARG
    assert dec(L, S=1025) == bw.ERR_INVALID_ARG
    assert dec(L, Hq=8, Hkv=3) == bw.ERR_INVALID_ARG
    assert dec(L, d=96) == bw.ERR_UNSUPPORTED
    # d = 64 is accepted: its workspace is sized for 64 channels and checked against that
    need64 = L.attn_decode_workspace_size(2, 8, 64, 4)
    assert 0 < need64 < need
    assert dec(L, d=64, wsb=need64 - 1) == bw.ERR_INVALID_ARG
    assert dec(L, d=64, B=0, q=None) == bw.OK
    # d = 256 likewise (bf16 caches; the FP8 cache stays d = 128)
    need256 = L.attn_decode_workspace_size(2, 8, 256, 4)
    assert need256 > need
    assert dec(L, d=256, wsb=need256 - 1) == bw.ERR_INVALID_ARG
    assert dec(L, d=256, B=0, q=None) == bw.OK
    assert dec(L, d=192) == bw.ERR_UNSUPPORTED
    assert dec(L, Hq=66, Hkv=1) == bw.ERR_UNSUPPORTED
    assert dec(L, nk=FAKE + 2) == bw.ERR_INVALID_ARG
    assert dec(L, B=0, q=None) == bw.OK


def test_varlen_argument_errors(L):
    def var(**kw):
        a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=None, cq=FAKE, ck=FAKE, n=3, tq=10, tk=30, mq=8, mk=16, Hq=8,
                 Hkv=2, d=128, causal=1, scale=0.1, ws=FAKE, wsb=1 << 30, stream=None)
        a.update(kw)
        return L.attn_varlen(a["q"], a["k"], a["v"], a["o"], a["lse"], a["cq"], a["ck"], a["n"], a["tq"], a["tk"],
                             a["mq"], a["mk"], a["Hq"], a["Hkv"], a["d"], a["causal"], a["scale"], a["ws"], a["wsb"],
                             a["stream"])
    assert var(cq=None) == bw.ERR_INVALID_ARG
    assert var(ws=None) == bw.ERR_INVALID_ARG
    assert var(wsb=16) == bw.ERR_INVALID_ARG
    assert var(Hq=8, Hkv=3) == bw.ERR_INVALID_ARG
    assert var(d=96) == bw.ERR_UNSUPPORTED
    assert var(d=64, wsb=16) == bw.ERR_INVALID_ARG
    assert var(d=64, n=0) == bw.OK
    assert var(n=0) == bw.OK
    assert L.attn_varlen_workspace_size(3, 16, 8, 2, 128) > 0


def test_window_argument_errors(L):
    def fw(window, **kw):
        a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=None, B=1, Hq=2, Hkv=1, Nq=8, Nk=8, d=128, scale=0.1,
                 dtype=bw.DTYPE_BF16, stream=None)
        a.update(kw)
        return L.attn_fwd_window(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["Hq"], a["Hkv"], a["Nq"],
                                 a["Nk"], a["d"], window, a["scale"], a["dtype"], a["stream"])

    def vw(window, **kw):
        a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=None, cq=FAKE, ck=FAKE, n=3, tq=10, tk=30, mq=8, mk=16, Hq=8,
                 Hkv=2, d=128, scale=0.1, ws=FAKE, wsb=1 << 30, stream=None)
        a.update(kw)
        return L.attn_varlen_window(a["q"], a["k"], a["v"], a["o"], a["lse"], a["cq"], a["ck"], a["n"], a["tq"],
                                    a["tk"], a["mq"], a["mk"], a["Hq"], a["Hkv"], a["d"], window, a["scale"], a["ws"],
                                    a["wsb"], a["stream"])
    for w in (0, -1, -(1 << 31)):
        assert fw(w) == bw.ERR_INVALID_ARG
        assert vw(w) == bw.ERR_INVALID_ARG
    assert fw(4, q=None) == bw.ERR_INVALID_ARG
    assert fw(4, d=96) == bw.ERR_UNSUPPORTED
    assert fw(4, B=0, q=None, k=None, v=None, o=None) == bw.OK
    assert vw(4, cq=None) == bw.ERR_INVALID_ARG
    assert vw(4, n=0) == bw.OK


def test_fp8_decode_argument_errors(L):
    def d8(**kw):
        a = dict(q=FAKE, k=FAKE, v=FAKE, ks=FAKE, vs=FAKE, o=FAKE, nk=FAKE, B=2, Hq=8, Hkv=2, cap=64, d=128, S=4,
                 scale=0.1, lse=None, ws=FAKE, wsb=1 << 30, stream=None)
        a.update(kw)
        return L.attn_decode_fp8(a["q"], a["k"], a["v"], a["ks"], a["vs"], a["o"], a["nk"], a["B"], a["Hq"], a["Hkv"],
                                 a["cap"], a["d"], a["S"], a["scale"], a["lse"], a["ws"], a["wsb"], a["stream"])

    def p8(**kw):
        a = dict(q=FAKE, k=FAKE, v=FAKE, ks=FAKE, vs=FAKE, o=FAKE, bt=FAKE, nk=FAKE, B=2, Hq=8, Hkv=2, ps=16, np_=8,
                 mp=4, d=128, S=4, scale=0.1, lse=None, ws=FAKE, wsb=1 << 30, stream=None)
        a.update(kw)
        return L.attn_decode_paged_fp8(a["q"], a["k"], a["v"], a["ks"], a["vs"], a["o"], a["bt"], a["nk"], a["B"],
                                       a["Hq"], a["Hkv"], a["ps"], a["np_"], a["mp"], a["d"], a["S"], a["scale"],
                                       a["lse"], a["ws"], a["wsb"], a["stream"])
    for f in (d8, p8):
        assert f(ks=None) == bw.ERR_INVALID_ARG
        assert f(vs=None) == bw.ERR_INVALID_ARG
        assert f(ks=FAKE + 4) == bw.ERR_INVALID_ARG  # scales are read as 16-byte vectors
        assert f(k=FAKE + 8) == bw.ERR_INVALID_ARG
        assert f(ws=None) == bw.ERR_INVALID_ARG
        assert f(d=64) == bw.ERR_UNSUPPORTED
        assert f(d=256) == bw.ERR_UNSUPPORTED
        assert f(Hq=8, Hkv=3) == bw.ERR_INVALID_ARG
        assert f(B=0, q=None) == bw.OK
    assert p8(ps=24) == bw.ERR_INVALID_ARG


def test_python_binding_fp8_checks():
    import torch
    q = torch.zeros(1, 2, 128)
    with pytest.raises(ValueError):
        bw.attn_decode_fp8(q, torch.zeros(1, 1, 4, 128, dtype=torch.uint8), torch.zeros(1, 1, 4, 128, dtype=torch.uint8),
                           torch.ones(1, 128), torch.ones(1, 128), torch.zeros(1, dtype=torch.int32), 1)


def test_fwd_host_argument_errors(L):
    HOSTP = 0x20000  # never dereferenced: validation fails (or the work is empty) before any copy

    def fh(**kw):
        a = dict(q=HOSTP, k=HOSTP, v=HOSTP, o=HOSTP, lse=None, B=2, Hq=4, Hkv=2, Nq=64, Nk=64, d=128, causal=1,
                 scale=0.1, dtype=bw.DTYPE_BF16, ws=0x40000, wsb=1 << 40, stream=None)
        a.update(kw)
        return L.attn_fwd_host(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["Hq"], a["Hkv"], a["Nq"], a["Nk"],
                               a["d"], a["causal"], a["scale"], a["dtype"], a["ws"], a["wsb"], a["stream"])
    need = L.attn_fwd_host_workspace_size(2, 4, 2, 64, 64, 128, bw.DTYPE_BF16)
    # two slots of (q, k, v, o, lse) for one chunk: units = 4, one unit per chunk
    assert need == 2 * (2 * 2 * 64 * 128 * 2 + 2 * 64 * 128 * 2 + 512)
    assert L.attn_fwd_host_workspace_size(2, 4, 3, 64, 64, 128, bw.DTYPE_BF16) == 0
    assert fh(ws=None) == bw.ERR_INVALID_ARG
    assert fh(ws=0x40000 + 16) == bw.ERR_INVALID_ARG  # 256-byte alignment
    assert fh(wsb=need - 1) == bw.ERR_INVALID_ARG
    assert fh(q=None) == bw.ERR_INVALID_ARG
    assert fh(d=96) == bw.ERR_UNSUPPORTED
    assert fh(dtype=7) == bw.ERR_UNSUPPORTED
    assert fh(scale=0.0) == bw.ERR_INVALID_ARG
    assert fh(causal=3) == bw.ERR_INVALID_ARG
    assert fh(B=0, q=None, k=None, v=None, o=None, ws=None) == bw.OK


def test_python_binding_rejects_window_without_causal():
    import torch
    q = torch.zeros(1, 1, 8, 64)
    with pytest.raises(ValueError):
        bw.attn_fwd(q, q, q, causal=False, window=4)


def test_python_binding_rejects_host_tensors():
    import torch
    q = torch.zeros(1, 1, 8, 64)
    with pytest.raises(ValueError):
        bw.attn_fwd(q, q, q)


def test_paged_decode_argument_errors(L):
    def pag(**kw):
        a = dict(q=FAKE, kp=FAKE, vp=FAKE, o=FAKE, table=FAKE, nk=FAKE, B=2, Hq=8, Hkv=2, ps=16, npages=64, mp=8,
                 d=128, S=4, scale=0.1, lse=None, ws=FAKE, wsb=1 << 30, stream=None)
        a.update(kw)
        return L.attn_decode_paged(a["q"], a["kp"], a["vp"], a["o"], a["table"], a["nk"], a["B"], a["Hq"], a["Hkv"],
                                   a["ps"], a["npages"], a["mp"], a["d"], a["S"], a["scale"], a["lse"], a["ws"],
                                   a["wsb"], a["stream"])
    assert pag(table=None) == bw.ERR_INVALID_ARG
    assert pag(ps=8) == bw.ERR_INVALID_ARG
    assert pag(ps=24) == bw.ERR_INVALID_ARG
    assert pag(npages=0) == bw.ERR_INVALID_ARG
    assert pag(table=FAKE + 2) == bw.ERR_INVALID_ARG
    assert pag(wsb=16) == bw.ERR_INVALID_ARG
    assert pag(d=96) == bw.ERR_UNSUPPORTED
    assert pag(d=64, wsb=16) == bw.ERR_INVALID_ARG
    assert pag(d=64, B=0, q=None) == bw.OK
    assert pag(B=0, q=None) == bw.OK
