"""GPU parity at the workloads' full sizes, every output element against the fp64 oracle.

Each workload runs through the same call, in the same launch configuration, as the benchmark
(the persistent prefill's band size and item list, the decode's split count and merge form are
those of the full-size problem, which no small case reproduces). The outputs are pre-filled
with NaN, so a work item that is dropped, or a row that no CTA writes, fails the comparison
instead of keeping whatever the allocator returned. The oracle then computes every row of
every head on the host cores ("Attention kernels", Code: the textbook result is the bar for
every tile size) and the comparison is element by element:

* O: max abs error <= 2e-2 and mean abs error <= 2e-3 over all elements (bf16 inputs, fp32
  accumulation, the oracle fed the same bf16 values);
* LSE: abs error <= 2e-3 for every row (the FP8 cache adds the per-row bound of its
  q * k_scale rounding, derived beside ``fp8_ref`` in the other parity file).
"""
import math

import numpy as np
import pytest
import torch

import exact_attention_flashattn_gb300 as bw
import oracle
from exact_attention_flashattn_gb300 import build as bw_build
from exact_attention_flashattn_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

TOL_BF16_MAX, TOL_BF16_MEAN, TOL_LSE = 2e-2, 2e-3, 2e-3


@pytest.fixture(scope="module", autouse=True)
def built():
    bw_build.build()
    bw.lib()
    torch.cuda.init()
    yield


def f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def nan_like(t, shape=None, dtype=None):
    return torch.full(t.shape if shape is None else shape, float("nan"), dtype=t.dtype if dtype is None else dtype,
                      device=t.device)


class Acc:
    """Running element-by-element comparison over chunks of one workload's outputs."""

    def __init__(self, what):
        self.what = what
        self.n = 0
        self.sum = 0.0
        self.max = 0.0
        self.lse_max = 0.0

    def add(self, o_gpu, o_ref, lse_gpu, lse_ref, lse_tol=TOL_LSE):
        err = np.abs(f64(o_gpu) - o_ref)
        assert np.all(np.isfinite(err)), (self.what, "non-finite or unwritten output")
        self.max = max(self.max, float(err.max()))
        self.sum += float(err.sum())
        self.n += err.size
        assert self.max <= TOL_BF16_MAX, (self.what, self.max)
        lg = f64(lse_gpu)
        assert np.all(~np.isnan(lg)), (self.what, "unwritten LSE")
        assert np.all(np.isneginf(lg) == np.isneginf(lse_ref)), self.what
        fin = np.isfinite(lse_ref)
        e = np.abs(lg[fin] - lse_ref[fin])
        tol = np.broadcast_to(lse_tol, lse_ref.shape)[fin]
        assert np.all(e <= tol), (self.what, float(e.max()))
        if e.size:
            self.lse_max = max(self.lse_max, float(e.max()))

    def finish(self):
        assert self.n > 0
        assert self.sum / self.n <= TOL_BF16_MEAN, (self.what, self.sum / self.n)


# ------------------------------------------------------------------ prefill


@pytest.mark.parametrize("name", ["prefill_causal_b4_h32_n4096_d128", "prefill_window_b4_h32_n4096_w1024_d128",
                                  "prefill_causal_b4_h16_n4096_d256", "prefill_causal_b4_h32_n4096_d64",
                                  "prefill_causal_b4_h32x8_n4096_d128"])
def test_prefill_workload_every_row(name):
    x = wl.make(name, device="cuda")
    w = x["w"]
    W = w.extra.get("window", 0)
    o = nan_like(x["q"])
    lse = nan_like(x["q"], (w.B, w.Hq, w.Nq), torch.float32)
    bw.attn_fwd(x["q"], x["k"], x["v"], causal=True, window=W, out=o, lse=lse)
    torch.cuda.synchronize()
    acc = Acc(name)
    for b in range(w.B):  # one sequence (all heads) at a time keeps the fp64 copies small
        o_ref, lse_ref = oracle.attention(f64(x["q"][b:b + 1]), f64(x["k"][b:b + 1]), f64(x["v"][b:b + 1]), True,
                                          method="tiled", block=128, window=W)
        acc.add(o[b:b + 1], o_ref, lse[b:b + 1], lse_ref)
    acc.finish()


def test_varlen_workload_every_row():
    x = wl.make("varlen_append_64seq_h32x8_d128", device="cuda")
    nq, nk = x["nq"], x["nk"]
    cq, ck = x["cu_q"].tolist(), x["cu_k"].tolist()
    o = nan_like(x["q"])
    lse = nan_like(x["q"], x["q"].shape[:2], torch.float32)
    bw.attn_varlen(x["q"], x["k"], x["v"], x["cu_q"].cuda(), x["cu_k"].cuda(), max(nq), max(nk), causal=True,
                   out=o, lse=lse)
    torch.cuda.synchronize()
    acc = Acc("varlen")
    for s in range(len(nq)):  # one sequence at a time through the oracle's varlen call
        qs, ks = slice(cq[s], cq[s + 1]), slice(ck[s], ck[s + 1])
        o_ref, lse_ref = oracle.varlen(f64(x["q"][qs]), f64(x["k"][ks]), f64(x["v"][ks]), [0, nq[s]], [0, nk[s]],
                                       True, method="tiled", block=128)
        acc.add(o[qs], o_ref, lse[qs], lse_ref)
    acc.finish()


# ------------------------------------------------------------------ decode


def decode_every_sequence(name, call, ref_one):
    """Run the workload's decode once, then compare every (sequence, KV head) group of query
    heads with the oracle, one group at a time (the long-context caches are 2 GB per KV head
    and sequence in fp64)."""
    x = wl.make(name, device="cuda")
    w = x["w"]
    g = w.Hq // w.Hkv
    o = nan_like(x["q"])
    lse = nan_like(x["q"], (w.B, w.Hq), torch.float32)
    call(x, w, o, lse)
    torch.cuda.synchronize()
    acc = Acc(name)
    for b in range(w.B):
        for hk in range(w.Hkv):
            sl = slice(hk * g, (hk + 1) * g)
            o_ref, lse_ref, tol = ref_one(x, w, b, hk, sl)
            acc.add(o[b:b + 1, sl], o_ref, lse[b:b + 1, sl], lse_ref, tol)
    acc.finish()


def _bf16_ref(x, w, b, hk, sl):
    o_ref, lse_ref = oracle.decode(f64(x["q"][b:b + 1, sl]), f64(x["kcache"][b:b + 1, hk:hk + 1]),
                                   f64(x["vcache"][b:b + 1, hk:hk + 1]), [w.Nk], method="splitk",
                                   workers=w.num_splits)
    return o_ref, lse_ref, TOL_LSE


@pytest.mark.parametrize("name", ["decode_gqa_b8_h32x8_n32768_d128", "decode_long_b1_h64x8_n262144_d128",
                                  "decode_gqa_b8_h32x8_n16384_d256"])
def test_decode_workload_every_sequence(name):
    def call(x, w, o, lse):
        bw.attn_decode(x["q"], x["kcache"], x["vcache"], x["nk"].cuda(), num_splits=w.num_splits, out=o, lse=lse)

    decode_every_sequence(name, call, _bf16_ref)


def _gather_pages(x, w, b, hk, key):
    """Sequence b's keys of KV head hk, gathered from its pages in order (data movement only)."""
    used = x["block_table"][b].long()
    pages = x[key].index_select(0, used)[:, :, hk]  # [pages, page_size, d]
    return pages.reshape(1, 1, w.Nk, w.d).contiguous()


def test_paged_decode_workload_every_sequence():
    def call(x, w, o, lse):
        bw.attn_decode_paged(x["q"], x["k_pages"], x["v_pages"], x["block_table"], x["nk"].cuda(),
                             num_splits=w.num_splits, out=o, lse=lse)

    def ref(x, w, b, hk, sl):
        kc, vc = _gather_pages(x, w, b, hk, "k_pages"), _gather_pages(x, w, b, hk, "v_pages")
        o_ref, lse_ref = oracle.decode(f64(x["q"][b:b + 1, sl]), f64(kc), f64(vc), [w.Nk], method="splitk",
                                       workers=w.num_splits)
        return o_ref, lse_ref, TOL_LSE

    decode_every_sequence("decode_paged_b8_h32x8_n32768_d128_p16", call, ref)


def _fp8_ref(q, k8, v8, ks, vs, n, S):
    """Oracle decode over the decoded codes, and the per-row LSE bar: 2e-3 plus the largest move
    of a visible score that rounding q * k_scale to f16 (2^-11 relative per product term) can
    cause."""
    o_ref, lse_ref = oracle.decode_fp8(f64(q), k8.cpu().numpy(), v8.cpu().numpy(), f64(ks), f64(vs), [n],
                                       method="splitk", workers=S)
    qd, kd, ksd = f64(q), oracle.e4m3_decode(k8.cpu().numpy()), f64(ks)
    _, Hq, d = qd.shape
    Hkv = kd.shape[1]
    g = Hq // Hkv
    tol = np.full((1, Hq), TOL_LSE)
    for hk in range(Hkv):
        qa = np.abs(qd[0, hk * g:(hk + 1) * g] * ksd[hk][None])
        bound = (np.abs(kd[0, hk, :n]) @ qa.T).max(axis=0)
        tol[0, hk * g:(hk + 1) * g] += 2.0 ** -11 * bound / math.sqrt(d)
    return o_ref, lse_ref, tol


@pytest.mark.parametrize("name", ["decode_fp8_gqa_b8_h32x8_n32768_d128", "decode_fp8_long_b1_h64x8_n262144_d128"])
def test_fp8_decode_workload_every_sequence(name):
    def call(x, w, o, lse):
        bw.attn_decode_fp8(x["q"], x["kcache"], x["vcache"], x["k_scale"], x["v_scale"], x["nk"].cuda(),
                           num_splits=w.num_splits, out=o, lse=lse)

    def ref(x, w, b, hk, sl):
        return _fp8_ref(x["q"][b:b + 1, sl], x["kcache"][b:b + 1, hk:hk + 1], x["vcache"][b:b + 1, hk:hk + 1],
                        x["k_scale"][hk:hk + 1], x["v_scale"][hk:hk + 1], w.Nk, w.num_splits)

    decode_every_sequence(name, call, ref)


def test_fp8_paged_decode_workload_every_sequence():
    def call(x, w, o, lse):
        bw.attn_decode_paged_fp8(x["q"], x["k_pages"], x["v_pages"], x["k_scale"], x["v_scale"], x["block_table"],
                                 x["nk"].cuda(), num_splits=w.num_splits, out=o, lse=lse)

    def ref(x, w, b, hk, sl):
        kc, vc = _gather_pages(x, w, b, hk, "k_pages"), _gather_pages(x, w, b, hk, "v_pages")
        return _fp8_ref(x["q"][b:b + 1, sl], kc, vc, x["k_scale"][hk:hk + 1], x["v_scale"][hk:hk + 1], w.Nk,
                        w.num_splits)

    decode_every_sequence("decode_fp8_paged_b8_h32x8_n32768_d128_p16", call, ref)
