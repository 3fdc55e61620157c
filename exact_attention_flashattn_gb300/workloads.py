"""Seeded synthetic inputs shaped like the pages' workloads.

This module is shared by the CUDA path's tests/benchmark and by the oracle's tests. It
holds no attention arithmetic: it only draws random tensors, rounds them to the kernel
dtype and packs them. Every draw is ``torch.randn`` (or ``torch.rand`` / ``torch.randint``)
from a ``torch.Generator`` seeded with the workload's seed, in fp32, then cast to the input
dtype with round-to-nearest-even. The same tensor (widened to float64) is what the oracle
sees, so both sides compute on identical values.

Workloads (names give their sizes):

* ``single_head_fp32_512x64``: one head, one sequence, causal, Q/K/V [512, 64] fp32
  N(0, 1), scale 1/8, key tile 128 (the size of the worked example in "Attention
  Computation in Practice", section 4).
* ``prefill_causal_b4_h32_n4096_d128``: causal prefill, B=4, 32 query heads = 32 KV heads,
  Nq = Nk = 4096, d = 128, bf16 N(0, 1); outputs O bf16 plus fp32 log-sum-exp.
* ``decode_gqa_b8_h32x8_n32768_d128``: single-query decode, B=8, 32 query heads over 8 KV
  heads, cache length 32768, d = 128, bf16 N(0, 1), 16 KV splits.
* ``decode_long_b1_h64x8_n262144_d128``: single-query decode, B=1, 64 query heads over 8 KV
  heads, cache length 262144, bf16 N(0, 1) keys and values times a per-channel scale
  c[Hkv, d] ~ U(0.5, 2) (separate draws for K and V), 128 KV splits.
* ``decode_paged_b8_h32x8_n32768_d128_p16``: the GQA decode workload with its caches scattered
  into 16-token pages in a seeded random order, read through a block table.
* ``varlen_append_64seq_h32x8_d128``: 64 sequences with KV length ~ U[1024, 16384] and new
  query count uniform over {1, 4, 8, 512}, packed with cu_seqlens, 32 query heads over 8
  KV heads, d = 128, bf16 N(0, 1), causal aligned to each sequence's end.
* ``prefill_causal_b4_h16_n4096_d256`` and ``decode_gqa_b8_h32x8_n16384_d256``: the prefill and
  the GQA decode at head dim 256 (the pages' third fast head dim), with the same bytes as their
  d = 128 counterparts (half the heads or half the keys); the decode takes 8 splits, 2048 keys
  each, as the d = 128 decode does.
* ``prefill_causal_b4_h32_n4096_d64``: the causal prefill workload at head dim 64 (the pages'
  smallest fast head dim), same B, heads and lengths.
* ``prefill_causal_b4_h32x8_n4096_d128``: the causal prefill workload with grouped-query heads
  (32 query heads over 8 KV heads, the grouping of the decode and varlen workloads).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

SEED_SINGLE_HEAD = 1001
SEED_PREFILL = 1002
SEED_DECODE = 1003
SEED_DECODE_LONG = 1004
SEED_VARLEN = 1005
SEED_FP8_GQA = 1006
SEED_FP8_LONG = 1007
SEED_D256 = 1008
SEED_D64 = 1009
SEED_GQA_PREFILL = 1010
# FP8 caches: N(0, 1) draws are quantised with 448 / 4.5 codes per unit, so |z| up to 4.5 is
# representable and larger draws saturate at the largest code
FP8_SIGMAS = 4.5
FP8_MAX = 448.0

VARLEN_NQ_CHOICES = (1, 4, 8, 512)


@dataclass
class Workload:
    name: str
    kind: str  # "fwd" | "decode" | "varlen"
    dtype: torch.dtype
    B: int = 1
    Hq: int = 1
    Hkv: int = 1
    Nq: int = 0
    Nk: int = 0
    d: int = 128
    causal: bool = True
    num_splits: int = 1
    seed: int = 0
    channel_scale: bool = False
    num_seqs: int = 0
    nk_range: tuple = (0, 0)
    extra: dict = field(default_factory=dict)


WORKLOADS = {
    "single_head_fp32_512x64": Workload("single_head_fp32_512x64", "fwd", torch.float32, B=1, Hq=1, Hkv=1,
                                        Nq=512, Nk=512, d=64, causal=True, seed=SEED_SINGLE_HEAD,
                                        extra={"key_tile": 128}),
    "prefill_causal_b4_h32_n4096_d128": Workload("prefill_causal_b4_h32_n4096_d128", "fwd", torch.bfloat16,
                                                 B=4, Hq=32, Hkv=32, Nq=4096, Nk=4096, d=128, causal=True,
                                                 seed=SEED_PREFILL),
    # the prefill inputs under a sliding window of 1024 keys ("Attention Computation in Practice",
    # Masking variants)
    "prefill_window_b4_h32_n4096_w1024_d128": Workload("prefill_window_b4_h32_n4096_w1024_d128", "fwd",
                                                       torch.bfloat16, B=4, Hq=32, Hkv=32, Nq=4096, Nk=4096,
                                                       d=128, causal=True, seed=SEED_PREFILL,
                                                       extra={"window": 1024}),
    "decode_gqa_b8_h32x8_n32768_d128": Workload("decode_gqa_b8_h32x8_n32768_d128", "decode", torch.bfloat16,
                                                B=8, Hq=32, Hkv=8, Nq=1, Nk=32768, d=128, causal=False,
                                                num_splits=16, seed=SEED_DECODE),
    "decode_long_b1_h64x8_n262144_d128": Workload("decode_long_b1_h64x8_n262144_d128", "decode",
                                                  torch.bfloat16, B=1, Hq=64, Hkv=8, Nq=1, Nk=262144, d=128,
                                                  causal=False, num_splits=128, seed=SEED_DECODE_LONG,
                                                  channel_scale=True),
    "decode_paged_b8_h32x8_n32768_d128_p16": Workload("decode_paged_b8_h32x8_n32768_d128_p16", "decode_paged",
                                                      torch.bfloat16, B=8, Hq=32, Hkv=8, Nq=1, Nk=32768, d=128,
                                                      causal=False, num_splits=16, seed=SEED_DECODE,
                                                      extra={"page_size": 16}),
    # FP8 E4M3 caches with per-(KV head, channel) scales: the GQA decode shape, its paged form,
    # and the long-context decode
    "decode_fp8_gqa_b8_h32x8_n32768_d128": Workload("decode_fp8_gqa_b8_h32x8_n32768_d128", "decode_fp8",
                                                    torch.uint8, B=8, Hq=32, Hkv=8, Nq=1, Nk=32768, d=128,
                                                    causal=False, num_splits=16, seed=SEED_FP8_GQA,
                                                    channel_scale=True),
    "decode_fp8_paged_b8_h32x8_n32768_d128_p16": Workload("decode_fp8_paged_b8_h32x8_n32768_d128_p16",
                                                          "decode_paged_fp8", torch.uint8, B=8, Hq=32, Hkv=8,
                                                          Nq=1, Nk=32768, d=128, causal=False, num_splits=16,
                                                          seed=SEED_FP8_GQA, channel_scale=True,
                                                          extra={"page_size": 16}),
    "decode_fp8_long_b1_h64x8_n262144_d128": Workload("decode_fp8_long_b1_h64x8_n262144_d128", "decode_fp8",
                                                      torch.uint8, B=1, Hq=64, Hkv=8, Nq=1, Nk=262144, d=128,
                                                      causal=False, num_splits=128, seed=SEED_FP8_LONG,
                                                      channel_scale=True),
    "varlen_append_64seq_h32x8_d128": Workload("varlen_append_64seq_h32x8_d128", "varlen", torch.bfloat16,
                                               Hq=32, Hkv=8, d=128, causal=True, seed=SEED_VARLEN,
                                               num_seqs=64, nk_range=(1024, 16384)),
    "prefill_causal_b4_h16_n4096_d256": Workload("prefill_causal_b4_h16_n4096_d256", "fwd", torch.bfloat16,
                                                 B=4, Hq=16, Hkv=16, Nq=4096, Nk=4096, d=256, causal=True,
                                                 seed=SEED_D256),
    "prefill_causal_b4_h32_n4096_d64": Workload("prefill_causal_b4_h32_n4096_d64", "fwd", torch.bfloat16,
                                                B=4, Hq=32, Hkv=32, Nq=4096, Nk=4096, d=64, causal=True,
                                                seed=SEED_D64),
    "prefill_causal_b4_h32x8_n4096_d128": Workload("prefill_causal_b4_h32x8_n4096_d128", "fwd", torch.bfloat16,
                                                   B=4, Hq=32, Hkv=8, Nq=4096, Nk=4096, d=128, causal=True,
                                                   seed=SEED_GQA_PREFILL),
    "decode_gqa_b8_h32x8_n16384_d256": Workload("decode_gqa_b8_h32x8_n16384_d256", "decode", torch.bfloat16,
                                                B=8, Hq=32, Hkv=8, Nq=1, Nk=16384, d=256, causal=False,
                                                num_splits=8, seed=SEED_D256),
}


def _gen(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _randn(shape, gen, dtype, device="cpu", chunk: int = 1 << 24) -> torch.Tensor:
    """N(0, 1) drawn in fp32 and rounded to ``dtype``; large tensors are drawn in chunks of
    ``chunk`` elements (in order) so that the fp32 staging copy stays small."""
    out = torch.empty(shape, dtype=dtype, device=device)
    flat = out.view(-1)
    n = flat.numel()
    step = max(1, chunk)
    for s in range(0, n, step):
        e = min(n, s + step)
        flat[s:e] = torch.randn(e - s, generator=gen, dtype=torch.float32, device=device).to(dtype)
    return out


def prefill_inputs(B, Hq, Hkv, Nq, Nk, d, dtype, seed, device="cpu"):
    """q [B, Hq, Nq, d]; k, v [B, Hkv, Nk, d], i.i.d. N(0, 1) rounded to ``dtype``."""
    g = _gen(seed, device)
    q = _randn((B, Hq, Nq, d), g, dtype, device)
    k = _randn((B, Hkv, Nk, d), g, dtype, device)
    v = _randn((B, Hkv, Nk, d), g, dtype, device)
    return q, k, v


def decode_inputs(B, Hq, Hkv, cap, d, dtype, seed, nk=None, channel_scale=False, device="cpu"):
    """q [B, Hq, d]; caches [B, Hkv, cap, d]; nk [B] int32 (default: every cache full).

    With ``channel_scale`` the keys and values are N(0, 1) times a per-channel factor
    c_K, c_V [Hkv, d] ~ U(0.5, 2), multiplied in fp32 before rounding to ``dtype``.
    """
    g = _gen(seed, device)
    q = _randn((B, Hq, d), g, dtype, device)
    if channel_scale:
        ck = 0.5 + 1.5 * torch.rand((Hkv, d), generator=g, dtype=torch.float32, device=device)
        cv = 0.5 + 1.5 * torch.rand((Hkv, d), generator=g, dtype=torch.float32, device=device)
        kc = torch.empty((B, Hkv, cap, d), dtype=dtype, device=device)
        vc = torch.empty((B, Hkv, cap, d), dtype=dtype, device=device)
        for b in range(B):
            for h in range(Hkv):
                kc[b, h] = (torch.randn((cap, d), generator=g, dtype=torch.float32, device=device)
                            * ck[h]).to(dtype)
            for h in range(Hkv):
                vc[b, h] = (torch.randn((cap, d), generator=g, dtype=torch.float32, device=device)
                            * cv[h]).to(dtype)
    else:
        kc = _randn((B, Hkv, cap, d), g, dtype, device)
        vc = _randn((B, Hkv, cap, d), g, dtype, device)
    if nk is None:
        nk = torch.full((B,), cap, dtype=torch.int32)
    else:
        nk = torch.as_tensor(nk, dtype=torch.int32)
    return q, kc, vc, nk


def fp8_decode_inputs(B, Hq, Hkv, cap, d, seed, nk=None, channel_scale=True, device="cpu"):
    """FP8 KV cache: q [B, Hq, d] bf16; k, v codes [B, Hkv, cap, d] uint8 (E4M3); k_scale,
    v_scale [Hkv, d] fp32; nk [B] int32.

    Each cached element is z ~ N(0, 1) (fp32) quantised as code = e4m3(clamp(z * 448 / 4.5)),
    round to nearest even, by torch's float8_e4m3fn cast; its scale is c * 4.5 / 448 with c the
    per-channel factor U(0.5, 2) of ``channel_scale`` (else 1), so code * scale ~ z * c.
    """
    g = _gen(seed, device)
    q = _randn((B, Hq, d), g, torch.bfloat16, device)
    if channel_scale:
        ck = 0.5 + 1.5 * torch.rand((Hkv, d), generator=g, dtype=torch.float32, device=device)
        cv = 0.5 + 1.5 * torch.rand((Hkv, d), generator=g, dtype=torch.float32, device=device)
    else:
        ck = torch.ones((Hkv, d), dtype=torch.float32, device=device)
        cv = torch.ones((Hkv, d), dtype=torch.float32, device=device)
    k_scale = (ck * (FP8_SIGMAS / FP8_MAX)).contiguous()
    v_scale = (cv * (FP8_SIGMAS / FP8_MAX)).contiguous()
    codes = []
    for _ in range(2):
        c = torch.empty((B, Hkv, cap, d), dtype=torch.uint8, device=device)
        for b in range(B):
            for h in range(Hkv):
                z = torch.randn((cap, d), generator=g, dtype=torch.float32, device=device)
                z = (z * (FP8_MAX / FP8_SIGMAS)).clamp_(-FP8_MAX, FP8_MAX)
                c[b, h] = z.to(torch.float8_e4m3fn).view(torch.uint8)
        codes.append(c)
    if nk is None:
        nk = torch.full((B,), cap, dtype=torch.int32)
    else:
        nk = torch.as_tensor(nk, dtype=torch.int32)
    return q, codes[0], codes[1], k_scale, v_scale, nk


def paged_from_dense(kcache, vcache, page_size, seed):
    """Scatter contiguous caches [B, Hkv, cap, d] into a shuffled page pool.

    Returns k_pages, v_pages [B * cap / page_size, page_size, Hkv, d] and block_table
    [B, cap / page_size] int32 (on the caches' device) such that key j of sequence b is row
    j % page_size of page block_table[b, j // page_size]. The page order is a seeded random
    permutation, so consecutive keys of a sequence are scattered over the pool.
    """
    B, Hkv, cap, d = kcache.shape
    if cap % page_size:
        raise ValueError("cache length must be a multiple of page_size")
    npg = cap // page_size
    g = _gen(seed + 104729)
    perm = torch.randperm(B * npg, generator=g).to(kcache.device)

    def scatter(c):
        pages = c.view(B, Hkv, npg, page_size, d).permute(0, 2, 3, 1, 4).reshape(B * npg, page_size, Hkv, d)
        out = torch.empty_like(pages)
        out[perm] = pages
        return out

    table = perm.view(B, npg).to(torch.int32)
    return scatter(kcache), scatter(vcache), table


def varlen_lengths(num_seqs, seed, nk_range=(1024, 16384), nq_choices=VARLEN_NQ_CHOICES):
    """Per-sequence (n_q, n_k): n_k ~ U[lo, hi] (inclusive integers), n_q uniform over
    ``nq_choices``; n_q never exceeds n_k (the KV length includes the new tokens)."""
    g = _gen(seed)
    lo, hi = nk_range
    nk = torch.randint(lo, hi + 1, (num_seqs,), generator=g, dtype=torch.int64)
    idx = torch.randint(0, len(nq_choices), (num_seqs,), generator=g, dtype=torch.int64)
    nq = torch.tensor([nq_choices[i] for i in idx.tolist()], dtype=torch.int64)
    nq = torch.minimum(nq, nk)
    return nq.tolist(), nk.tolist()


def cu_seqlens(lengths) -> torch.Tensor:
    out = [0]
    for n in lengths:
        out.append(out[-1] + int(n))
    return torch.tensor(out, dtype=torch.int32)


def varlen_inputs(nq_list, nk_list, Hq, Hkv, d, dtype, seed, device="cpu"):
    """Packed q [sum n_q, Hq, d]; k, v [sum n_k, Hkv, d]; cu_seqlens_q, cu_seqlens_k int32."""
    g = _gen(seed + 7919, device)
    tq, tk = int(sum(nq_list)), int(sum(nk_list))
    q = _randn((tq, Hq, d), g, dtype, device)
    k = _randn((tk, Hkv, d), g, dtype, device)
    v = _randn((tk, Hkv, d), g, dtype, device)
    return q, k, v, cu_seqlens(nq_list), cu_seqlens(nk_list)


def make(name: str, device="cpu"):
    """Inputs of a named workload as a dict of tensors and sizes."""
    w = WORKLOADS[name]
    if w.kind == "fwd":
        q, k, v = prefill_inputs(w.B, w.Hq, w.Hkv, w.Nq, w.Nk, w.d, w.dtype, w.seed, device)
        return {"q": q, "k": k, "v": v, "w": w}
    if w.kind in ("decode", "decode_paged"):
        q, kc, vc, nk = decode_inputs(w.B, w.Hq, w.Hkv, w.Nk, w.d, w.dtype, w.seed,
                                      channel_scale=w.channel_scale, device=device)
        if w.kind == "decode":
            return {"q": q, "kcache": kc, "vcache": vc, "nk": nk, "w": w}
        kp, vp, table = paged_from_dense(kc, vc, w.extra["page_size"], w.seed)
        del kc, vc
        return {"q": q, "k_pages": kp, "v_pages": vp, "block_table": table, "nk": nk, "w": w}
    if w.kind in ("decode_fp8", "decode_paged_fp8"):
        q, k8, v8, ks, vs, nk = fp8_decode_inputs(w.B, w.Hq, w.Hkv, w.Nk, w.d, w.seed,
                                                  channel_scale=w.channel_scale, device=device)
        if w.kind == "decode_fp8":
            return {"q": q, "kcache": k8, "vcache": v8, "k_scale": ks, "v_scale": vs, "nk": nk, "w": w}
        kp, vp, table = paged_from_dense(k8, v8, w.extra["page_size"], w.seed)
        del k8, v8
        return {"q": q, "k_pages": kp, "v_pages": vp, "k_scale": ks, "v_scale": vs, "block_table": table,
                "nk": nk, "w": w}
    nq_list, nk_list = varlen_lengths(w.num_seqs, w.seed, w.nk_range)
    q, k, v, cq, ck = varlen_inputs(nq_list, nk_list, w.Hq, w.Hkv, w.d, w.dtype, w.seed, device)
    return {"q": q, "k": k, "v": v, "cu_q": cq, "cu_k": ck, "nq": nq_list, "nk": nk_list, "w": w}
