"""Algorithmic work and traffic counts used for the roofline figures (host-side accounting).

"Algorithmic" means what the method itself must compute or move, not what a particular
kernel happens to do:

* prefill FLOPs: two contractions (Q.K^T and P.V) of 2*d FLOPs per (query, key) pair, so
  4*d per pair; with a causal mask the pairs are counted as half of Nq*Nk (the convention
  of the throughput figures in "Attention Computation in Practice", section 7, and of the
  A100 table there).
* prefill bytes: Q, K, V read once and O written once, plus the fp32 log-sum-exp row.
* decode bytes: every cached K and V element of every visible key read once; GQA means each
  KV head is read once for all the query heads that share it ("Attention Computation in
  Practice", GQA in the kernel).
* the two HBM-traffic models of "Attention kernels", Maths (FlashAttention section 3.2 and
  Theorem 2): standard attention moves 4*N*d + 4*N^2 elements, tiled attention with M
  elements of SRAM moves 2*N*d + T_c*(3*N*d + 4*N) with B_c = ceil(M / 4d), T_c = ceil(N / B_c).
"""
from __future__ import annotations

import math


def prefill_flops(B: int, Hq: int, Nq: int, Nk: int, d: int, causal: bool) -> float:
    pairs = float(Nq) * float(Nk)
    if causal:
        pairs *= 0.5
    return 4.0 * d * pairs * B * Hq


def prefill_visible_pairs(Nq: int, Nk: int, causal: bool, window: int = 0) -> int:
    """Exact count of visible (query, key) pairs for one head (causal aligned to the end;
    ``window`` > 0 keeps the last ``window`` keys up to each query's limit)."""
    if not causal:
        return Nq * Nk
    total = 0
    for i in range(Nq):
        hi = min(Nk, i + (Nk - Nq) + 1)
        lo = max(0, i + (Nk - Nq) + 1 - window) if window > 0 else 0
        total += max(0, hi - lo)
    return total


def window_prefill_flops(B: int, Hq: int, Nq: int, Nk: int, d: int, window: int) -> float:
    """Sliding-window prefill: 4*d FLOPs per visible pair, pairs counted exactly (there is no
    half-of-the-square convention for a band)."""
    return 4.0 * d * float(prefill_visible_pairs(Nq, Nk, True, window)) * B * Hq


def prefill_bytes(B: int, Hq: int, Hkv: int, Nq: int, Nk: int, d: int, elem_bytes: int,
                  with_lse: bool = True) -> float:
    q_o = 2.0 * B * Hq * Nq * d * elem_bytes
    kv = 2.0 * B * Hkv * Nk * d * elem_bytes
    lse = 4.0 * B * Hq * Nq if with_lse else 0.0
    return q_o + kv + lse


def decode_kv_bytes(nk_per_seq, Hkv: int, d: int, elem_bytes: int = 2) -> float:
    return 2.0 * float(sum(int(n) for n in nk_per_seq)) * Hkv * d * elem_bytes


def decode_flops(nk_per_seq, Hq: int, d: int) -> float:
    return 4.0 * d * Hq * float(sum(int(n) for n in nk_per_seq))


def decode_partial_bytes(B: int, Hq: int, d: int, num_splits: int) -> float:
    """fp32 (m, l, o[d]) per (sequence, query head, split), written once and read once."""
    return 4.0 * B * Hq * num_splits * (d + 2)


def varlen_flops(nq_list, nk_list, Hq: int, d: int, causal: bool) -> float:
    """Exact visible pairs per sequence (causal aligned to each sequence's end)."""
    total = 0.0
    for nq, nk in zip(nq_list, nk_list):
        if causal:
            # query i sees min(nk, i + nk - nq + 1) keys
            pairs = sum(max(0, min(nk, i + nk - nq + 1)) for i in range(nq))
        else:
            pairs = nq * nk
        total += 4.0 * d * Hq * pairs
    return total


def varlen_bytes(nq_list, nk_list, Hq: int, Hkv: int, d: int, elem_bytes: int = 2) -> float:
    tq, tk = sum(nq_list), sum(nk_list)
    return 2.0 * tq * Hq * d * elem_bytes + 2.0 * tk * Hkv * d * elem_bytes + 4.0 * tq * Hq


def varlen_roofline_seconds(nq_list, nk_list, Hq, Hkv, d, causal, peak_flops, peak_bytes_per_s,
                            elem_bytes: int = 2) -> float:
    """Sum over sequences of max(FLOPs / peak FLOP/s, bytes / peak B/s)."""
    t = 0.0
    for nq, nk in zip(nq_list, nk_list):
        f = varlen_flops([nq], [nk], Hq, d, causal)
        b = varlen_bytes([nq], [nk], Hq, Hkv, d, elem_bytes)
        t += max(f / peak_flops, b / peak_bytes_per_s)
    return t


def standard_attention_elements(N: int, d: int) -> int:
    """Elements moved by standard attention for one head: 4*N*d + 4*N^2."""
    return 4 * N * d + 4 * N * N


def tiled_attention_elements(N: int, d: int, sram_elements: int) -> int:
    """Elements moved by tiled attention with M elements of SRAM: 2*N*d + T_c*(3*N*d + 4*N)."""
    bc = math.ceil(sram_elements / (4 * d))
    tc = math.ceil(N / bc)
    return 2 * N * d + tc * (3 * N * d + 4 * N)


def decode_step_kv_bytes(layers: int, Hkv: int, d: int, elem_bytes: int, S: int, B: int) -> float:
    """KV bytes one decode step reads over all layers (K and V)."""
    return 2.0 * layers * Hkv * d * elem_bytes * S * B
