"""Pins for the fp64 oracle: each test checks it against something other than itself.

What pins what (page titles and sections as cited in ``oracle/attention_oracle.cpp``):

* tiled == naive for every tile size from 1 key to the whole sequence, split-K == naive for
  1 to 1,500 workers over 1,000 keys, both to 1e-12 ("Attention kernels", Code: the stated
  tests of that page);
* rows of the naive softmax sum to 1; causal row 0 returns V[0] exactly; brute force on 4x4
  inputs with an independent pure-Python softmax;
* closed forms: zero queries give the mean of the visible values and LSE = ln(n); a single
  dominant key gives a two-level softmax in closed form (pins the 1/sqrt(d) scale and the
  mask alignment); a common key component shifts every score of a row by the same amount;
* invariants: linearity in V, permutation equivariance, masked positions never read
  (poisoned with NaN), GQA by index == GQA by copy ("Attention Computation in Practice",
  exercise C), varlen == per-sequence, decode == dense;
* library routines that share no code with the oracle: torch's fp64 CPU
  scaled_dot_product_attention with an explicit mask, scipy's logsumexp;
* the printed shapes of the page widgets (48x48, d=16, tile 8; 1 query x 4096 keys, 4
  workers) and the "l >= 1 for every non-empty partial" property of the printed partials.
"""
import math

import numpy as np
import pytest
import torch
from scipy.special import logsumexp

import oracle


def rng(seed):
    return np.random.default_rng(seed)


def randn(r, *shape):
    return r.standard_normal(shape)


def dense(r, B, Hq, Hkv, Nq, Nk, d):
    return randn(r, B, Hq, Nq, d), randn(r, B, Hkv, Nk, d), randn(r, B, Hkv, Nk, d)


def visible(i, nq, nk, causal):
    return nk if not causal else max(0, min(nk, i + nk - nq + 1))


# ---------------------------------------------------------------- the pages' stated tests


@pytest.mark.parametrize("causal", [True, False])
def test_tiled_equals_naive_every_tile_size(causal):
    r = rng(1)
    q, k, v = dense(r, 1, 2, 2, 48, 48, 16)
    on, ln = oracle.attention(q, k, v, causal, method="naive")
    for block in range(1, 49):
        ot, lt = oracle.attention(q, k, v, causal, method="tiled", block=block)
        assert np.max(np.abs(ot - on)) <= 1e-12, block
        assert np.max(np.abs(lt - ln)) <= 1e-12, block


def test_tiled_equals_naive_single_head_512x64():
    # the worked example's shape: one head, S=512, D=64, N(0,1), causal, key block 128
    r = rng(2)
    q, k, v = dense(r, 1, 1, 1, 512, 512, 64)
    on, _ = oracle.attention(q, k, v, True, method="naive")
    for block in (1, 2, 3, 7, 64, 127, 128, 129, 511, 512):
        ot, _ = oracle.attention(q, k, v, True, method="tiled", block=block)
        assert np.max(np.abs(ot - on)) <= 1e-12, block
    ot, _ = oracle.attention(q, k, v, True, method="tiled", block=128)
    # the page prints a max difference of about 1e-15 for this comparison
    assert np.max(np.abs(ot - on)) < 1e-13


def test_splitk_1_to_1500_workers_over_1000_keys():
    r = rng(3)
    q, k, v = dense(r, 1, 1, 1, 1, 1000, 16)
    on, ln = oracle.attention(q, k, v, False, method="naive")
    for w in range(1, 1501):
        os_, ls = oracle.attention(q, k, v, False, method="splitk", workers=w)
        assert np.max(np.abs(os_ - on)) <= 1e-12, w
        assert np.max(np.abs(ls - ln)) <= 1e-12, w


def test_widget_shapes():
    # 48 queries x 48 keys, d = 16, tile 8 (printed 1.6e-15) and one query over 4,096 keys
    # merged from 4 partials (printed 1.5e-15): the same magnitude must hold here.
    r = rng(4)
    q, k, v = dense(r, 1, 1, 1, 48, 48, 16)
    on, _ = oracle.attention(q, k, v, False, method="naive")
    ot, _ = oracle.attention(q, k, v, False, method="tiled", block=8)
    assert np.max(np.abs(ot - on)) < 1e-13
    q, k, v = dense(r, 1, 1, 1, 1, 4096, 16)
    on, _ = oracle.attention(q, k, v, False, method="naive")
    os_, _ = oracle.attention(q, k, v, False, method="splitk", workers=4)
    assert np.max(np.abs(os_ - on)) < 1e-13


def test_partials_have_l_at_least_one():
    # each non-empty partial contains its own max term, exp(0) = 1, so 1 <= l <= n_keys; the
    # widget's printed partials (l = 2.0, 1.8, 2.9, 2.6 for 1,024-key slices) satisfy this.
    r = rng(5)
    n, d = 4096, 16
    q, k, v = randn(r, d) * 3.0, randn(r, n, d), randn(r, n, d)
    for w in (1, 4, 7, 64, 4096, 5000):
        m, l, o = oracle.partials(q, k, v, w)
        chunk = -(-n // w)
        for i in range(w):
            size = max(0, min(n, (i + 1) * chunk) - min(n, i * chunk))
            if size == 0:
                assert l[i] == 0.0 and m[i] == -math.inf and not np.any(o[i])
            else:
                assert 1.0 <= l[i] <= size


# ---------------------------------------------------------------- definitions and brute force


@pytest.mark.parametrize("causal", [True, False])
def test_softmax_rows_sum_to_one(causal):
    r = rng(6)
    q, k = randn(r, 37, 16) * 2.0, randn(r, 53, 16)
    p = oracle.probs(q, k, causal)
    for i in range(37):
        n = visible(i, 37, 53, causal)
        assert abs(p[i, :n].sum() - 1.0) <= 1e-14
        assert np.all(p[i, :n] > 0.0)
        assert np.all(p[i, n:] == 0.0)


def test_causal_row_zero_is_v0_exactly():
    r = rng(7)
    q, k, v = dense(r, 2, 4, 2, 64, 64, 32)
    for method, kw in (("naive", {}), ("tiled", {"block": 1}), ("tiled", {"block": 16}),
                       ("splitk", {"workers": 1}), ("splitk", {"workers": 9})):
        o, lse = oracle.attention(q, k, v, True, method=method, **kw)
        for b in range(2):
            for h in range(4):
                assert np.array_equal(o[b, h, 0], v[b, h // 2, 0])
                s0 = float(np.dot(q[b, h, 0], k[b, h // 2, 0])) / math.sqrt(32)
                assert abs(lse[b, h, 0] - s0) <= 1e-15 * max(1.0, abs(s0))


def brute_force(q, k, v, causal, scale):
    """Softmax by its definition exp(s_ij) / sum_k exp(s_ik), no max subtraction, scalar loops."""
    nq, d = len(q), len(q[0])
    nk = len(k)
    out, lses = [], []
    for i in range(nq):
        n = visible(i, nq, nk, causal)
        s = [scale * sum(q[i][c] * k[j][c] for c in range(d)) for j in range(n)]
        e = [math.exp(x) for x in s]
        z = sum(e)
        out.append([sum(e[j] / z * v[j][c] for j in range(n)) for c in range(d)])
        lses.append(math.log(z))
    return np.array(out), np.array(lses)


@pytest.mark.parametrize("causal", [True, False])
def test_brute_force_4x4(causal):
    r = rng(8)
    q, k, v = randn(r, 4, 4), randn(r, 4, 4), randn(r, 4, 4)
    ob, lb = brute_force(q.tolist(), k.tolist(), v.tolist(), causal, 0.5)
    q4, k4, v4 = q[None, None], k[None, None], v[None, None]
    for method, kw in (("naive", {}), ("tiled", {"block": 1}), ("tiled", {"block": 3}),
                       ("tiled", {"block": 4}), ("splitk", {"workers": 2}), ("splitk", {"workers": 5})):
        o, lse = oracle.attention(q4, k4, v4, causal, method=method, **kw)
        assert np.max(np.abs(o[0, 0] - ob)) <= 1e-14, method
        assert np.max(np.abs(lse[0, 0] - lb)) <= 1e-14, method


def test_brute_force_rectangular_bottom_right():
    # 3 queries against 5 keys, causal aligned to the end: row i sees i + 3 keys
    r = rng(9)
    q, k, v = randn(r, 3, 4), randn(r, 5, 4), randn(r, 5, 4)
    ob, lb = brute_force(q.tolist(), k.tolist(), v.tolist(), True, 0.5)
    o, lse = oracle.attention(q[None, None], k[None, None], v[None, None], True, method="tiled", block=2)
    assert np.max(np.abs(o[0, 0] - ob)) <= 1e-14
    assert np.max(np.abs(lse[0, 0] - lb)) <= 1e-14


# ---------------------------------------------------------------- closed forms


@pytest.mark.parametrize("d", [8, 256])
@pytest.mark.parametrize("nq,nk,causal", [(8, 8, True), (5, 11, True), (8, 8, False), (1, 33, False)])
def test_zero_queries_give_mean_of_visible_values(nq, nk, causal, d):
    r = rng(10)
    q = np.zeros((1, 1, nq, d))
    k, v = randn(r, 1, 1, nk, d), randn(r, 1, 1, nk, d)
    for method, kw in (("naive", {}), ("tiled", {"block": 3}), ("splitk", {"workers": 4})):
        o, lse = oracle.attention(q, k, v, causal, method=method, **kw)
        for i in range(nq):
            n = visible(i, nq, nk, causal)
            assert np.max(np.abs(o[0, 0, i] - v[0, 0, :n].mean(axis=0))) <= 1e-14
            assert abs(lse[0, 0, i] - math.log(n)) <= 1e-14


@pytest.mark.parametrize("scale", [None, 0.3])
def test_single_dominant_key_closed_form(scale):
    # keys are zero except key t = c * e0 and queries are a_i * e0, so row i has one score
    # s = a_i * c * scale at key t (if visible) and zeros elsewhere:
    #   O_i = (e^s v_t + sum_{j != t} v_j) / (e^s + n - 1),  LSE_i = ln(e^s + n - 1)
    r = rng(11)
    nq = nk = 12
    d, t, c = 16, 5, 2.0
    sc = 1.0 / math.sqrt(d) if scale is None else scale
    a = r.uniform(-3.0, 3.0, nq)
    q = np.zeros((1, 1, nq, d))
    q[0, 0, :, 0] = a
    k = np.zeros((1, 1, nk, d))
    k[0, 0, t, 0] = c
    v = randn(r, 1, 1, nk, d)
    o, lse = oracle.attention(q, k, v, True, scale=scale, method="tiled", block=4)
    for i in range(nq):
        n = i + 1
        vis = v[0, 0, :n]
        if t < n:
            s = a[i] * c * sc
            num = math.exp(s) * vis[t] + (vis.sum(axis=0) - vis[t])
            den = math.exp(s) + n - 1
        else:
            num, den = vis.sum(axis=0), float(n)
        assert np.max(np.abs(o[0, 0, i] - num / den)) <= 1e-13
        assert abs(lse[0, 0, i] - math.log(den)) <= 1e-13


def test_common_key_component_shifts_scores():
    # k_j = k'_j + u shifts every score of row i by scale * q_i . u: O is unchanged and the
    # log-sum-exp moves by exactly that amount.
    r = rng(12)
    q, k, v = dense(r, 1, 1, 1, 20, 20, 8)
    u = randn(r, 8) * 4.0
    o0, l0 = oracle.attention(q, k, v, True, method="tiled", block=6)
    o1, l1 = oracle.attention(q, k + u, v, True, method="tiled", block=6)
    shift = (q[0, 0] @ u) / math.sqrt(8)
    assert np.max(np.abs(o1 - o0)) <= 1e-12
    assert np.max(np.abs(l1[0, 0] - l0[0, 0] - shift)) <= 1e-12


def test_dominant_key_at_large_scores_is_one_hot():
    # safe softmax: scores near 1e3 must not overflow; a key whose score leads by > 745
    # makes every other weight underflow to zero, so O is exactly that value row.
    d = 4
    q = np.zeros((1, 1, 1, d))
    q[0, 0, 0, 0] = 100.0
    k = np.zeros((1, 1, 6, d))
    k[0, 0, :, 0] = [1.0, 2.0, 30.0, 3.0, 4.0, 5.0]
    v = rng(13).standard_normal((1, 1, 6, d))
    for method, kw in (("naive", {}), ("tiled", {"block": 1}), ("tiled", {"block": 4}), ("splitk", {"workers": 3})):
        o, lse = oracle.attention(q, k, v, False, scale=1.0, method=method, **kw)
        assert np.array_equal(o[0, 0, 0], v[0, 0, 2]), method
        assert lse[0, 0, 0] == 3000.0


# ---------------------------------------------------------------- invariants


def test_linear_in_values():
    r = rng(14)
    q, k, v = dense(r, 1, 2, 1, 30, 30, 8)
    o, _ = oracle.attention(q, k, v, True, method="tiled", block=7)
    o2, _ = oracle.attention(q, k, 2.5 * v - 1.25, True, method="tiled", block=7)
    assert np.max(np.abs(o2 - (2.5 * o - 1.25))) <= 1e-12


def test_permutation_equivariance_without_mask():
    r = rng(15)
    q, k, v = dense(r, 1, 1, 1, 16, 40, 8)
    o, l = oracle.attention(q, k, v, False, method="tiled", block=5)
    pk = r.permutation(40)
    pq = r.permutation(16)
    o2, l2 = oracle.attention(q[:, :, pq], k[:, :, pk], v[:, :, pk], False, method="tiled", block=5)
    assert np.max(np.abs(o2 - o[:, :, pq])) <= 1e-12
    assert np.max(np.abs(l2 - l[:, :, pq])) <= 1e-12


def test_masked_positions_are_never_read():
    r = rng(16)
    q, k, v = dense(r, 1, 1, 1, 24, 24, 8)
    o, l = oracle.attention(q, k, v, True, method="tiled", block=8)
    k2, v2 = k.copy(), v.copy()
    k2[0, 0, -1] = np.nan
    v2[0, 0, -1] = np.nan
    o2, l2 = oracle.attention(q, k2, v2, True, method="tiled", block=8)
    # only the last query sees the last key
    assert np.array_equal(o2[0, 0, :-1], o[0, 0, :-1])
    assert np.array_equal(l2[0, 0, :-1], l[0, 0, :-1])
    assert np.all(np.isnan(o2[0, 0, -1]))


def test_rows_without_visible_keys():
    # more queries than keys, causal aligned to the end: the first Nq - Nk rows see nothing
    r = rng(17)
    q, k, v = dense(r, 1, 1, 1, 6, 4, 8)
    for method, kw in (("naive", {}), ("tiled", {"block": 2}), ("splitk", {"workers": 3})):
        o, lse = oracle.attention(q, k, v, True, method=method, **kw)
        assert np.all(o[0, 0, :2] == 0.0) and np.all(lse[0, 0, :2] == -math.inf)
        assert np.all(np.isfinite(lse[0, 0, 2:]))


def test_gqa_by_index_equals_gqa_by_copy():
    r = rng(18)
    q, k, v = dense(r, 2, 8, 2, 10, 17, 8)
    o1, l1 = oracle.attention(q, k, v, True, method="tiled", block=4)
    kc = np.repeat(k, 4, axis=1)  # materialised copies: head h -> KV head h // 4
    vc = np.repeat(v, 4, axis=1)
    o2, l2 = oracle.attention(q, kc, vc, True, method="tiled", block=4)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_varlen_equals_per_sequence_dense():
    r = rng(19)
    nq, nk = [1, 4, 9, 3], [5, 4, 20, 3]
    Hq, Hkv, d = 4, 2, 8
    q = randn(r, sum(nq), Hq, d)
    k = randn(r, sum(nk), Hkv, d)
    v = randn(r, sum(nk), Hkv, d)
    cq = np.concatenate([[0], np.cumsum(nq)]).astype(np.int32)
    ck = np.concatenate([[0], np.cumsum(nk)]).astype(np.int32)
    o, lse = oracle.varlen(q, k, v, cq, ck, True, method="tiled", block=3)
    for s in range(4):
        qs = q[cq[s]:cq[s + 1]].transpose(1, 0, 2)[None]
        ks = k[ck[s]:ck[s + 1]].transpose(1, 0, 2)[None]
        vs = v[ck[s]:ck[s + 1]].transpose(1, 0, 2)[None]
        od, ld = oracle.attention(qs, ks, vs, True, method="tiled", block=3)
        assert np.array_equal(o[cq[s]:cq[s + 1]], od[0].transpose(1, 0, 2))
        assert np.array_equal(lse[cq[s]:cq[s + 1]], ld[0].T)


def test_decode_equals_dense_and_ignores_tail_of_cache():
    r = rng(20)
    B, Hq, Hkv, cap, d = 3, 8, 2, 40, 16
    q = randn(r, B, Hq, d)
    kc, vc = randn(r, B, Hkv, cap, d), randn(r, B, Hkv, cap, d)
    nk = np.array([40, 7, 1], dtype=np.int32)
    o, lse = oracle.decode(q, kc, vc, nk, method="splitk", workers=16)  # 16 > 7 and 1: empty splits
    kp, vp = kc.copy(), vc.copy()
    for b in range(B):
        kp[b, :, nk[b]:] = np.nan
        vp[b, :, nk[b]:] = np.nan
    o2, l2 = oracle.decode(q, kp, vp, nk, method="splitk", workers=16)
    assert np.array_equal(o, o2) and np.array_equal(lse, l2)
    for b in range(B):
        n = int(nk[b])
        od, ld = oracle.attention(q[b][None, :, None], kc[b][None, :, :n], vc[b][None, :, :n], False,
                                  method="naive")
        assert np.max(np.abs(o[b] - od[0, :, 0])) <= 1e-12
        assert np.max(np.abs(lse[b] - ld[0, :, 0])) <= 1e-12


# ---------------------------------------------------------------- merge rule


def test_merge_rule():
    r = rng(21)
    d, n = 8, 30
    q, k, v = randn(r, d), randn(r, n, d), randn(r, n, d)
    m, l, o = oracle.partials(q, k, v, 3)
    # empty partial is the identity, on either side
    e = np.zeros(d)
    mm, ll, oo = oracle.merge(m[0], l[0], o[0], -math.inf, 0.0, e)
    assert (mm, ll) == (m[0], l[0]) and np.array_equal(oo, o[0])
    mm, ll, oo = oracle.merge(-math.inf, 0.0, e, m[1], l[1], o[1])
    assert (mm, ll) == (m[1], l[1]) and np.array_equal(oo, o[1])
    # commutative and associative up to rounding; merging all parts gives the whole row
    ab = oracle.merge(m[0], l[0], o[0], m[1], l[1], o[1])
    ba = oracle.merge(m[1], l[1], o[1], m[0], l[0], o[0])
    assert ab[0] == ba[0] and abs(ab[1] - ba[1]) <= 1e-14 * ab[1] and np.max(np.abs(ab[2] - ba[2])) <= 1e-13
    left = oracle.merge(*ab, m[2], l[2], o[2])
    bc = oracle.merge(m[1], l[1], o[1], m[2], l[2], o[2])
    right = oracle.merge(m[0], l[0], o[0], *bc)
    assert abs(left[1] - right[1]) <= 1e-13 * left[1] and np.max(np.abs(left[2] - right[2])) <= 1e-12
    full_m, full_l, full_o = oracle.partials(q, k, v, 1)
    assert left[0] == full_m[0]
    assert abs(left[1] - full_l[0]) <= 1e-13 * full_l[0]
    assert np.max(np.abs(left[2] - full_o[0])) <= 1e-12


# ---------------------------------------------------------------- independent library routines


@pytest.mark.parametrize("nq,nk,causal", [(33, 33, True), (7, 50, True), (20, 45, False)])
def test_matches_torch_sdpa_fp64(nq, nk, causal):
    r = rng(22)
    q, k, v = dense(r, 2, 4, 2, nq, nk, 16)
    o, _ = oracle.attention(q, k, v, causal, method="tiled", block=8)
    mask = torch.ones(nq, nk, dtype=torch.bool)
    if causal:
        mask = torch.tensor([[j < visible(i, nq, nk, True) for j in range(nk)] for i in range(nq)])
    tq = torch.from_numpy(q)
    tk = torch.from_numpy(np.repeat(k, 2, axis=1))
    tv = torch.from_numpy(np.repeat(v, 2, axis=1))
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask).numpy()
    assert np.max(np.abs(o - ref)) <= 1e-12


def test_lse_matches_scipy_logsumexp():
    r = rng(23)
    q, k, v = dense(r, 1, 2, 2, 25, 25, 16)
    _, lse = oracle.attention(q, k, v, True, method="splitk", workers=6)
    s = np.einsum("bhid,bhjd->bhij", q, k) / 4.0
    for h in range(2):
        for i in range(25):
            assert abs(lse[0, h, i] - logsumexp(s[0, h, i, :i + 1])) <= 1e-12


def test_paged_decode_gathers_the_same_keys():
    # scattering a contiguous cache into shuffled pages and reading it back through the block
    # table must reproduce the contiguous decode exactly ("Attention Computation in Practice",
    # PagedAttention's kernel difference)
    from exact_attention_flashattn_gb300 import workloads as wl
    q, kc, vc, nk = wl.decode_inputs(3, 8, 2, 64, 16, torch.float32, seed=61, nk=[64, 17, 30])
    kp, vp, table = wl.paged_from_dense(kc, vc, 16, seed=61)
    assert sorted(table.flatten().tolist()) == list(range(3 * 4))
    o1, l1 = oracle.decode(q.numpy(), kc.numpy(), vc.numpy(), nk.numpy(), method="splitk", workers=3)
    o2, l2 = oracle.decode_paged(q.numpy(), kp.numpy(), vp.numpy(), table.numpy(), nk.numpy(), method="splitk",
                                 workers=3)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    # and a page that the table never references does not matter
    kp2 = kp.clone()
    kp2[int(table[1, 3])] = float("nan")  # sequence 1 has 17 keys: pages 0 and 1 only
    o3, _ = oracle.decode_paged(q.numpy(), kp2.numpy(), vp.numpy(), table.numpy(), nk.numpy(), method="splitk",
                                workers=3)
    assert np.array_equal(o1, o3)


# ---------------------------------------------------------------- sliding window
# "Attention Computation in Practice", Masking variants: sliding window i - W < j <= i.


def test_window_at_least_the_sequence_is_plain_causal():
    r = rng(31)
    q, k, v = dense(r, 1, 2, 1, 40, 55, 8)
    o0, l0 = oracle.attention(q, k, v, True, method="tiled", block=8)
    for w in (55, 56, 1000):
        o1, l1 = oracle.attention(q, k, v, True, method="tiled", block=8, window=w)
        assert np.array_equal(o0, o1) and np.array_equal(l0, l1)


def test_window_of_one_returns_the_diagonal_value():
    r = rng(32)
    q, k, v = dense(r, 1, 1, 1, 20, 20, 8)
    for method, kw in (("naive", {}), ("tiled", {"block": 3}), ("splitk", {"workers": 4})):
        o, lse = oracle.attention(q, k, v, True, method=method, window=1, **kw)
        assert np.array_equal(o[0, 0], v[0, 0])
        s = np.einsum("id,id->i", q[0, 0], k[0, 0]) / math.sqrt(8)
        assert np.max(np.abs(lse[0, 0] - s)) <= 1e-14


@pytest.mark.parametrize("nq,nk,w", [(16, 16, 5), (6, 30, 7), (30, 30, 1)])
def test_window_zero_queries_mean_over_window(nq, nk, w):
    r = rng(33)
    q = np.zeros((1, 1, nq, 4))
    k, v = randn(r, 1, 1, nk, 4), randn(r, 1, 1, nk, 4)
    for method, kw in (("naive", {}), ("tiled", {"block": 4}), ("splitk", {"workers": 3})):
        o, lse = oracle.attention(q, k, v, True, method=method, window=w, **kw)
        for i in range(nq):
            hi = visible(i, nq, nk, True)
            lo = max(0, hi - w)
            assert np.max(np.abs(o[0, 0, i] - v[0, 0, lo:hi].mean(axis=0))) <= 1e-14
            assert abs(lse[0, 0, i] - math.log(hi - lo)) <= 1e-14


def test_window_brute_force_and_varlen():
    r = rng(34)
    q, k, v = randn(r, 5, 4), randn(r, 7, 4), randn(r, 7, 4)
    w = 3
    # brute force with the window restricting the visible range: keys [hi - 3, hi)
    nq, nk = 5, 7
    ref_o, ref_l = [], []
    for i in range(nq):
        hi = visible(i, nq, nk, True)
        lo = max(0, hi - w)
        s = [0.5 * sum(q[i][c] * k[j][c] for c in range(4)) for j in range(lo, hi)]
        e = [math.exp(x) for x in s]
        z = sum(e)
        ref_o.append([sum(e[j - lo] / z * v[j][c] for j in range(lo, hi)) for c in range(4)])
        ref_l.append(math.log(z))
    o, lse = oracle.attention(q[None, None], k[None, None], v[None, None], True, window=w, method="tiled", block=2)
    assert np.max(np.abs(o[0, 0] - np.array(ref_o))) <= 1e-14
    assert np.max(np.abs(lse[0, 0] - np.array(ref_l))) <= 1e-14
    # the packed form with the window equals the per-sequence dense form
    nqs, nks = [1, 5, 3], [9, 7, 3]
    Q = randn(r, sum(nqs), 2, 4)
    K = randn(r, sum(nks), 1, 4)
    V = randn(r, sum(nks), 1, 4)
    cq = np.concatenate([[0], np.cumsum(nqs)]).astype(np.int32)
    ck = np.concatenate([[0], np.cumsum(nks)]).astype(np.int32)
    ov, lv = oracle.varlen(Q, K, V, cq, ck, True, window=2, method="tiled", block=2)
    for s_ in range(3):
        od, ld = oracle.attention(Q[cq[s_]:cq[s_ + 1]].transpose(1, 0, 2)[None],
                                  K[ck[s_]:ck[s_ + 1]].transpose(1, 0, 2)[None],
                                  V[ck[s_]:ck[s_ + 1]].transpose(1, 0, 2)[None], True, window=2, method="tiled",
                                  block=2)
        assert np.array_equal(ov[cq[s_]:cq[s_ + 1]], od[0].transpose(1, 0, 2))


# ---------------------------------------------------------------- FP8 (E4M3) KV cache
# The cached value is e4m3(code) * scale[KV head, channel] ("Attention from the kernel's side",
# Why a quantised cache needs a fused kernel); the code format is the OCP FP8 E4M3 float.


def test_e4m3_decode_matches_torch_for_every_code():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_decode(codes)
    theirs = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(theirs)
    assert np.array_equal(np.isnan(ours), nan)
    assert list(np.flatnonzero(nan)) == [0x7F, 0xFF]
    assert np.array_equal(ours[~nan], theirs[~nan])
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(theirs[~nan]))


def test_e4m3_landmarks_and_order():
    v = oracle.e4m3_decode(np.arange(256, dtype=np.uint8))
    assert v[0x38] == 1.0 and v[0x30] == 0.5 and v[0x40] == 2.0
    assert v[0x7E] == 448.0                 # largest finite
    assert v[0x01] == 2.0 ** -9             # smallest subnormal
    assert v[0x08] == 2.0 ** -6             # smallest normal
    assert v[0x07] == 7 * 2.0 ** -9         # largest subnormal
    assert v[0x00] == 0.0 and np.signbit(v[0x80]) and v[0x80] == 0.0
    pos = v[:0x7F]
    assert np.all(np.diff(pos) > 0)        # codes 0..126 strictly increasing
    assert np.array_equal(v[0x80:0xFF], -pos)  # sign-magnitude
    # spacing: 8 values per binade above the subnormals
    for e in range(1, 15):
        run = pos[8 * e:8 * e + 8]
        assert np.allclose(np.diff(run), 2.0 ** (e - 7) / 8, rtol=0, atol=0)


def test_e4m3_round_trip_through_torch_quantiser():
    r = rng(61)
    x = torch.from_numpy(np.clip(randn(r, 4096) * 100, -448, 448)).to(torch.float32)
    codes = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    back = x.to(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(oracle.e4m3_decode(codes), back)
    # relative rounding error of a normal value is at most half a unit in the last place (2^-4)
    xn = x.double().numpy()
    big = np.abs(xn) >= 2.0 ** -6
    assert np.max(np.abs(back[big] - xn[big]) / np.abs(xn[big])) <= 2.0 ** -4


def fp8_cache(r, B, Hkv, cap, d):
    k = r.integers(0, 256, size=(B, Hkv, cap, d), dtype=np.uint8)
    v = r.integers(0, 256, size=(B, Hkv, cap, d), dtype=np.uint8)
    # no NaN codes: a saturating quantiser never writes them
    k[(k & 0x7F) == 0x7F] = 0x7E
    v[(v & 0x7F) == 0x7F] = 0x7E
    ks = r.uniform(0.5, 2.0, size=(Hkv, d)) / 64
    vs = r.uniform(0.5, 2.0, size=(Hkv, d)) / 64
    return k, v, ks, vs


def test_decode_fp8_matches_torch_sdpa_on_torch_dequantised_cache():
    r = rng(62)
    B, Hq, Hkv, cap, d = 2, 4, 2, 40, 16
    k8, v8, ks, vs = fp8_cache(r, B, Hkv, cap, d)
    q = randn(r, B, Hq, d)
    nk = np.array([40, 17], dtype=np.int32)
    o, lse = oracle.decode_fp8(q, k8, v8, ks, vs, nk, method="splitk", workers=3)

    def deq(c, s):
        return torch.from_numpy(c).view(torch.float8_e4m3fn).to(torch.float64) * torch.from_numpy(s)[None, :, None, :]
    K, V = deq(k8, ks), deq(v8, vs)
    for b in range(B):
        for h in range(Hq):
            kk = K[b, h // 2, :nk[b]][None, None]
            vv = V[b, h // 2, :nk[b]][None, None]
            qq = torch.from_numpy(q[b, h])[None, None, None]
            ref = torch.nn.functional.scaled_dot_product_attention(qq, kk, vv)[0, 0, 0].numpy()
            assert np.max(np.abs(o[b, h] - ref)) <= 1e-12
            s = (kk[0, 0].numpy() @ q[b, h]) / math.sqrt(d)
            assert abs(lse[b, h] - logsumexp(s)) <= 1e-12


def test_decode_fp8_closed_forms():
    r = rng(63)
    B, Hq, Hkv, cap, d = 1, 2, 1, 33, 8
    k8, v8, ks, vs = fp8_cache(r, B, Hkv, cap, d)
    nk = np.array([33], dtype=np.int32)
    # zero query: the mean of the decoded values times the value scale, LSE = ln n
    o, lse = oracle.decode_fp8(np.zeros((B, Hq, d)), k8, v8, ks, vs, nk, method="naive")
    torch_v = torch.from_numpy(v8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    mean = torch_v[0, 0].mean(axis=0) * vs[0]
    assert np.max(np.abs(o[0] - mean[None])) <= 1e-14
    assert np.max(np.abs(lse - math.log(33))) <= 1e-14
    # doubling the value scale doubles O exactly; the key scale acts like the softmax scale
    q = randn(r, B, Hq, d)
    o1, l1 = oracle.decode_fp8(q, k8, v8, ks, vs, nk, method="tiled", block=4)
    o2, l2 = oracle.decode_fp8(q, k8, v8, ks, 2 * vs, nk, method="tiled", block=4)
    assert np.array_equal(o2, 2 * o1) and np.array_equal(l1, l2)
    ones = np.ones_like(ks)
    o3, l3 = oracle.decode_fp8(q, k8, v8, 3 * ones, vs, nk, method="naive")
    o4, l4 = oracle.decode_fp8(q, k8, v8, ones, vs, nk, method="naive", scale=3 / math.sqrt(d))
    # (the codes reach 448, so scores and LSE are large: compare LSE relative to its size)
    assert np.max(np.abs(o3 - o4)) <= 1e-13 and np.max(np.abs(l3 - l4) / np.maximum(1, np.abs(l3))) <= 1e-14
    # NaN codes decode to NaN (the format has no infinities)
    bad = k8.copy()
    bad[0, 0, 0, 0] = 0x7F
    o5, _ = oracle.decode_fp8(q, bad, v8, ks, vs, nk, method="naive")
    assert np.isnan(o5).all()
