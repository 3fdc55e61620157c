"""attn_decode_static: the decode entry point that allocates nothing.

Some callers cannot call cudaMalloc or hand the library a workspace (a plugin host that gives
a kernel only its input and output buffers, code whose device memory belongs to another
allocator, a latency-critical loop that cannot take cudaMalloc's device-wide
synchronisation). For them the library keeps the split-K partial states in a fixed device
array. This test calls that entry point through the C-ABI several times in a row with
different problems (each call runs over the previous call's leftovers in the shared array), and
compares each result with the fp64 oracle and with attn_decode's, within the bf16 tolerances of
the other parity tests. It lives in a file of its own, collected last, and passes alone or
after the others.
"""
import ctypes

import numpy as np
import pytest
import torch

import exact_attention_flashattn_gb300 as bw
import oracle
from exact_attention_flashattn_gb300 import build as bw_build
from exact_attention_flashattn_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

TOL_MAX, TOL_MEAN, TOL_LSE = 2e-2, 2e-3, 2e-3
SCRATCH_BYTES = 8 * 1024 * 1024


@pytest.fixture(scope="module")
def static_fn():
    bw_build.build()
    L = ctypes.CDLL(bw.LIB_PATH)  # own handle: the binding's prototypes stay untouched
    f = L.attn_decode_static
    vp, ci = ctypes.c_void_p, ctypes.c_int
    f.argtypes = [vp, vp, vp, vp, vp] + [ci] * 6 + [ctypes.c_float, vp, vp]
    f.restype = ci
    torch.cuda.init()
    return f


def run_static(f, q, kc, vc, nk, S, with_lse=True):
    B, Hq, d = q.shape
    _, Hkv, cap, _ = kc.shape
    o = torch.full_like(q, float("nan"))  # every element must be written by the call
    lse = torch.full((B, Hq), float("nan"), dtype=torch.float32, device=q.device) if with_lse else None
    rc = f(q.data_ptr(), kc.data_ptr(), vc.data_ptr(), o.data_ptr(), nk.data_ptr(), B, Hq, Hkv, cap, d, S,
           1.0 / d ** 0.5, lse.data_ptr() if with_lse else None, torch.cuda.current_stream().cuda_stream)
    return rc, o, lse


def f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def close(a, b, what):
    err = (a.float() - b.float()).abs()
    assert torch.isfinite(err).all(), what
    assert float(err.max()) <= TOL_MAX and float(err.mean()) <= TOL_MEAN, (what, float(err.max()))


def test_static_decode_matches_oracle_and_workspace_decode(static_fn):
    cases = [
        # GQA decode with ragged lengths and one empty sequence, 16 splits
        dict(B=4, Hq=32, Hkv=8, cap=4096, nk=[4096, 1000, 0, 37], S=16, seed=71),
        # a different shape reusing the same array: g = 8, many small splits
        dict(B=1, Hq=64, Hkv=8, cap=20000, nk=[19999], S=96, seed=72),
        # the long-context decode's form: g = 8 over 128 splits (4.3 MB of partials), no LSE output
        dict(B=1, Hq=64, Hkv=8, cap=65536, nk=[65536], S=128, seed=75, lse=False),
        # head dim 64 over the same array
        dict(B=3, Hq=16, Hkv=2, cap=3000, nk=[3000, 5, 1234], S=24, seed=73, d=64),
        # head dim 256 (warp pairs) over the same array
        dict(B=2, Hq=16, Hkv=4, cap=5000, nk=[5000, 777], S=12, seed=74, d=256),
    ]
    for c in cases:
        with_lse = c.get("lse", True)
        q, kc, vc, nk = wl.decode_inputs(c["B"], c["Hq"], c["Hkv"], c["cap"], c.get("d", 128), torch.bfloat16,
                                         c["seed"], nk=c["nk"], device="cuda")
        nk = nk.cuda()
        o_ws, l_ws = bw.attn_decode(q, kc, vc, nk, num_splits=c["S"])
        rc, o, lse = run_static(static_fn, q, kc, vc, nk, c["S"], with_lse)
        torch.cuda.synchronize()
        assert rc == bw.OK, bw.status_string(rc)
        # against the fp64 oracle (split-K with the same number of splits, then the merge rule)
        o_ref, l_ref = oracle.decode(f64(q), f64(kc), f64(vc), nk.cpu().numpy(), method="splitk", workers=c["S"])
        err = np.abs(f64(o) - o_ref)
        assert np.all(np.isfinite(err)), c
        assert err.max() <= TOL_MAX and err.mean() <= TOL_MEAN, (c, err.max(), err.mean())
        # against the workspace entry point
        close(o, o_ws, c)
        if with_lse:
            lg = f64(lse)
            assert np.all(np.isneginf(lg) == np.isneginf(l_ref)), c
            fin = np.isfinite(l_ref)
            assert np.abs(lg[fin] - l_ref[fin]).max() <= TOL_LSE, c
            fin_t = torch.isfinite(l_ws)
            assert torch.equal(torch.isneginf(lse), torch.isneginf(l_ws))
            assert float((lse[fin_t] - l_ws[fin_t]).abs().max()) <= TOL_LSE


def test_static_decode_rejects_partials_beyond_the_array(static_fn):
    # B * Hq * num_splits * (d + 2) * 4 bytes above 8 MiB must be refused before any launch
    B, Hq, Hkv, cap, S = 2, 64, 8, 16, 1024
    assert bw.decode_workspace_size(B, Hq, 128, S) > SCRATCH_BYTES
    q = torch.zeros((B, Hq, 128), dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros((B, Hkv, cap, 128), dtype=torch.bfloat16, device="cuda")
    nk = torch.full((B,), cap, dtype=torch.int32, device="cuda")
    n0 = bw.launch_count()
    rc, _, _ = run_static(static_fn, q, kc, kc, nk, S)
    assert rc == bw.ERR_UNSUPPORTED
    assert bw.launch_count() == n0
