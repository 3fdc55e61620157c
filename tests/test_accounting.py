"""Host-side accounting (algorithmic FLOPs and bytes) pinned to the numbers the pages print.

Fixtures live in ``tests/golden/``; each names the page and section it comes from.
"""
import json
import math
import os

from exact_attention_flashattn_gb300 import roofline

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def test_hbm_traffic_simulator_defaults():
    g = load("hbm_traffic_simulator.json")
    i, p = g["inputs"], g["printed"]
    eb = i["bytes_per_element"]
    std = roofline.standard_attention_elements(i["N"], i["d"]) * eb
    til = roofline.tiled_attention_elements(i["N"], i["d"], i["sram_bytes"] // eb) * eb
    bw = i["bandwidth_bytes_per_s"] * i["bandwidth_fraction"]
    assert round(std / 1e6, 1) == p["standard_MB"]
    assert round(til / 1e6, 1) == p["tiled_MB"]
    assert round(std / bw * 1e6, 1) == p["standard_us"]
    assert round(til / bw * 1e6, 1) == p["tiled_us"]
    assert round(std / til, 1) == p["reduction"]
    assert round(i["N"] * i["N"] * eb / 1e6, 1) == p["nxn_MB"]


def test_decode_kv_bytes_example():
    g = load("decode_kv_bytes.json")
    i, p = g["inputs"], g["printed"]
    b = roofline.decode_step_kv_bytes(i["layers"], i["kv_heads"], i["head_dim"], i["bytes_per_element"], i["S"],
                                      i["B"])
    assert round(b / 1e9) == p["kv_GB_per_step"]
    assert round(b / i["hbm_bytes_per_s"] * 1e3) == p["ms_per_step"]
    # the same count through the per-layer decode accounting used by the benchmark
    per_layer = roofline.decode_kv_bytes([i["S"]] * i["B"], i["kv_heads"], i["head_dim"], i["bytes_per_element"])
    assert per_layer * i["layers"] == b


def test_score_matrix_sizes():
    g = load("score_matrix_sizes.json")
    c = g["cases"]
    sz = [x["N"] * x["N"] * x["heads"] * x["bytes_per_element"] * x["matrices"] for x in c]
    assert sz[0] / 2**30 == c[0]["printed_GiB"]
    assert round(sz[1] / 1e9, 1) == c[1]["printed_GB"]
    assert round(sz[2] / 1e6) == c[2]["printed_MB"]
    assert sz[3] / 2**20 == c[3]["printed_MiB"]
    gr = g["growth"]
    assert (gr["to_N"] / gr["from_N"]) ** 2 == gr["printed_factor"]


def test_prefill_flops_causal_is_half():
    f = roofline.prefill_flops(4, 32, 4096, 4096, 128, True)
    assert f == 4 * 128 * 4096 * 4096 / 2 * 4 * 32
    assert abs(f - 5.497558e11) / f < 1e-6
    # the exact count of visible pairs differs from half by the diagonal
    exact = roofline.prefill_visible_pairs(4096, 4096, True)
    assert exact == 4096 * 4097 // 2


def test_varlen_flops_match_visible_pairs():
    nq, nk = [1, 4, 512], [1024, 2000, 4096]
    f = roofline.varlen_flops(nq, nk, 32, 128, True)
    pairs = sum(roofline.prefill_visible_pairs(a, b, True) for a, b in zip(nq, nk))
    assert f == 4 * 128 * 32 * pairs
    # a sequence with one new query sees every key
    assert roofline.prefill_visible_pairs(1, 1024, True) == 1024


def test_decode_bytes_of_workloads():
    b = roofline.decode_kv_bytes([32768] * 8, 8, 128)
    assert b == 2 * 8 * 8 * 32768 * 128 * 2 == 1073741824
    b4 = roofline.decode_kv_bytes([262144], 8, 128)
    assert b4 == b
    assert math.isclose(roofline.decode_partial_bytes(8, 32, 128, 16), 8 * 32 * 16 * 130 * 4)


def test_window_pairs_closed_form():
    # square, window W: rows i < W see i + 1 keys, the rest see W
    for n, w in ((4096, 1024), (100, 1), (100, 100), (37, 500)):
        wc = min(w, n)
        closed = wc * (wc + 1) // 2 + (n - wc) * wc
        assert roofline.prefill_visible_pairs(n, n, True, w) == closed
    assert roofline.prefill_visible_pairs(300, 300, True, 10**6) == roofline.prefill_visible_pairs(300, 300, True)
    # bottom-right alignment: 2 queries over 10 keys, W 3 -> keys 6..8 and 7..9
    assert roofline.prefill_visible_pairs(2, 10, True, 3) == 6
    assert roofline.window_prefill_flops(1, 1, 2, 10, 64, 3) == 4 * 64 * 6
