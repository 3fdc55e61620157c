"""Benchmark of the exact-attention hot path on GB300; prints ONE JSON line (rank 0).

Headline workload: causal bf16 prefill, B=4, 32 heads, Nq = Nk = 4096, d = 128 (outputs O bf16 and
fp32 LSE), measured as prefill TFLOP/s with causal FLOPs counted as half (4*d*Nq*Nk/2 per head).
The same line carries the decode KV-cache GB/s of the decode workloads (contiguous and paged), the
sliding-window prefill, the varlen append workload and the head-dim-256 prefill and decode in
``breakdown``, each with its own roofline, so that one run covers every step of the path (prefill
tiles, split-K decode + merge, paged gather, window, varlen dispatch, both d = 256 kernels).

Timing: W untimed warm-up steps, then K steps bracketed by a barrier and a device synchronize,
CUDA events on the launching stream; every workload's inputs are larger than L2 (129 MB), so no
flush is needed between steps. ``e2e`` repeats the headline through the host-buffer entry point
(``attn_fwd_host``) with pinned host buffers: the host-to-device copies of the inputs and the
device-to-host copies of O and LSE are inside the timed region (chunked and overlapped with the
kernels by the library). ``cpu_baseline`` times the fp64 oracle (as it stands) on a bounded sample.

``--impl reference`` times the oracle itself on the host cores as the reference arm (a bounded
sample of the headline workload per step). With ``--gpus N`` under torchrun every rank runs an
independent replica (the path is single-GPU; nothing is exchanged), ``value`` is the work of all
ranks divided by the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import exact_attention_flashattn_gb300 as bw  # noqa: E402
from exact_attention_flashattn_gb300 import roofline as rl  # noqa: E402
from exact_attention_flashattn_gb300 import workloads as wl  # noqa: E402

HEADLINE = "prefill_causal_b4_h32_n4096_d128"

# DRAM traffic of the dominant kernel from the committed ncu capture, per full launch, valid
# only while the kernel source is the profiled one (checked by hash); otherwise reported null.
PROFILED_TRAFFIC = {
    # the tcgen05 prefill kernel, the PTX wrappers it is built from and the host code that sizes
    # its item-list bands, hashed in this order
    "kernel_sources": [
        "exact_attention_flashattn_gb300/csrc/prefill_tc.cu",
        "exact_attention_flashattn_gb300/csrc/ptx.cuh",
        "exact_attention_flashattn_gb300/csrc/api.cu",
    ],
    "sha256": "4a42f06d2f3ffa639d3a5c8d525fda36bf81f8de4a32581b7c382824f6e3ded8",
    # (201.63 MB read + 46.83 MB written) at B=2, from the ncu capture summarised under profiles/,
    # scaled x2 to the B=4 launch: traffic grows with the number of (batch, head) units
    "bytes_per_launch": 496902144,
}
PROFILED_TRAFFIC_D256 = {
    # the head-dim-256 prefill kernel, its PTX wrappers and the band sizing, hashed in this order
    "kernel_sources": [
        "exact_attention_flashattn_gb300/csrc/prefill_tc256.cu",
        "exact_attention_flashattn_gb300/csrc/ptx.cuh",
        "exact_attention_flashattn_gb300/csrc/api.cu",
    ],
    "sha256": "ed382ad63bcd39cc126497cffc6c9355df4525849c2c11fe00c560ba319a12cf",
    # (201.60 MB read + 43.77 MB written) at B=2, from the ncu capture summarised under profiles/,
    # scaled x2 to the B=4 launch of prefill_causal_b4_h16_n4096_d256
    "bytes_per_launch": 490757120,
}
METRIC = "prefill TFLOP/s and decode KV GB/s, 1×GB300, as fraction of roofline"
# nominal GB300 figures, the second roofline basis: HBM3e bandwidth of about 8 TB/s and the dense
# (no 2:4 sparsity) bf16 tensor-core peak of 2.25 PFLOP/s
NOMINAL = {"hbm_gbs": 8000.0, "bf16_tflops": 2250.0}
L2_BYTES = 129 * 1024 * 1024


def profiled_traffic(spec=None):
    """Measured DRAM bytes per launch of a profiled kernel, or None once its sources changed."""
    import hashlib
    spec = PROFILED_TRAFFIC if spec is None else spec
    h = hashlib.sha256()
    for rel in spec["kernel_sources"]:
        p = os.path.join(ROOT, rel)
        if not os.path.exists(p):
            return None
        with open(p, "rb") as f:
            h.update(f.read())
    return spec["bytes_per_launch"] if h.hexdigest() == spec["sha256"] else None


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# ------------------------------------------------------------------ distributed plumbing


def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    """Largest value over all ranks (the slowest rank's time sets the job's time)."""
    if world <= 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank, world, ms_max):
    """Whole-job rate: the units all ranks processed divided by the slowest rank's time."""
    return units_per_rank * world / (ms_max * 1e-3)


# ------------------------------------------------------------------ clocks


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.dev = device_index
        self.proc = None
        # raw samples go to the temp directory; the bench line carries their summary
        self.path = os.path.join(tempfile.gettempdir(), f"bwattn_bench_clocks_rank{device_index}_{os.getpid()}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return None
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


# ------------------------------------------------------------------ timing helpers


def time_steps(fn, steps, warmup, world, stream):
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    n0 = bw.launch_count()
    for i in range(steps):
        starts[i].record(stream)
        fn()
        ends[i].record(stream)
    torch.cuda.synchronize()
    launches = bw.launch_count() - n0
    barrier(world)
    per = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    return per, launches


def cpu_baseline_prefill(seconds_budget=15.0):
    """fp64 oracle on whole heads of the headline workload (bounded: ~10-30 s of CPU work)."""
    import numpy as np
    import oracle
    w = wl.WORKLOADS[HEADLINE]
    q, k, v = wl.prefill_inputs(1, 4, 4, w.Nq, w.Nk, w.d, torch.bfloat16, seed=w.seed)
    qs, ks, vs = (x.float().numpy().astype(np.float64) for x in (q, k, v))
    heads, t = 0, 0.0
    while t < seconds_budget and heads < w.B * w.Hq:
        h = heads % 4
        t0 = time.perf_counter()
        oracle.attention(qs[:, h:h + 1], ks[:, h:h + 1], vs[:, h:h + 1], True, method="tiled", block=128)
        t += time.perf_counter() - t0
        heads += 1
    flops = rl.prefill_flops(1, heads, w.Nq, w.Nk, w.d, True)
    return {"value": flops / t / 1e12, "unit": "TFLOP/s", "cores": oracle.hardware_threads(), "kind": "oracle",
            "sample": f"{heads} whole heads (4096 causal rows, d=128) of the headline workload, tiled fp64 oracle, "
                      f"{t:.1f} s"}


# ------------------------------------------------------------------ reference arm


def run_reference(args, rank, world):
    import numpy as np
    import oracle
    if rank != 0:
        return
    w = wl.WORKLOADS[HEADLINE]
    q, k, v = wl.prefill_inputs(1, 1, 1, w.Nq, w.Nk, w.d, torch.bfloat16, seed=w.seed)
    qs, ks, vs = (x.float().numpy().astype(np.float64) for x in (q, k, v))
    step = lambda: oracle.attention(qs, ks, vs, True, method="tiled", block=128)  # noqa: E731
    for _ in range(args.warmup):
        step()
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        step()
        times.append(time.perf_counter() - t0)
    flops = rl.prefill_flops(1, 1, w.Nq, w.Nk, w.d, True)
    ms = 1e3 * statistics.mean(times)
    val = flops / (ms * 1e-3) / 1e12
    cores = oracle.hardware_threads()
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": HEADLINE, "sample": "one whole head (b=0, h=0: 4096 causal rows, d=128) per step",
                       "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "Nq": w.Nq, "Nk": w.Nk, "d": w.d, "causal": True},
            "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                             "sample": "one whole head of the headline workload per step, tiled fp64 oracle"},
            "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


# ------------------------------------------------------------------ single-part runs (profiling aid)


def r4(x):
    """4 significant digits (keeps the bench line short)."""
    return float(f"{x:.4g}")


def roofline_entry(bound, achieved, peaks, unit, **extra):
    """Roofline object on both bases: the measured peak (MEASURED_PEAKS.json, else the fallback)
    and the nominal one (8 TB/s HBM3e; 2.25 PFLOP/s dense bf16). A tensor-bound entry also
    carries the measured sustained bf16 figure (cuBLAS looped for seconds under the power cap),
    the fair denominator when many timed steps run the GPU into that cap."""
    key = "hbm_gbs" if bound == "hbm" else "bf16_tflops"
    out = {"bound": bound, "achieved": r4(achieved), "peak": peaks[key], "unit": unit,
           "frac": r4(achieved / peaks[key]), "peak_nominal": NOMINAL[key],
           "frac_nominal": r4(achieved / NOMINAL[key])}
    if bound == "tensor":
        out["peak_sustained"] = peaks["bf16_tflops_sustained"]
        out["frac_sustained"] = r4(achieved / peaks["bf16_tflops_sustained"])
    out.update(extra)
    return out


def decode_call(x, w, nk, ws, o, lse):
    """The decode entry point of a workload, as a closure over its inputs and outputs."""
    if w.kind == "decode":
        return lambda: bw.attn_decode(x["q"], x["kcache"], x["vcache"], nk, w.num_splits, workspace=ws, out=o,
                                      lse=lse)
    if w.kind == "decode_paged":
        return lambda: bw.attn_decode_paged(x["q"], x["k_pages"], x["v_pages"], x["block_table"], nk, w.num_splits,
                                            workspace=ws, out=o, lse=lse)
    if w.kind == "decode_fp8":
        return lambda: bw.attn_decode_fp8(x["q"], x["kcache"], x["vcache"], x["k_scale"], x["v_scale"], nk,
                                          w.num_splits, workspace=ws, out=o, lse=lse)
    return lambda: bw.attn_decode_paged_fp8(x["q"], x["k_pages"], x["v_pages"], x["k_scale"], x["v_scale"],
                                            x["block_table"], nk, w.num_splits, workspace=ws, out=o, lse=lse)


def bench_decode(name, args, world, stream, dev, peaks):
    """Decode KV-cache GB/s: every cached K and V element read once (bf16: 2 bytes, FP8: 1)."""
    x = wl.make(name, device=dev)
    w = x["w"]
    nk = x["nk"].to(dev)
    o = torch.empty_like(x["q"])
    lse = torch.empty((w.B, w.Hq), dtype=torch.float32, device=dev)
    ws = torch.empty(bw.decode_workspace_size(w.B, w.Hq, w.d, w.num_splits), dtype=torch.uint8, device=dev)
    per, _ = time_steps(decode_call(x, w, nk, ws, o, lse), args.steps, args.warmup, world, stream)
    ms = max_over_ranks(statistics.mean(per), world)
    fp8 = w.kind.endswith("fp8")
    kvb = rl.decode_kv_bytes([w.Nk] * w.B, w.Hkv, w.d, elem_bytes=1 if fp8 else 2)
    gbs = kvb / (ms * 1e-3) / 1e9
    out = {"GB/s": r4(gbs * world), "ms": r4(ms), "splits": w.num_splits,
           "roofline": roofline_entry("hbm", gbs, peaks, "GB/s", bytes=kvb)}
    del x, o, lse, ws, nk
    torch.cuda.empty_cache()
    return out


def bench_prefill(name, args, world, stream, dev, peaks):
    """Prefill TFLOP/s of a dense workload (causal counted as half; a window counts its visible
    pairs exactly)."""
    w = wl.WORKLOADS[name]
    x = wl.make(name, device=dev)
    W = w.extra.get("window", 0)
    o = torch.empty_like(x["q"])
    lse = torch.empty((w.B, w.Hq, w.Nq), dtype=torch.float32, device=dev)
    fn = lambda: bw.attn_fwd(x["q"], x["k"], x["v"], causal=True, window=W, out=o, lse=lse)  # noqa: E731
    per, _ = time_steps(fn, args.steps, args.warmup, world, stream)
    ms = max_over_ranks(statistics.mean(per), world)
    f = rl.window_prefill_flops(w.B, w.Hq, w.Nq, w.Nk, w.d, W) if W else rl.prefill_flops(w.B, w.Hq, w.Nq, w.Nk,
                                                                                          w.d, True)
    t = f / (ms * 1e-3) / 1e12
    traffic = profiled_traffic(PROFILED_TRAFFIC_D256) if w.d == 256 else None
    out = {"TFLOP/s": r4(t * world), "ms": r4(ms), "roofline": roofline_entry("tensor", t, peaks, "TFLOP/s",
                                                                             traffic=traffic)}
    del x, o, lse
    torch.cuda.empty_cache()
    return out


def bench_varlen(args, world, stream, dev, peaks):
    """Varlen append workload: measured time against the sum over sequences of
    max(FLOPs / bf16 peak, bytes / HBM peak), on both bases."""
    xv = wl.make("varlen_append_64seq_h32x8_d128", device=dev)
    wv = xv["w"]
    cq, ck = xv["cu_q"].to(dev), xv["cu_k"].to(dev)
    ov = torch.empty_like(xv["q"])
    lv = torch.empty((xv["q"].shape[0], wv.Hq), dtype=torch.float32, device=dev)
    mq, mk = max(xv["nq"]), max(xv["nk"])
    wsv = torch.empty(bw.varlen_workspace_size(wv.num_seqs, mk, wv.Hq, wv.Hkv, wv.d), dtype=torch.uint8, device=dev)
    fn = lambda: bw.attn_varlen(xv["q"], xv["k"], xv["v"], cq, ck, mq, mk, causal=True,  # noqa: E731
                                workspace=wsv, out=ov, lse=lv)
    per, _ = time_steps(fn, args.steps, args.warmup, world, stream)
    ms = max_over_ranks(statistics.mean(per), world)
    fv = rl.varlen_flops(xv["nq"], xv["nk"], wv.Hq, wv.d, True)
    roof = {}
    for tag, pk in (("", peaks), ("_nominal", NOMINAL)):
        roof["roofline_ms" + tag] = r4(1e3 * rl.varlen_roofline_seconds(xv["nq"], xv["nk"], wv.Hq, wv.Hkv, wv.d, True,
                                                                        pk["bf16_tflops"] * 1e12,
                                                                        pk["hbm_gbs"] * 1e9))
        roof["frac" + tag] = r4(roof["roofline_ms" + tag] / ms)
    out = {"TFLOP/s": r4(fv * world / (ms * 1e-3) / 1e12), "ms": r4(ms),
           "roofline": {"bound": "mixed", **roof}}
    del xv, ov, lv, wsv
    torch.cuda.empty_cache()
    return out


def run_case(args, world, stream, dev, peaks):
    out = {"case": args.case}
    if args.case == "prefill":
        w = wl.WORKLOADS[HEADLINE]
        B = args.batch or w.B
        q, k, v = wl.prefill_inputs(B, w.Hq, w.Hkv, w.Nq, w.Nk, w.d, torch.bfloat16, w.seed, device=dev)
        o = torch.empty_like(q)
        lse = torch.empty((B, w.Hq, w.Nq), dtype=torch.float32, device=dev)
        per, n = time_steps(lambda: bw.attn_fwd(q, k, v, causal=True, out=o, lse=lse), args.steps, args.warmup,
                            world, stream)
        ms = statistics.mean(per)
        out.update({"B": B, "ms": ms, "tflops": rl.prefill_flops(B, w.Hq, w.Nq, w.Nk, w.d, True) / ms / 1e9,
                    "launches": n})
    elif args.case == "window":
        w = wl.WORKLOADS["prefill_window_b4_h32_n4096_w1024_d128"]
        B, W = args.batch or w.B, w.extra["window"]
        q, k, v = wl.prefill_inputs(B, w.Hq, w.Hkv, w.Nq, w.Nk, w.d, torch.bfloat16, w.seed, device=dev)
        o = torch.empty_like(q)
        lse = torch.empty((B, w.Hq, w.Nq), dtype=torch.float32, device=dev)
        per, n = time_steps(lambda: bw.attn_fwd(q, k, v, causal=True, window=W, out=o, lse=lse), args.steps,
                            args.warmup, world, stream)
        ms = statistics.mean(per)
        out.update({"B": B, "window": W, "ms": ms,
                    "tflops": rl.window_prefill_flops(B, w.Hq, w.Nq, w.Nk, w.d, W) / ms / 1e9, "launches": n})
    elif args.case == "fp8":
        for name in ("decode_fp8_gqa_b8_h32x8_n32768_d128", "decode_fp8_paged_b8_h32x8_n32768_d128_p16",
                     "decode_fp8_long_b1_h64x8_n262144_d128"):
            out[name] = bench_decode(name, args, world, stream, dev, peaks)
    elif args.case == "paged":
        x = wl.make("decode_paged_b8_h32x8_n32768_d128_p16", device=dev)
        wd = x["w"]
        nk = x["nk"].to(dev)
        ws = torch.empty(bw.decode_workspace_size(wd.B, wd.Hq, wd.d, wd.num_splits), dtype=torch.uint8, device=dev)
        per, n = time_steps(lambda: bw.attn_decode_paged(x["q"], x["k_pages"], x["v_pages"], x["block_table"], nk,
                                                         wd.num_splits, workspace=ws), args.steps, args.warmup, world,
                            stream)
        ms = statistics.mean(per)
        out[wd.name] = {"ms": ms, "GB/s": rl.decode_kv_bytes([wd.Nk] * wd.B, wd.Hkv, wd.d) / ms / 1e6, "launches": n}
    elif args.case == "decode":
        for name in ("decode_gqa_b8_h32x8_n32768_d128", "decode_long_b1_h64x8_n262144_d128"):
            x = wl.make(name, device=dev)
            wd = x["w"]
            nk = x["nk"].to(dev)
            ws = torch.empty(bw.decode_workspace_size(wd.B, wd.Hq, wd.d, wd.num_splits), dtype=torch.uint8,
                             device=dev)
            per, n = time_steps(lambda: bw.attn_decode(x["q"], x["kcache"], x["vcache"], nk, wd.num_splits,
                                                       workspace=ws), args.steps, args.warmup, world, stream)
            ms = statistics.mean(per)
            out[name] = {"ms": ms, "GB/s": rl.decode_kv_bytes([wd.Nk] * wd.B, wd.Hkv, wd.d) / ms / 1e6,
                         "launches": n}
            del x, ws
            torch.cuda.empty_cache()
    elif args.case == "d256":
        w = wl.WORKLOADS["prefill_causal_b4_h16_n4096_d256"]
        B = args.batch or w.B
        q, k, v = wl.prefill_inputs(B, w.Hq, w.Hkv, w.Nq, w.Nk, w.d, torch.bfloat16, w.seed, device=dev)
        o = torch.empty_like(q)
        lse = torch.empty((B, w.Hq, w.Nq), dtype=torch.float32, device=dev)
        per, n = time_steps(lambda: bw.attn_fwd(q, k, v, causal=True, out=o, lse=lse), args.steps, args.warmup,
                            world, stream)
        ms = statistics.mean(per)
        out.update({"B": B, "d": w.d, "ms": ms, "tflops": rl.prefill_flops(B, w.Hq, w.Nq, w.Nk, w.d, True) / ms / 1e9,
                    "launches": n})
    elif args.case == "d256_decode":
        x = wl.make("decode_gqa_b8_h32x8_n16384_d256", device=dev)
        wd = x["w"]
        nk = x["nk"].to(dev)
        ws = torch.empty(bw.decode_workspace_size(wd.B, wd.Hq, wd.d, wd.num_splits), dtype=torch.uint8, device=dev)
        per, n = time_steps(lambda: bw.attn_decode(x["q"], x["kcache"], x["vcache"], nk, wd.num_splits, workspace=ws),
                            args.steps, args.warmup, world, stream)
        ms = statistics.mean(per)
        out[wd.name] = {"ms": ms, "GB/s": rl.decode_kv_bytes([wd.Nk] * wd.B, wd.Hkv, wd.d) / ms / 1e6, "launches": n}
    else:
        x = wl.make("varlen_append_64seq_h32x8_d128", device=dev)
        cq, ck = x["cu_q"].to(dev), x["cu_k"].to(dev)
        mq, mk = max(x["nq"]), max(x["nk"])
        wv = x["w"]
        ws = torch.empty(bw.varlen_workspace_size(wv.num_seqs, mk, wv.Hq, wv.Hkv, wv.d), dtype=torch.uint8,
                         device=dev)
        per, n = time_steps(lambda: bw.attn_varlen(x["q"], x["k"], x["v"], cq, ck, mq, mk, causal=True,
                                                   workspace=ws), args.steps, args.warmup, world, stream)
        ms = statistics.mean(per)
        out.update({"ms": ms, "tflops": rl.varlen_flops(x["nq"], x["nk"], wv.Hq, wv.d, True) / ms / 1e9,
                    "launches": n})
    print(json.dumps(out))


# ------------------------------------------------------------------ main arm


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="own", choices=["own", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-breakdown", action="store_true")
    ap.add_argument("--case", default="all",
                    choices=["all", "prefill", "window", "decode", "paged", "fp8", "varlen", "d256", "d256_decode"],
                    help="profiling aid: run one part only (no e2e, no CPU baseline)")
    ap.add_argument("--batch", type=int, default=0, help="profiling aid: override the prefill batch size")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)

    if args.impl == "reference":
        rank = int(os.environ.get("RANK", "0"))
        world = int(os.environ.get("WORLD_SIZE", "1"))
        run_reference(args, rank, world)
        return

    rank, world, local = dist_setup(args.gpus)
    peaks = load_peaks()
    stream = torch.cuda.current_stream()
    dev = torch.device("cuda", torch.cuda.current_device())

    if args.case != "all":
        run_case(args, world, stream, dev, peaks)
        return

    # ---------------- headline: causal prefill
    x = wl.make(HEADLINE, device=dev)
    w = x["w"]
    q, k, v = x["q"], x["k"], x["v"]
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.Hq, w.Nq), dtype=torch.float32, device=dev)
    step = lambda: bw.attn_fwd(q, k, v, causal=True, out=o, lse=lse)  # noqa: E731
    with ClockSampler(torch.cuda.current_device()) as clk:
        per, launches = time_steps(step, args.steps, args.warmup, world, stream)
    clocks = clk.summary()
    ms = max_over_ranks(statistics.mean(per), world)
    flops = rl.prefill_flops(w.B, w.Hq, w.Nq, w.Nk, w.d, True)
    value = job_throughput(flops, world, ms) / 1e12
    achieved = flops / (ms * 1e-3) / 1e12
    in_bytes = 3 * q.numel() * q.element_size()

    # ---------------- e2e through the public API with pinned host buffers
    hq, hk, hv = (t.cpu().pin_memory() for t in (q, k, v))
    ho = torch.empty(o.shape, dtype=o.dtype).pin_memory()
    hl = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()

    ws_host = torch.empty(bw.fwd_host_workspace_size(w.B, w.Hq, w.Hkv, w.Nq, w.Nk, w.d), dtype=torch.uint8,
                          device=dev)

    def e2e_step():
        # the host-buffer entry point: copies in, kernels and copies out, chunked and overlapped
        bw.attn_fwd_host(hq, hk, hv, causal=True, out=ho, lse=hl, workspace=ws_host, stream=stream)

    e2e_steps = max(3, min(args.steps, 10))
    per_e2e, _ = time_steps(e2e_step, e2e_steps, 3, world, stream)
    ms_e2e = max_over_ranks(statistics.mean(per_e2e), world)
    del hq, hk, hv
    e2e = {"value": flops * world / (ms_e2e * 1e-3) / 1e12, "unit": "TFLOP/s",
           "h2d_bytes_per_step": in_bytes, "d2h_bytes_per_step": o.numel() * o.element_size() + lse.numel() * 4}
    del x, q, k, v, o, lse
    torch.cuda.empty_cache()

    # ---------------- breakdown: every other workload, the decode and varlen ones last so that
    # they sit in the end of the line (compact entries, 4 significant digits)
    breakdown = {}
    if not args.no_breakdown:
        for name in ("prefill_causal_b4_h16_n4096_d256", "prefill_window_b4_h32_n4096_w1024_d128",
                     "prefill_causal_b4_h32_n4096_d64", "prefill_causal_b4_h32x8_n4096_d128"):
            breakdown[name] = bench_prefill(name, args, world, stream, dev, peaks)
        breakdown["decode_gqa_b8_h32x8_n16384_d256"] = bench_decode("decode_gqa_b8_h32x8_n16384_d256", args, world,
                                                                    stream, dev, peaks)
        for name in ("decode_fp8_gqa_b8_h32x8_n32768_d128", "decode_fp8_paged_b8_h32x8_n32768_d128_p16",
                     "decode_fp8_long_b1_h64x8_n262144_d128", "decode_paged_b8_h32x8_n32768_d128_p16"):
            breakdown[name] = bench_decode(name, args, world, stream, dev, peaks)
        breakdown["varlen_append_64seq_h32x8_d128"] = bench_varlen(args, world, stream, dev, peaks)
        for name in ("decode_long_b1_h64x8_n262144_d128", "decode_gqa_b8_h32x8_n32768_d128"):
            breakdown[name] = bench_decode(name, args, world, stream, dev, peaks)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline_prefill()

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": HEADLINE, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "Nq": w.Nq, "Nk": w.Nk, "d": w.d,
                       "causal": True, "flops_per_step": flops, "flop_convention": "causal counted as half",
                       "l2": f"inputs larger than L2 ({in_bytes / 1e6:.0f} MB of Q/K/V per step), no flush",
                       "parallelism": "replicas" if world > 1 else "single GPU"},
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                         "frac": achieved / peaks["bf16_tflops"], "traffic": profiled_traffic(),
                         "peak_source": f"{peaks['source']} bf16 burst",
                         "peak_nominal": NOMINAL["bf16_tflops"], "frac_nominal": achieved / NOMINAL["bf16_tflops"]},
            "e2e": e2e, "gpu_launches": launches, "clocks": clocks, "cpu_baseline": cpu, "breakdown": breakdown,
        }
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
