"""Benchmark of the Mamba-2 layer forward on GB300.

Headline: batch-1 decode tokens/s of the Nemotron-H-8B-like layer (hidden 4096,
128 heads x 64, d_state 128, 8 groups, conv 4; FP8 E4M3 128x128 block-scaled
in_proj [18560x4096] and out_proj [4096x8192]), one step = one token through
all eight steps of the layer.  Inputs are seeded synthetic data resident in
HBM.  To keep the timed working set above the L2 size, the steps rotate over
`replicas` copies of the layer (weights + per-sequence state), as consecutive
layers of a deep model would.

Also reported (extra keys): batch-64 decode tokens/s of the same layer and
1024-token prefill tokens/s, per-kernel times from the library's event trace,
the roofline of the dominant kernel, an end-to-end number through the C ABI
with host buffers, and the CPU oracle timed on a bounded sample.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
L2_BYTES_NOMINAL = 129 * 2 ** 20


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--no-extras", action="store_true", help="headline only (skip b64/prefill/e2e/cpu legs)")
    p.add_argument("--quick", action="store_true", help="fewer steps in the extra legs (profiling runs)")
    return p.parse_args()


def layer_bytes_per_token(d, B):
    """Algorithmic HBM bytes of one decode step for B sequences."""
    d_inner = d["nheads"] * d["head_dim"]
    d_xbc = d_inner + 2 * d["n_groups"] * d["d_state"]
    n_in = d_inner + d_xbc + d["nheads"]
    hid = d["hidden"]
    w_in = n_in * hid + math.ceil(n_in / 128) * math.ceil(hid / 128) * 2
    w_out = hid * d_inner + math.ceil(hid / 128) * math.ceil(d_inner / 128) * 2
    params = hid * 2 + d_xbc * d["d_conv"] * 2 + d_xbc * 2 + 3 * d["nheads"] * 4 + d_inner * 2
    state = B * d["nheads"] * d["head_dim"] * d["d_state"] * 4 * 2          # read + write
    conv = B * d_xbc * 2 * d["d_conv"]                                       # 3 slots read + 1 written
    io = B * hid * 2 * 2                                                     # hidden in + out
    return w_in + w_out + params + state + conv + io


def inproj_bytes(d, B):
    d_inner = d["nheads"] * d["head_dim"]
    d_xbc = d_inner + 2 * d["n_groups"] * d["d_state"]
    n_in = d_inner + d_xbc + d["nheads"]
    hid = d["hidden"]
    return (n_in * hid + math.ceil(n_in / 128) * math.ceil(hid / 128) * 2 + B * hid * 2 + B * n_in * 2
            + B * d_xbc * 2 * d["d_conv"] + d_xbc * (d["d_conv"] + 1) * 2)


def sources_sha256(paths) -> str:
    import hashlib
    h = hashlib.sha256()
    for rel in paths:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def captured_traffic(kernel: str, workload: str):
    """DRAM bytes (read + write) per launch of `kernel` on `workload` from the
    ncu capture recorded in profiles/traffic.txt, or None when there is none or
    the kernel's sources changed since it was taken (the line stores their
    sha256)."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    for line in open(path):
        f = line.split()
        if len(f) != 5 or line.startswith("#") or f[0] != kernel or f[1] != workload:
            continue
        try:
            if sources_sha256(f[3].split(",")) == f[4]:
                return float(f[2])
        except OSError:
            return None
    return None


def max_over_ranks(x: float, world: int, device="cpu") -> float:
    """Max of a per-rank scalar over all ranks (all-reduce MAX); x itself at world 1."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_rank: float, world: int, ms_max: float) -> float:
    """Whole-job throughput: the units all ranks processed over the slowest rank's time."""
    return world * units_per_rank / (ms_max / 1e3)


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            j = json.load(open(p))
            hbm = j.get("hbm_gbs") or j.get("hbm_GBps")
            return float(hbm), "measured", j
        except Exception:
            pass
    return FALLBACK_HBM_GBS, "fallback", {}


class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons while the timed region runs."""

    def __init__(self, index: int):
        self.index = index
        self.rows = []
        self.proc = None

    def __enter__(self):
        q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={q}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            t0 = time.time()
            while not self.rows and time.time() - t0 < 3.0 and self.proc.poll() is None:
                time.sleep(0.01)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append([x.strip() for x in line.split(",")])

    def __exit__(self, *a):
        time.sleep(0.12)  # one more sample after the timed region
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if not self.rows:
            return None
        sm = [float(r[0]) for r in self.rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows for i in range(4) if len(r) > 4 + i and r[4 + i] == "Active"})
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.rows)}


def oracle_decode_rate(budget_s: float):
    """The CPU oracle as it stands: decode tokens of the 8B-like layer, B=1."""
    from mamba_ssm_layer_gb300 import synth
    from oracle import oracle
    lay = synth.make_layer(synth.NEMOTRON_H_8B, synth.WL_8B_DECODE_B1)
    L = oracle.OracleLayer(lay)
    st = L.new_state()
    n = 0
    t0 = time.perf_counter()
    while True:
        hid = synth.make_hidden(1, 4096, synth.WL_8B_DECODE_B1, 0, n)
        L.run(hid, *st)
        n += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    cores = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    return n / dt, n, dt, cores


def run_reference(args, rank, world):
    """Reference arm: the CPU oracle, timed on this host's cores."""
    if rank != 0:
        return
    from mamba_ssm_layer_gb300 import synth
    from oracle import oracle
    oracle.build()
    lay = synth.make_layer(synth.NEMOTRON_H_8B, synth.WL_8B_DECODE_B1)
    L = oracle.OracleLayer(lay)
    st = L.new_state()
    for w in range(args.warmup):
        L.run(synth.make_hidden(1, 4096, synth.WL_8B_DECODE_B1, 1, w), *st)
    t0 = time.perf_counter()
    for k in range(args.steps):
        L.run(synth.make_hidden(1, 4096, synth.WL_8B_DECODE_B1, 2, k), *st)
    dt = time.perf_counter() - t0
    v = args.steps / dt
    cores = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    print(json.dumps({
        "impl": "reference", "metric": "decode tokens/s (Mamba-2 layer, batch 1)", "value": v,
        "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": {"workload": "nemotron_h_8b_like_decode_b1", "batch": 1},
        "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"{args.steps} sequential decode tokens of the 8B-like layer"},
        "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    args = parse()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return

    import torch
    import torch.distributed as dist
    from __graft_entry__ import build
    from mamba_ssm_layer_gb300 import abi, synth
    from mamba_ssm_layer_gb300.layer import DeviceLayer, to_dev

    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", torch.cuda.current_device())
    if rank == 0:
        build()
    if world > 1:
        dist.barrier()
    abi.lib()

    def barrier():
        if world > 1:
            dist.barrier()

    d = synth.NEMOTRON_H_8B
    B = 1
    lay = synth.make_layer(d, synth.WL_8B_DECODE_B1)
    base = DeviceLayer(lay)
    per_rep = layer_bytes_per_token(d, B)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size or L2_BYTES_NOMINAL
    # replicas (weights + state) so the rotating working set is >= 8x L2 and the
    # per-sequence states alone exceed L2
    state_b = B * d["nheads"] * d["head_dim"] * d["d_state"] * 4
    R = max(3, math.ceil(8 * l2 / per_rep), math.ceil(1.5 * l2 / state_b))
    reps = []
    for r in range(R):
        dl = DeviceLayer(lay) if r == 0 else _clone_layer(base, torch)
        reps.append((dl, dl.new_state(B)))
    ws = base.workspace(B, 0)
    K, W = args.steps, args.warmup
    hiddens = [to_dev(synth.make_hidden(B, d["hidden"], synth.WL_8B_DECODE_B1, rank, i)) for i in range(64)]

    # Each step hints the layer that follows it (the next replica, as the next
    # layer of a model): the first DeviceLayer.AHEAD_BYTES of that layer's
    # in_proj weights are pulled toward L2 during the step's out_proj.
    hint = {"on": True}

    def step(i):
        dl, st = reps[i % R]
        dl.decode(hiddens[i % 64], st, ws, ahead=reps[(i + 1) % R][0] if hint["on"] else None)

    for i in range(W):
        step(i)
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    launches0 = abi.m2_launch_count()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(torch.cuda.current_device()) as clk:
        e0.record()
        for i in range(K):
            step(W + i)
        e1.record()
        torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    launches = abi.m2_launch_count() - launches0
    ms_eager = max_over_ranks(e0.elapsed_time(e1), world, dev)
    eager = {"value": job_rate(K * B, world, ms_eager), "ms_per_step": ms_eager / K, "steps": K}

    # The same steps replayed from a CUDA graph: one pass over the replicas is
    # captured once (the library's launches, with their programmatic-dependent
    # edges) and replayed, as a serving loop would run a fixed decode step;
    # this removes the host's per-launch cost from the timed region.
    graph_info, ms, K_run, clk_g = None, ms_eager, K, None
    try:
        cap = torch.cuda.Stream()
        cap.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            for i in range(R):
                step(W + i)
        torch.cuda.current_stream().wait_stream(cap)
        reps_g = max(1, round(K / R))
        g.replay()
        torch.cuda.synchronize()
        barrier()
        torch.cuda.synchronize()
        with ClockSampler(torch.cuda.current_device()) as clk_g:
            e0.record()
            for _ in range(reps_g):
                g.replay()
            e1.record()
            torch.cuda.synchronize()
        barrier()
        torch.cuda.synchronize()
        ms_g = max_over_ranks(e0.elapsed_time(e1), world, dev)
        graph_info = {"value": job_rate(reps_g * R * B, world, ms_g), "ms_per_step": ms_g / (reps_g * R),
                      "steps": reps_g * R, "steps_per_graph": R}
        if graph_info["value"] > eager["value"]:
            ms, K_run = ms_g, reps_g * R
        # the same graph without the L2 hint, for comparison
        hint["on"] = False
        g2 = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g2, stream=cap):
            for i in range(R):
                step(W + i)
        torch.cuda.current_stream().wait_stream(cap)
        hint["on"] = True
        g2.replay()
        torch.cuda.synchronize()
        e0.record()
        for _ in range(reps_g):
            g2.replay()
        e1.record()
        torch.cuda.synchronize()
        ms_g2 = max_over_ranks(e0.elapsed_time(e1), world, dev)
        graph_info["without_l2_hint"] = {"value": job_rate(reps_g * R * B, world, ms_g2),
                                         "ms_per_step": ms_g2 / (reps_g * R)}
    except Exception as ex:  # capture unsupported here: the eager number stands
        graph_info = {"error": f"{type(ex).__name__}: {ex}"[:200]}
    ms_step = ms / K_run
    value = job_rate(K_run * B, world, ms)
    use_graph = K_run != K or ms != ms_eager
    launches_per_step = launches / K

    # per-kernel device time of the same steps, from the library's event trace
    # (events between launches serialise them; these are per-launch durations)
    abi.trace_begin(16 * K)
    for i in range(K):
        step(W + K + i)
    tr = abi.trace_end()
    # the dominant kernel: the single-launch step when it ran, else the in_proj GEMV
    if "decode_step_fused" in tr:
        rk, rk_desc, rk_bytes = "decode_step_fused", "decode_step_fused (whole layer step, one launch)", per_rep
    else:
        rk, rk_desc, rk_bytes = "gemv_fp8_inproj_conv", "gemv_fp8 (in_proj, conv1d fused)", inproj_bytes(d, B)
    rk_ms, rk_n = tr.get(rk, (0.0, 0))
    tr_rk = rk_ms / rk_n if rk_n else None
    hbm_peak, peak_src, peaks = measured_peaks()
    roof = None
    if tr_rk:
        achieved = rk_bytes / (tr_rk / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s", "frac": achieved / hbm_peak,
                "traffic": captured_traffic(rk, "decode_b1"), "kernel": rk_desc, "bytes_per_launch": rk_bytes,
                "launch_us": tr_rk * 1e3, "peak_source": f"{peak_src} hbm_gbs"}

    # the same steps in the other form of the batch-1 step (eager), for comparison
    prev = abi.m2_set_fused_decode(not ("decode_step_fused" in tr))
    Kc = min(K, 200)
    for i in range(3):
        step(i)
    torch.cuda.synchronize()
    e0.record()
    for i in range(Kc):
        step(W + i)
    e1.record()
    torch.cuda.synchronize()
    abi.m2_set_fused_decode(prev)
    msc = max_over_ranks(e0.elapsed_time(e1), world, dev)
    alt = {"value": job_rate(Kc * B, world, msc), "ms_per_step": msc / Kc, "steps": Kc,
           "launch": ("eager, three kernels per step" if "decode_step_fused" in tr
                      else "eager, one cooperative kernel per step (m2_set_fused_decode)")}

    out = {
        "metric": "decode tokens/s (Mamba-2 layer, batch 1)", "value": value, "unit": "tokens/s",
        "n_gpus": world, "steps": K_run, "warmup": W, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3 weights x bf16 activations, fp32 accumulate", "data": "synthetic",
        "config": {"workload": "nemotron_h_8b_like_decode_b1", "batch": B, "hidden": 4096, "nheads": 128,
                   "head_dim": 64, "d_state": 128, "n_groups": 8, "d_conv": 4,
                   "weights": "e4m3 128x128 block-scaled, bf16 scales", "activations": "bf16",
                   "l2": f"rotating {R} layer replicas ({R * per_rep / 1e9:.2f} GB) > L2 {l2 / 2**20:.0f} MiB",
                   "parallelism": f"replicas x{world}",
                   "launch": ("cuda_graph replay of the library's launches" if use_graph else "eager calls")
                   + "; each step hints the next layer (its first in_proj weights pulled toward L2 during the"
                   " step's out_proj: mamba2_layer_decode_prefetch)"},
        "step_hbm": {"bytes_per_token": per_rep, "gbs": per_rep / (ms_step / 1e3) / 1e9,
                     "frac": per_rep / (ms_step / 1e3) / 1e9 / hbm_peak},
        "roofline": roof,
        "gpu_launches": int(round(launches_per_step * K_run)),
        "eager": eager,
        "graph": graph_info,
        "other_form": alt,
        "kernels_ms_per_step": {k: v[0] / K for k, v in tr.items()},
        "clocks": (clk_g.summary() if use_graph and clk_g is not None else clk.summary()),
    }

    if not args.no_extras:
        out["decode_tiny"] = _bench_tiny(torch, synth, DeviceLayer, to_dev, 100 if args.quick else 400)
        out["decode_b64"] = _bench_b64(torch, synth, DeviceLayer, to_dev, abi, lay, 8 if args.quick else 64)
        out["prefill_1k"] = _bench_prefill(torch, synth, DeviceLayer, to_dev, abi, 2 if args.quick else 5)
        out["prefill_1k_w8a8"] = _bench_prefill(torch, synth, DeviceLayer, to_dev, abi, 2 if args.quick else 5,
                                                w8a8=True)
        out["stack8"] = _bench_stack8(torch, synth, to_dev)
        out["e2e"] = _bench_e2e(torch, synth, reps, ws, d, B, min(K, 100))
        if rank == 0:
            v, n, dt, cores = oracle_decode_rate(4.0 if args.quick else 15.0)
            out["cpu_baseline"] = {"value": v, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                                   "sample": f"{n} sequential batch-1 decode tokens of the 8B-like layer ({dt:.1f} s)"}
    if abi.m2_device_status() != 0:
        out["device_status"] = abi.m2_device_status()
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        dist.destroy_process_group()


def _clone_layer(base, torch):
    import copy
    new = copy.copy(base)
    new.t = {k: (None if v is None else v.clone()) for k, v in base.t.items()}
    from mamba_ssm_layer_gb300 import abi
    t = new.t
    d = base.dims_dict
    new.struct = abi.M2Layer(
        t["norm_w"].data_ptr(),
        abi.weight_struct(t["in_w"], t["in_s"], base.n_in, d["hidden"], base.struct.in_proj.fmt),
        t["conv_w"].data_ptr(), t["conv_b"].data_ptr(), t["A_log"].data_ptr(), t["D"].data_ptr(),
        t["dt_bias"].data_ptr(), t["gnorm_w"].data_ptr(),
        abi.weight_struct(t["out_w"], t["out_s"], d["hidden"], base.d_inner, base.struct.out_proj.fmt))
    return new


def _bench_b64(torch, synth, DeviceLayer, to_dev, abi, lay, steps):
    d = synth.NEMOTRON_H_8B
    B = 64
    dl = DeviceLayer(lay)
    sts = [dl.new_state(B) for _ in range(2)]  # 2 x 268 MB of state > L2
    ws = dl.workspace(B, 0)
    hs = [to_dev(synth.make_hidden(B, d["hidden"], synth.WL_8B_DECODE_B64, 0, i)) for i in range(4)]
    for i in range(64):  # 32 warm-up steps of random inputs for each of the two state sets
        dl.decode(hs[i % 4], sts[i % 2], ws)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(steps):
        dl.decode(hs[i % 4], sts[i % 2], ws)
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    per = layer_bytes_per_token(d, B)
    hbm, _, _ = measured_peaks()
    abi.trace_begin(16 * steps)
    for i in range(steps):
        dl.decode(hs[i % 4], sts[i % 2], ws)
    tr = abi.trace_end()
    return {"value": B / (ms / 1e3), "unit": "tokens/s", "ms_per_step": ms, "batch": B,
            "hbm_gbs": per / (ms / 1e3) / 1e9, "hbm_frac": per / (ms / 1e3) / 1e9 / hbm,
            "kernels_ms_per_step": {k: v[0] / steps for k, v in tr.items()}}


def _bench_tiny(torch, synth, DeviceLayer, to_dev, steps):
    """Tiny layer (hidden 256), batch-1 decode: launch-latency bound, L2-resident."""
    d = synth.TINY
    lay = synth.make_layer(d, synth.WL_TINY_DECODE)
    dl = DeviceLayer(lay)
    st = dl.new_state(1)
    ws = dl.workspace(1, 0)
    hs = [to_dev(synth.make_hidden(1, d["hidden"], synth.WL_TINY_DECODE, 3, i)) for i in range(16)]
    for i in range(10):
        dl.decode(hs[i % 16], st, ws)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(steps):
        dl.decode(hs[i % 16], st, ws)
    e1.record()
    torch.cuda.synchronize()
    ms_eager = e0.elapsed_time(e1) / steps
    ms, launch = ms_eager, "eager"
    try:  # the same steps replayed from a CUDA graph of 16 steps
        cap = torch.cuda.Stream()
        cap.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            for i in range(16):
                dl.decode(hs[i], st, ws)
        torch.cuda.current_stream().wait_stream(cap)
        reps = max(1, steps // 16)
        g.replay()
        torch.cuda.synchronize()
        e0.record()
        for _ in range(reps):
            g.replay()
        e1.record()
        torch.cuda.synchronize()
        ms_g = e0.elapsed_time(e1) / (reps * 16)
        if ms_g < ms:
            ms, launch = ms_g, "cuda_graph replay"
    except Exception:  # capture unsupported: the eager number stands
        pass
    return {"value": 1.0 / (ms / 1e3), "unit": "tokens/s", "ms_per_step": ms, "batch": 1, "launch": launch,
            "ms_per_step_eager": ms_eager, "bound": "launch latency (weights and state L2-resident)"}


def _bench_prefill(torch, synth, DeviceLayer, to_dev, abi, reps, w8a8=False):
    """1024-token prefill of one sequence (w8a8: the FP8-activation arm)."""
    d = synth.NEMOTRON_H_8B
    T = 1024
    lay = synth.make_layer(d, synth.WL_8B_PREFILL_1K)
    dl = DeviceLayer(lay)
    ws = dl.workspace_varlen(1, T)
    hid = synth.make_hidden(T, d["hidden"], synth.WL_8B_PREFILL_1K, 0, 0)
    xs = [to_dev(hid) for _ in range(reps + 1)]
    st = dl.new_state(1)
    s1 = (st[0][:1], st[1][:1], st[2][:1])

    def run(x):
        dl.prefill_varlen(x, [0, T], s1, ws, w8a8=w8a8)

    run(xs[0])
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(reps):
        run(xs[i + 1])
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / reps
    abi.trace_begin(64)
    run(xs[0])
    tr = abi.trace_end()
    gemm_ms = tr.get("gemm_tc", (0.0, 0))[0]
    flops = 2.0 * T * (synth.derived(d)["n_in"] * d["hidden"] + d["hidden"] * synth.derived(d)["d_inner"])
    return {"value": T / (ms / 1e3), "unit": "tokens/s", "ms_per_prefill": ms, "tokens": T,
            "arm": "w8a8 (E4M3 activations, kind::f8f6f4)" if w8a8 else "w8a16 (bf16 activations, kind::f16)",
            "gemm_tflops": flops / (gemm_ms / 1e3) / 1e12 if gemm_ms else None,
            "kernels_ms": {k: v[0] for k, v in tr.items()}}


def _bench_stack8(torch, synth, to_dev):
    """Eight-layer stack (layers 2 and 5 BF16): 16 prompts of 64..512 tokens
    prefilled together (one varlen call per layer), then 256 decode steps of
    all 16 sequences.  Inputs (prompts and the per-step decode rows) are
    resident on the device before the timed region; the stack's 1.1 GB of
    weights and 0.5 GB of states exceed L2.  Timed once after an untimed run."""
    from mamba_ssm_layer_gb300.stack import DeviceStack
    spec, d = synth.STACK8, synth.NEMOTRON_H_8B
    hid = d["hidden"]
    lens = synth.stack_prompt_lengths(spec)
    S, steps = spec["n_seqs"], spec["decode_steps"]
    stk = DeviceStack(synth.stack_layers(d, spec))
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    ws = stk.workspace(S, int(cu[-1]), S)
    prompts = to_dev(np.concatenate([synth.stack_prompt(s, int(lens[s]), hid) for s in range(S)]))
    rows = to_dev(np.stack([synth.stack_decode_rows(k, S, hid) for k in range(steps)]))
    res = {}
    for rep in range(2):
        st = stk.new_state(S)
        xs = prompts.clone()
        rw = rows.clone()
        torch.cuda.synchronize()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        ev[0].record()
        stk.prefill_varlen(xs, cu, st, ws)  # all prompts, one call per layer
        ev[1].record()
        for k in range(steps):
            stk.decode(rw[k], st, ws)
        ev[2].record()
        torch.cuda.synchronize()
        pre, dec = ev[0].elapsed_time(ev[1]), ev[1].elapsed_time(ev[2])
        ntok = int(lens.sum()) + S * steps
        res = {"value": ntok / ((pre + dec) / 1e3), "unit": "tokens/s", "ms_total": pre + dec,
               "prefill_tokens_per_s": int(lens.sum()) / (pre / 1e3), "prefill_ms": pre,
               "decode_tokens_per_s": S * steps / (dec / 1e3), "decode_ms": dec,
               "decode_ms_per_step": dec / steps, "prompt_tokens": int(lens.sum()), "seqs": S,
               "decode_steps": steps, "layers": spec["n_layers"], "bf16_layers": list(spec["bf16_layers"])}
    return res


def _bench_e2e(torch, synth, reps, ws, d, B, K):
    """Same decode metric through the C ABI with host buffers: per step the
    hidden row is copied from pinned host memory to the device and the layer
    output back, inside the timed region.  Three forms are timed and the
    fastest is reported: (a) cudaMemcpyAsync and kernels on one stream; (b)
    copies on a second stream, double-buffered, so that step i+1's input lands
    while step i runs and step i's output drains while step i+1 runs (events
    order them); (c) the library's m2_copy kernels on the one stream, which keep
    the launch chain unbroken."""
    R = len(reps)
    host_in = [torch.from_numpy(synth.make_hidden(B, d["hidden"], 9, 9, i).view(np.int16)).pin_memory()
               for i in range(8)]
    host_out = [torch.empty((B, d["hidden"]), dtype=torch.int16).pin_memory() for _ in range(2)]
    devs = [torch.empty((B, d["hidden"]), dtype=torch.int16, device="cuda") for _ in range(2)]
    nbytes = B * d["hidden"] * 2
    comp = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def one_stream():
        e0.record()
        for i in range(K):
            devs[0].copy_(host_in[i % 8], non_blocking=True)
            dl, st = reps[i % R]
            dl.decode(devs[0], st, ws, ahead=reps[(i + 1) % R][0])
            host_out[0].copy_(devs[0], non_blocking=True)
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / K

    def two_streams():
        copy = torch.cuda.Stream()
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_dec = [torch.cuda.Event() for _ in range(2)]
        ev_out = [torch.cuda.Event() for _ in range(2)]
        e0.record(comp)
        copy.wait_stream(comp)
        with torch.cuda.stream(copy):
            devs[0].copy_(host_in[0], non_blocking=True)
            ev_in[0].record(copy)
        for i in range(K):
            b, nb = i % 2, (i + 1) % 2
            if i + 1 < K:
                with torch.cuda.stream(copy):
                    if i >= 1:
                        copy.wait_event(ev_out[nb])  # step i-1's output has left devs[nb]
                    devs[nb].copy_(host_in[(i + 1) % 8], non_blocking=True)
                    ev_in[nb].record(copy)
            comp.wait_event(ev_in[b])
            dl, st = reps[i % R]
            dl.decode(devs[b], st, ws, ahead=reps[(i + 1) % R][0])
            ev_dec[b].record(comp)
            with torch.cuda.stream(copy):
                copy.wait_event(ev_dec[b])
                host_out[b].copy_(devs[b], non_blocking=True)
                ev_out[b].record(copy)
        comp.wait_event(ev_out[(K - 1) % 2])
        e1.record(comp)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / K

    def copy_kernels():
        # the library's staging copy (a kernel in the same launch chain)
        from mamba_ssm_layer_gb300 import abi
        e0.record()
        for i in range(K):
            abi.m2_copy(devs[0], host_in[i % 8], nbytes, comp)
            dl, st = reps[i % R]
            dl.decode(devs[0], st, ws, ahead=reps[(i + 1) % R][0])
            abi.m2_copy(host_out[0], devs[0], nbytes, comp)
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / K

    forms = {"one stream, cudaMemcpyAsync": one_stream, "copy stream, double-buffered": two_streams,
             "one stream, m2_copy kernels": copy_kernels}
    for f in forms.values():  # warm every form
        f()
    times = {k: f() for k, f in forms.items()}
    best = min(times, key=times.get)
    ms = times[best]
    return {"value": B / (ms / 1e3), "unit": "tokens/s", "h2d_bytes_per_step": nbytes, "d2h_bytes_per_step": nbytes,
            "ms_per_step": ms, "form": best, "ms_per_step_by_form": times}


if __name__ == "__main__":
    main()
