"""Throughput of the fused 4-bit GEMV on GB300: weight-stream GB/s and the
fraction of the HBM roofline.

Workload (one step): a Qwen3-4B-shaped decode layer at N = 1 — the QKV triple
(Q4_K 4096x2560, Q4_K 1024x2560, Q6_K 1024x2560), Wo (Q4_K 2560x4096) fused
with the fp16 residual add, the gate/up pair (2 x Q4_K 9728x2560) and down
(Q6_K 2560x9728): 63,866,880 packed weight bytes.  Steps rotate over 36
distinct synthetic layers (2.3 GB, far above the 129 MB L2), so every step
streams its weights from HBM.  Inputs are resident in HBM when timing starts;
the timed steps are one CUDA graph replay.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Prints one JSON line.  Under torchrun (N > 1) every rank runs the same
workload on its own GPU (replicas; weak scaling) and rank 0 reports the sum.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

N_LAYERS = 36
METRIC = "weight-stream GB/s and % of GB300 HBM roofline for 4-bit GEMV, N=1..32"
WORKLOAD = "qwen3_4b_decode_layer_n1"


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 20 ms by one
    background nvidia-smi process; only samples taken inside the timed window
    (mark_start / mark_end) are summarised."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.lines = []
        self.proc = None
        self.t0 = self.t1 = None
        self._reader = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)

            def read():
                for line in self.proc.stdout:
                    self.lines.append((time.time(), line.strip()))
            self._reader = threading.Thread(target=read, daemon=True)
            self._reader.start()
            time.sleep(0.3)  # first samples before the timed window opens
        except Exception:
            self.proc = None
        return self

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()
        # keep sampling briefly so the window's last interval is covered
        time.sleep(0.05)

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        inside = [l for (t, l) in self.lines if self.t0 is not None and self.t0 - 0.03 <= t <= (self.t1 or 0) + 0.03]
        rows = [[v.strip() for v in l.split(",")] for l in inside]
        rows = [r for r in rows if len(r) >= 9]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = sorted(float(r[1]) for r in rows)
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for name, v in zip(names, r[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": float(rows[0][2]),
                "reasons": sorted(reasons), "samples": len(rows),
                "power_w_max": max(float(r[3]) for r in rows if r[3].replace('.', '', 1).isdigit())}


def _kernel_source_sha():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "skinny_gemm_q4_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f.endswith((".cu", ".cuh")):
            with open(os.path.join(csrc, f), "rb") as fh:
                h.update(fh.read())
    return h.hexdigest()[:16]


def _traffic_record():
    """DRAM bytes per launch of the dominant kernel from the committed ncu
    summary, or None if the kernel sources changed since it was taken."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        rec = json.load(f)
    if rec.get("source_sha") != _kernel_source_sha():
        return None
    return rec.get("dram_bytes_per_launch")


def aggregate_ranks(ms_local, world, wbytes, steps, dist=None, device=None):
    """Whole-job timing of a replicated run: the slowest rank's time (max
    over ranks) and the bytes all ranks streamed divided by it, in GB/s."""
    import torch
    ms = float(ms_local)
    if dist is not None:
        t = torch.tensor([ms], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    return ms, world * wbytes * steps / (ms / 1e3) / 1e9


def layer_weight_bytes():
    from skinny_gemm_q4_gb300 import synth
    return sum(M * synth.row_bytes(qt, K) for _, qt, M, K in synth.LAYER)


# ---------------------------------------------------------------- reference

def run_reference(args):
    """The CPU oracle on a bounded sample of the same workload, timed on this
    host's cores (single-threaded: the oracle as it stands)."""
    import numpy as np

    import oracle
    from skinny_gemm_q4_gb300 import synth
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    oracle.build()
    # Bounded sample: every frac-th row of each matrix of one layer, frac chosen
    # so that warmup + steps take about a minute on this host in total.
    full = []
    for i, (role, qt, M, K) in enumerate(synth.LAYER):
        w, sc, g = synth.weights(qt, M, K, seed=0, stream=100 + i)
        x = synth.activations(1, K, seed=0, stream=200 + i)
        full.append((qt, w, M, K, x))

    def make(frac):
        mats = [(qt, w, M, K, np.arange(0, M, frac), x) for qt, w, M, K, x in full]
        nbytes = sum(len(r) * synth.row_bytes(qt, K) for qt, w, M, K, r, x in mats)
        return mats, nbytes

    def step(mats):
        for qt, w, M, K, rows, x in mats:
            oracle.qgemv(qt, w, M, K, x, rows=rows)

    probe, probe_bytes = make(256)
    t0 = time.perf_counter()
    step(probe)
    sec_per_byte = (time.perf_counter() - t0) / probe_bytes
    budget = 60.0 / (args.steps + args.warmup)
    frac = 16
    while frac < 4096 and make(frac)[1] * sec_per_byte > budget:
        frac *= 2
    mats, sample_bytes = make(frac)
    for _ in range(args.warmup):
        step(mats)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step(mats)
    dt = (time.perf_counter() - t0) / args.steps
    gbs = sample_bytes / dt / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "N": 1, "layers": 1,
                   "sample": f"every {frac}th row of each of the 7 matrices"},
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"1/{frac} of the rows of one decode layer "
                                   f"({sample_bytes} weight bytes) per step"},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


# ---------------------------------------------------------------- our path

def run_ours(args):
    import numpy as np
    import torch

    from skinny_gemm_q4_gb300 import build as b
    from skinny_gemm_q4_gb300 import qgemv as qg
    from skinny_gemm_q4_gb300 import synth

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    b.build()
    qg.load()
    dev = torch.device("cuda", local)

    # 36 synthetic layers generated on the device.
    layers = []
    for L in range(N_LAYERS):
        hs = {}
        for i, (role, qt, M, K) in enumerate(synth.LAYER):
            w, sc, g = synth.device_weights(qt, M, K, seed=rank, stream=1000 * L + i, device=dev)
            hs[role] = qg.QGemv(qt, M, K, w, sc, g, max_tokens=32)
        layers.append(hs)
    x_qkv = synth.device_activations(1, 2560, 0, 1, dev)
    x_o = synth.device_activations(1, 4096, 0, 2, dev)
    res = synth.device_activations(1, 2560, 0, 3, dev)
    x_ffn = synth.device_activations(1, 2560, 0, 4, dev)
    x_dn = synth.device_activations(1, 9728, 0, 5, dev)
    f16 = torch.float16
    yq = torch.empty((1, 4096), dtype=f16, device=dev)
    yk = torch.empty((1, 1024), dtype=f16, device=dev)
    yv = torch.empty((1, 1024), dtype=f16, device=dev)
    yo = torch.empty((1, 2560), dtype=f16, device=dev)
    yg = torch.empty((1, 9728), dtype=f16, device=dev)
    yu = torch.empty((1, 9728), dtype=f16, device=dev)
    yd = torch.empty((1, 2560), dtype=f16, device=dev)

    part = args.part
    rows = max(1, args.rows) if part == "gate" else 1
    x_g = synth.device_activations(rows, 2560, 0, 7, dev)
    y_g = torch.empty((rows, 9728), dtype=f16, device=dev)

    def step(L):
        h = layers[L]
        s = torch.cuda.current_stream().cuda_stream
        if part in ("layer", "qkv"):
            qg.qgemv_triple_run(h["wq"].h, h["wk"].h, h["wv"].h, x_qkv.data_ptr(), 1,
                                yq.data_ptr(), yk.data_ptr(), yv.data_ptr(), qg.OUT_F16, s)
        if part in ("layer", "wo"):
            qg.qgemv_run_add(h["wo"].h, x_o.data_ptr(), 1, res.data_ptr(), yo.data_ptr(), s)
        if part in ("layer", "pair"):
            qg.qgemv_pair_run(h["gate"].h, h["up"].h, x_ffn.data_ptr(), 1, yg.data_ptr(),
                              yu.data_ptr(), qg.OUT_F16, s)
        if part in ("layer", "down"):
            qg.qgemv_run(h["down"].h, x_dn.data_ptr(), 1, yd.data_ptr(), qg.OUT_F16, s)
        if part == "gate":
            qg.qgemv_run(h["gate"].h, x_g.data_ptr(), rows, y_g.data_ptr(), qg.OUT_F16, s)

    roles = {"layer": [r for r, _, _, _ in synth.LAYER], "qkv": ["wq", "wk", "wv"],
             "wo": ["wo"], "pair": ["gate", "up"], "down": ["down"], "gate": ["gate"]}[part]
    wbytes = sum(M * synth.row_bytes(qt, K) for r, qt, M, K in synth.LAYER if r in roles)
    # N = 1: one product kernel per call (x staged in-kernel)
    launches_per_step = 4 if part == "layer" else 1
    if part == "gate":
        launches_per_step = layers[0]["gate"].plan_info(rows)[2]

    for i in range(args.warmup):
        step(i % N_LAYERS)
    torch.cuda.synchronize()

    # Capture exactly K steps as one graph (launch-bound otherwise: a step is
    # ~10 us of GPU time).
    side = torch.cuda.Stream(device=dev)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            for i in range(args.steps):
                step(i % N_LAYERS)
    graph.replay()  # untimed
    torch.cuda.synchronize()

    def barrier():
        if dist is not None:
            dist.barrier()

    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        barrier()
        torch.cuda.synchronize()
        clk.mark_start()
        start.record()
        graph.replay()
        end.record()
        torch.cuda.synchronize()
        clk.mark_end()
        barrier()
    ms, value = aggregate_ranks(start.elapsed_time(end), world, wbytes, args.steps, dist, dev)
    ms_step = ms / args.steps

    # Dominant kernel: the gate/up pair product (44% of the layer's bytes),
    # timed alone back to back over the 36 layers (graph), CUDA events on the
    # launching stream.
    pair_bytes = 2 * 9728 * synth.row_bytes(synth.Q4_K, 2560)
    reps = N_LAYERS * 4
    pg = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(pg, stream=side):
            for i in range(reps):
                h = layers[i % N_LAYERS]
                qg.qgemv_pair_run(h["gate"].h, h["up"].h, x_ffn.data_ptr(), 1, yg.data_ptr(),
                                  yu.data_ptr(), qg.OUT_F16, torch.cuda.current_stream().cuda_stream)
    pg.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    pg.replay()
    e1.record()
    torch.cuda.synchronize()
    pair_us = e0.elapsed_time(e1) * 1e3 / reps
    peak, peak_kind = _peaks()
    achieved = pair_bytes / (pair_us * 1e-6) / 1e9

    # Skinny sweep on the gate matrices (Q4_K 9728 x 2560): one call per
    # layer, N rows, graph replay over the 36 layers (cold), CUDA events.
    sweep = None
    if part == "layer" and not args.no_sweep:
        sweep = {"matrix": "Q4_K 9728x2560 (gate of each layer)", "unit": "GB/s", "points": []}
        xs = synth.device_activations(32, 2560, 0, 6, dev)
        ys = torch.empty((32, 9728), dtype=f16, device=dev)
        gbytes = 9728 * synth.row_bytes(synth.Q4_K, 2560)
        for n in (1, 2, 4, 8, 16, 32):
            sg = torch.cuda.CUDAGraph()
            with torch.cuda.stream(side):
                with torch.cuda.graph(sg, stream=side):
                    for i in range(reps):
                        qg.qgemv_run(layers[i % N_LAYERS]["gate"].h, xs.data_ptr(), n,
                                     ys.data_ptr(), qg.OUT_F16,
                                     torch.cuda.current_stream().cuda_stream)
            sg.replay()
            torch.cuda.synchronize()
            e0.record()
            sg.replay()
            e1.record()
            torch.cuda.synchronize()
            us = e0.elapsed_time(e1) * 1e3 / reps
            sweep["points"].append({"N": n, "us_per_call": round(us, 3),
                                    "GBps": round(gbytes / (us * 1e-6) / 1e9, 1),
                                    "frac_of_measured": round(gbytes / (us * 1e-6) / 1e9 / peak, 4)})
            del sg

    # End to end through the host-buffer entry point: per matrix, x from
    # pinned host memory, y back to pinned host memory, synchronized.
    e2e_steps = min(args.steps, N_LAYERS) if part == "layer" else 0
    hx = {K: torch.from_numpy(np.random.default_rng(K).standard_normal((1, K)).astype(np.float16))
          .pin_memory() for K in (2560, 4096, 9728)}
    hy = {M: torch.empty((1, M), dtype=f16).pin_memory() for M in (4096, 1024, 2560, 9728)}
    h2d = sum(K * 2 for _, _, M, K in synth.LAYER)
    d2h = sum(M * 2 for _, _, M, K in synth.LAYER)
    s = torch.cuda.current_stream().cuda_stream
    for L in range(2 if e2e_steps else 0):
        for role, qt, M, K in synth.LAYER:
            qg.qgemv_run_host(layers[L][role].h, hx[K].data_ptr(), 1, hy[M].data_ptr(),
                              qg.OUT_F16, s)
    barrier()
    t0 = time.perf_counter()
    for i in range(e2e_steps):
        for role, qt, M, K in synth.LAYER:
            qg.qgemv_run_host(layers[i % N_LAYERS][role].h, hx[K].data_ptr(), 1,
                              hy[M].data_ptr(), qg.OUT_F16, s)
    e2e_s = (time.perf_counter() - t0) / max(e2e_steps, 1)
    barrier()
    e2e_val = world * wbytes / e2e_s / 1e9 if e2e_steps else None

    if rank != 0:
        return
    # CPU baseline: the oracle on one whole layer (N = 1), single thread.
    cpu = None
    if not args.no_cpu_baseline and world == 1 and part == "layer":
        import oracle
        oracle.build()
        t_cpu = 0.0
        for i, (role, qt, M, K) in enumerate(synth.LAYER):
            h = layers[0][role]
            w = h._w.cpu().numpy()
            sc = None if h._scales is None else h._scales.cpu().numpy()
            x = synth.activations(1, K, seed=0, stream=300 + i)
            t0 = time.perf_counter()
            oracle.qgemv(qt, w, M, K, x, scales=sc)
            t_cpu += time.perf_counter() - t0
        cpu = {"value": round(wbytes / t_cpu / 1e9, 4), "unit": "GB/s", "cores": 1,
               "kind": "oracle",
               "sample": "one whole decode layer (7 matrices, 63.9 MB of weights), N=1"}

    clocks = clk.summary()
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f16 x, fp32 accumulate, 4-bit weights",
        "data": "synthetic",
        "config": {"workload": WORKLOAD if part == "layer" else WORKLOAD + ":" + part, "N": rows,
                   "layers_rotated": N_LAYERS,
                   "weight_bytes_per_step": wbytes,
                   "cold": "36 distinct layers (2.3 GB) > L2; no flush needed",
                   "pct_of_nominal_8TBps": round(100 * value / world / 8000.0, 2),
                   "pct_of_measured_hbm": round(100 * value / world / peak, 2)},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": _traffic_record(),
                     "kernel": "gate/up pair call: gemv_kernel<Q4_K> (one launch, N=1)",
                     "per_launch_us": round(pair_us, 3), "bytes_per_launch": pair_bytes,
                     "peak_kind": peak_kind},
        "cpu_baseline": cpu,
        "e2e": None if e2e_val is None else {"value": round(e2e_val, 3), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "how": "qgemv_run_host per matrix (pinned host x and y, synchronized)"},
        "sweep": sweep,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
    }
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3600)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sweep", action="store_true", help="skip the N = 1..32 sweep line")
    ap.add_argument("--part", default="layer", choices=["layer", "qkv", "wo", "pair", "down", "gate"],
                    help="time one call of the layer only (profiling); default: the whole layer")
    ap.add_argument("--rows", type=int, default=1,
                    help="N for --part gate (the gate matrix alone at N rows: the skinny and "
                         "prefill kernels, for profiling)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
