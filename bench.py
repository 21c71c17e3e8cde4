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
import math
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


def _tensor_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), "measured (bf16 dense burst; fp16 runs at the same rate)"
    return 1900.0, "fallback"


# The sources the N <= 8 kernels (the calls `traffic` covers) are built from.
_N8_SOURCES = ("qg_api.cu", "qg_inst.cuh", "qg_inst_q4k.cu", "qg_inst_q6k.cu", "qg_kernels.cuh",
               "qg_launch.cuh", "qg_ptx.cuh")


def _kernel_source_sha():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "skinny_gemm_q4_gb300", "csrc")
    for f in _N8_SOURCES:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def _traffic_record(call):
    """DRAM bytes per launch of one layer call's kernel from the committed ncu
    summary (profiles/traffic.json), or None if the kernel sources changed
    since it was taken or the call was not captured."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        rec = json.load(f)
    if rec.get("source_sha") != _kernel_source_sha():
        return None
    c = rec.get("calls", {}).get(call)
    return None if c is None else c.get("dram_bytes_per_launch")


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


# ---------------------------------------------------------------- CPU oracle

def host_cores() -> int:
    """Cores this process may run on (the cgroup / affinity set, else all)."""
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def oracle_rows_timed(mats, cores):
    """Run the oracle over every (matrix, rows) item, rows split into `cores`
    contiguous parts run on that many threads (the C oracle releases the GIL;
    rows are independent, so the results are those of one thread).  Returns
    the wall time in seconds."""
    import numpy as np

    import oracle
    from concurrent.futures import ThreadPoolExecutor
    jobs = []
    for qt, w, M, K, rows, x, sc in mats:
        for part in np.array_split(rows, cores):
            if part.size:
                jobs.append((qt, w, M, K, part, x, sc))

    def one(j):
        qt, w, M, K, part, x, sc = j
        oracle.qgemv(qt, w, M, K, x, scales=sc, rows=part)

    t0 = time.perf_counter()
    if cores == 1:
        for j in jobs:
            one(j)
    else:
        with ThreadPoolExecutor(max_workers=cores) as ex:
            list(ex.map(one, jobs))
    return time.perf_counter() - t0


# ---------------------------------------------------------------- reference

def run_reference(args):
    """The CPU oracle on a bounded sample of the same workload, timed on this
    host's cores (rows split over every core; the oracle itself as it stands)."""
    import numpy as np

    import oracle
    from skinny_gemm_q4_gb300 import synth
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    oracle.build()
    cores = host_cores()
    # Bounded sample: every frac-th row of each matrix of one layer, frac chosen
    # so that warmup + steps take about a minute on this host in total.
    full = []
    for i, (role, qt, M, K) in enumerate(synth.LAYER):
        w, sc, g = synth.weights(qt, M, K, seed=0, stream=100 + i)
        x = synth.activations(1, K, seed=0, stream=200 + i)
        full.append((qt, w, M, K, x, sc))

    def make(frac):
        mats = [(qt, w, M, K, np.arange(0, M, frac), x, sc) for qt, w, M, K, x, sc in full]
        nbytes = sum(len(m[4]) * synth.row_bytes(m[0], m[3]) for m in mats)
        return mats, nbytes

    probe, probe_bytes = make(64)
    sec_per_byte = oracle_rows_timed(probe, cores) / probe_bytes
    budget = 60.0 / (args.steps + args.warmup)
    frac = 1
    while frac < 4096 and make(frac)[1] * sec_per_byte > budget:
        frac *= 2
    mats, sample_bytes = make(frac)
    for _ in range(args.warmup):
        oracle_rows_timed(mats, cores)
    dt = 0.0
    for _ in range(args.steps):
        dt += oracle_rows_timed(mats, cores)
    dt /= args.steps
    gbs = sample_bytes / dt / 1e9
    what = "one whole decode layer" if frac == 1 else f"every {frac}th row of one decode layer"
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "N": 1, "layers": 1,
                   "sample": f"{what} (7 matrices), N=1"},
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": f"{what}: {sample_bytes} weight bytes per step, rows split "
                                   f"over {cores} threads"},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


# ---------------------------------------------------------------- our path

def _graph_us(torch, side, ncalls, call, e0, e1):
    """Capture ncalls calls call(i, stream) as one CUDA graph on `side`, replay
    it once untimed, then time one replay with CUDA events: us per call."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            for i in range(ncalls):
                call(i, torch.cuda.current_stream().cuda_stream)
    g.replay()
    torch.cuda.synchronize()
    e0.record()
    g.replay()
    e1.record()
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / ncalls
    del g
    return us


def _kernel_name(call, n):
    """The product kernel that serves one layer call at n tokens."""
    types = {"qkv": "Q4_K|Q6_K", "wo": "Q4_K", "pair": "Q4_K", "gate": "Q4_K", "down": "Q6_K",
             "nvfp4": "NVFP4"}[call]
    what = {"qkv": "QKV triple", "wo": "Wo + residual", "pair": "gate/up pair", "gate": "gate",
            "down": "down", "nvfp4": "27648 x 5120"}[call]
    # N = 2..8 on Q4_K/Q5_K matrices of at most 4096 rows (Wo) runs the
    # K-sliced kernel too
    n8 = n == 1 or (n <= 8 and call != "wo")
    kern = "qg_n8_kernel" if n8 else ("qg_sk_kernel" if n <= 32 else "qg_tc_kernel")
    return f"{kern}<{types}> ({what}, N={n})"


def _bw(nbytes, us, peak):
    gbs = nbytes / (us * 1e-6) / 1e9
    return {"us_per_call": round(us, 3), "GBps": round(gbs, 1),
            "frac_of_measured": round(gbs / peak, 4), "frac_of_8TBps": round(gbs / 8000.0, 4)}


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
    peak, peak_kind = _peaks()
    tpeak, tpeak_kind = _tensor_peak()

    # 36 synthetic layers generated on the device (128-token staging so the
    # same handles serve the prefill chunks).
    layers = []
    for L in range(N_LAYERS):
        hs = {}
        for i, (role, qt, M, K) in enumerate(synth.LAYER):
            w, sc, g = synth.device_weights(qt, M, K, seed=rank, stream=1000 * L + i, device=dev)
            hs[role] = qg.QGemv(qt, M, K, w, sc, g, max_tokens=128)
        layers.append(hs)
    # --part nvfp4: six copies of the NVFP4 27648 x 5120 matrix (478 MB > L2)
    NV_M, NV_K = 27648, 5120
    nv = []
    if args.part == "nvfp4":
        for c in range(6):
            w, sc, g = synth.device_weights(synth.NVFP4, NV_M, NV_K, seed=rank, stream=9000 + c,
                                            device=dev)
            nv.append(qg.QGemv(synth.NVFP4, NV_M, NV_K, w, sc, g))
    all_handles = [h for hs in layers for h in hs.values()]
    part = args.part
    rows = max(1, args.rows) if part in ("gate", "prefill", "nvfp4") else 1
    nl = rows if part == "prefill" else 1  # tokens of the layer calls
    x_qkv = synth.device_activations(nl, 2560, 0, 1, dev)
    x_o = synth.device_activations(nl, 4096, 0, 2, dev)
    res = synth.device_activations(nl, 2560, 0, 3, dev)
    x_ffn = synth.device_activations(nl, 2560, 0, 4, dev)
    x_dn = synth.device_activations(nl, 9728, 0, 5, dev)
    f16 = torch.float16
    yq = torch.empty((nl, 4096), dtype=f16, device=dev)
    yk = torch.empty((nl, 1024), dtype=f16, device=dev)
    yv = torch.empty((nl, 1024), dtype=f16, device=dev)
    yo = torch.empty((nl, 2560), dtype=f16, device=dev)
    yg = torch.empty((nl, 9728), dtype=f16, device=dev)
    yu = torch.empty((nl, 9728), dtype=f16, device=dev)
    yd = torch.empty((nl, 2560), dtype=f16, device=dev)

    x_g = synth.device_activations(rows, 2560, 0, 7, dev)
    x_nv = synth.device_activations(rows, NV_K, 0, 8, dev)
    y_nv = torch.empty((rows, NV_M), dtype=f16, device=dev)
    y_g = torch.empty((rows, 9728), dtype=f16, device=dev)

    def call_qkv(h, s):
        qg.qgemv_triple_run(h["wq"].h, h["wk"].h, h["wv"].h, x_qkv.data_ptr(), nl,
                            yq.data_ptr(), yk.data_ptr(), yv.data_ptr(), qg.OUT_F16, s)

    def call_wo(h, s):
        qg.qgemv_run_add(h["wo"].h, x_o.data_ptr(), nl, res.data_ptr(), yo.data_ptr(), s)

    def call_pair(h, s):
        qg.qgemv_pair_run(h["gate"].h, h["up"].h, x_ffn.data_ptr(), nl, yg.data_ptr(),
                          yu.data_ptr(), qg.OUT_F16, s)

    def call_down(h, s):
        qg.qgemv_run(h["down"].h, x_dn.data_ptr(), nl, yd.data_ptr(), qg.OUT_F16, s)

    def call_pair_swiglu(h, s):
        qg.qgemv_pair_swiglu_run(h["gate"].h, h["up"].h, x_ffn.data_ptr(), nl, yg.data_ptr(),
                                 qg.OUT_F16, s)

    CALLS = [("qkv", call_qkv, ["wq", "wk", "wv"]), ("wo", call_wo, ["wo"]),
             ("pair", call_pair, ["gate", "up"]), ("down", call_down, ["down"])]

    # The layer's four calls as one decode chain (qgemv_chain_run): one
    # persistent launch at N <= 8; at larger N the calls run one by one.
    chain = None
    if args.layer_api != "calls":
        chain = qg.Chain(qg.CHAIN_PERSISTENT if args.layer_api == "persistent" else 0)
    chain_calls = []
    if chain is not None:
        for hs in layers:
            chain_calls.append(qg.make_calls([
                (qg.CALL_TRIPLE, [hs["wq"].h, hs["wk"].h, hs["wv"].h], x_qkv.data_ptr(), nl,
                 [yq.data_ptr(), yk.data_ptr(), yv.data_ptr()], qg.OUT_F16, None),
                (qg.CALL_RUN_ADD, [hs["wo"].h], x_o.data_ptr(), nl, [yo.data_ptr()], qg.OUT_F16,
                 res.data_ptr()),
                (qg.CALL_PAIR, [hs["gate"].h, hs["up"].h], x_ffn.data_ptr(), nl,
                 [yg.data_ptr(), yu.data_ptr()], qg.OUT_F16, None),
                (qg.CALL_RUN, [hs["down"].h], x_dn.data_ptr(), nl, [yd.data_ptr()], qg.OUT_F16,
                 None)]))

    def step(L):
        h = layers[L]
        s = torch.cuda.current_stream().cuda_stream
        if chain is not None and part in ("layer", "prefill"):
            qg.qgemv_chain_run(chain.c, chain_calls[L], s)
            return
        if part == "nvfp4":
            qg.qgemv_run(nv[L % len(nv)].h, x_nv.data_ptr(), rows, y_nv.data_ptr(), qg.OUT_F16, s)
            return
        for name, fn, _ in CALLS:
            if part in ("layer", "prefill", name):
                fn(h, s)
        if part == "gate":
            qg.qgemv_run(h["gate"].h, x_g.data_ptr(), rows, y_g.data_ptr(), qg.OUT_F16, s)

    roles = {"layer": [r for r, _, _, _ in synth.LAYER], "prefill": [r for r, _, _, _ in synth.LAYER],
             "qkv": ["wq", "wk", "wv"], "nvfp4": [],
             "wo": ["wo"], "pair": ["gate", "up"], "down": ["down"], "gate": ["gate"]}[part]
    wbytes = sum(M * synth.row_bytes(qt, K) for r, qt, M, K in synth.LAYER if r in roles)
    if part == "nvfp4":  # codes, e4m3 scales (one per 16 weights), the tensor scale
        wbytes = NV_M * (synth.row_bytes(synth.NVFP4, NV_K) + NV_K // 16) + 4
    # N = 1: one product kernel per call (x staged in-kernel)
    launches_per_step = (1 if args.layer_api == "persistent" else 4) if part == "layer" else 1
    if part == "gate":
        launches_per_step = layers[0]["gate"].plan_info(rows)[2]
    if part == "prefill":  # staging + product per call (one launch for the mixed-format triple)
        launches_per_step = sum(layers[0][r].plan_info(rows)[2] for r in ("wq", "wo", "gate", "down"))

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

    # Sustained: the same K-step graph replayed back to back for at least
    # ~0.3 s (so the clock record has many samples); reported beside `value`.
    reps = max(1, int(math.ceil(300.0 / max(ms_step * args.steps, 1e-3))))
    reps = min(reps, 20000)
    with ClockSampler(local) as clk2:
        torch.cuda.synchronize()
        clk2.mark_start()
        start.record()
        for _ in range(reps):
            graph.replay()
        end.record()
        torch.cuda.synchronize()
        clk2.mark_end()
    sus_ms = start.elapsed_time(end) / (reps * args.steps)
    sustained = {"ms_per_step": round(sus_ms, 5), "steps": reps * args.steps,
                 "GBps": round(wbytes / (sus_ms * 1e-3) / 1e9, 1), "clocks": clk2.summary()}
    del graph

    # Every kernel's bounded waits finished in time (a timed-out pipeline
    # would return early with wrong results).
    bad = [h for h in all_handles if h.device_status() != 0]
    if chain is not None and chain.status() != 0:
        bad.append(chain)
    if bad:
        print(json.dumps({"error": f"{len(bad)} handles report a device timeout"}))
        sys.exit(3)

    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ncalls = N_LAYERS * 4

    # Each call of the layer alone, back to back over the 36 layers.
    calls = {}
    if part in ("layer", "prefill"):
        for name, fn, rl in CALLS:
            nb_ = sum(M * synth.row_bytes(qt, K) for r, qt, M, K in synth.LAYER if r in rl)
            us = _graph_us(torch, side, ncalls, lambda i, s, fn=fn: fn(layers[i % N_LAYERS], s),
                           e0, e1)
            calls[name] = dict(_bw(nb_, us, peak), bytes_per_call=nb_,
                               flops_per_call=2 * nl * sum(M * K for r, _, M, K in synth.LAYER
                                                           if r in rl))
        dom = max(calls, key=lambda k: calls[k]["us_per_call"])
        if part == "layer":
            # the gate/up pair with the fused SwiGLU epilogue (h = silu(g) * u),
            # not part of the step: the layer's pair returns g and u
            nb_ = 2 * 9728 * synth.row_bytes(synth.Q4_K, 2560)
            us = _graph_us(torch, side, ncalls,
                           lambda i, s: call_pair_swiglu(layers[i % N_LAYERS], s), e0, e1)
            calls["pair_swiglu"] = dict(_bw(nb_, us, peak), bytes_per_call=nb_)
            # the whole layer as one persistent launch (QG_CHAIN_PERSISTENT),
            # for comparison with the step's launch per call
            pchain = qg.Chain(qg.CHAIN_PERSISTENT)
            lb = sum(M * synth.row_bytes(qt, K) for _, qt, M, K in synth.LAYER)
            us = _graph_us(torch, side, ncalls,
                           lambda i, s: qg.qgemv_chain_run(pchain.c, chain_calls[i % N_LAYERS], s),
                           e0, e1) if chain_calls else 0.0
            if chain_calls:
                calls["layer_persistent_chain"] = dict(_bw(lb, us, peak), bytes_per_call=lb)
                if pchain.status() != 0:
                    print(json.dumps({"error": "persistent chain reports a device timeout"}))
                    sys.exit(3)
    elif part == "nvfp4":
        dom = "nvfp4"
        us = _graph_us(torch, side, ncalls,
                       lambda i, s: qg.qgemv_run(nv[i % len(nv)].h, x_nv.data_ptr(), rows,
                                                 y_nv.data_ptr(), qg.OUT_F16, s), e0, e1)
        calls[dom] = dict(_bw(wbytes, us, peak), bytes_per_call=wbytes,
                          flops_per_call=2 * rows * NV_M * NV_K)
    elif part == "gate":
        dom = "gate"
        nb_ = 9728 * synth.row_bytes(synth.Q4_K, 2560)
        us = _graph_us(torch, side, ncalls,
                       lambda i, s: qg.qgemv_run(layers[i % N_LAYERS]["gate"].h, x_g.data_ptr(),
                                                 rows, y_g.data_ptr(), qg.OUT_F16, s), e0, e1)
        calls[dom] = dict(_bw(nb_, us, peak), bytes_per_call=nb_, flops_per_call=2 * rows * 9728 * 2560)
    else:
        dom = part
        rl = dict((n, r) for n, _, r in CALLS)[dom]
        fn = dict((n, f) for n, f, _ in CALLS)[dom]
        nb_ = sum(M * synth.row_bytes(qt, K) for r, qt, M, K in synth.LAYER if r in rl)
        us = _graph_us(torch, side, ncalls, lambda i, s: fn(layers[i % N_LAYERS], s), e0, e1)
        calls[dom] = dict(_bw(nb_, us, peak), bytes_per_call=nb_)
    d = calls[dom]
    ntok = rows if part in ("gate", "prefill", "nvfp4") else 1
    kname = _kernel_name(dom, ntok)
    flops = d.get("flops_per_call", 0)
    if ntok >= 33 and flops / (tpeak * 1e12) > d["bytes_per_call"] / (peak * 1e9):
        # more tensor time than weight-stream time at this token count
        tf = flops / (d["us_per_call"] * 1e-6) / 1e12
        roofline = {"bound": "tensor", "achieved": round(tf, 1), "peak": tpeak, "unit": "TFLOP/s",
                    "frac": round(tf / tpeak, 4), "traffic": None,
                    "kernel": kname + ": the costliest call, timed alone",
                    "per_launch_us": d["us_per_call"], "flops_per_launch": flops,
                    "weight_GBps": d["GBps"], "peak_kind": tpeak_kind}
    else:
        roofline = {"bound": "hbm", "achieved": d["GBps"], "peak": peak, "unit": "GB/s",
                    "frac": round(d["GBps"] / peak, 4),
                    "traffic": _traffic_record(dom) if ntok == 1 else None,
                    "kernel": kname + ": the costliest call, timed alone",
                    "per_launch_us": d["us_per_call"], "bytes_per_launch": d["bytes_per_call"],
                    "peak_kind": peak_kind}

    configs = None
    if part == "layer" and not args.no_configs:
        configs = run_configs(args, torch, qg, synth, layers, side, e0, e1, peak, tpeak, dev)

    # End to end through the public API, as a user runs a decode step: one
    # qgemv_chain_run_host call copies the step's inputs (x of the four calls
    # and the residual, one pinned host buffer, a new one each step out of
    # four) to the device, runs the layer's calls, copies every output back to
    # pinned host memory and synchronizes the stream.
    e2e_steps = min(args.steps, 4 * N_LAYERS) if part == "layer" else 0
    e2e_val = None
    h2d = d2h = 0
    if e2e_steps:
        kin = {"qkv": 2560, "o": 4096, "res": 2560, "ffn": 2560, "dn": 9728}
        kout = {"q": 4096, "k": 1024, "v": 1024, "o": 2560, "g": 9728, "u": 9728, "d": 2560}
        din = torch.empty(sum(kin.values()), dtype=f16, device=dev)
        dout = torch.empty(sum(kout.values()), dtype=f16, device=dev)
        hins = [torch.from_numpy(np.random.default_rng(100 + r).standard_normal(din.numel())
                                 .astype(np.float16)).pin_memory() for r in range(4)]
        hout = torch.empty(dout.numel(), dtype=f16).pin_memory()
        h2d, d2h = din.numel() * 2, dout.numel() * 2

        def views(buf, sizes):
            out, o = {}, 0
            for k, n in sizes.items():
                out[k] = buf[o:o + n]
                o += n
            return out
        vi, vo = views(din, kin), views(dout, kout)
        ptr = lambda t: t.data_ptr()
        e2e_calls = [qg.make_calls([
            (qg.CALL_TRIPLE, [hs["wq"].h, hs["wk"].h, hs["wv"].h], ptr(vi["qkv"]), 1,
             [ptr(vo["q"]), ptr(vo["k"]), ptr(vo["v"])], qg.OUT_F16, None),
            (qg.CALL_RUN_ADD, [hs["wo"].h], ptr(vi["o"]), 1, [ptr(vo["o"])], qg.OUT_F16,
             ptr(vi["res"])),
            (qg.CALL_PAIR, [hs["gate"].h, hs["up"].h], ptr(vi["ffn"]), 1,
             [ptr(vo["g"]), ptr(vo["u"])], qg.OUT_F16, None),
            (qg.CALL_RUN, [hs["down"].h], ptr(vi["dn"]), 1, [ptr(vo["d"])], qg.OUT_F16, None)])
            for hs in layers]
        echain = qg.Chain()
        cs = torch.cuda.current_stream()

        def e2e_step(i):
            # inputs in, the layer, outputs out, synchronized: one library call
            qg.qgemv_chain_run_host(echain.c, e2e_calls[i % N_LAYERS], hins[i % 4].data_ptr(),
                                    din.data_ptr(), h2d, dout.data_ptr(), hout.data_ptr(), d2h,
                                    cs.cuda_stream)

        for i in range(max(args.warmup, 3)):
            e2e_step(i)
        barrier()
        t0 = time.perf_counter()
        for i in range(e2e_steps):
            e2e_step(i)
        e2e_s = (time.perf_counter() - t0) / e2e_steps
        barrier()
        e2e_val = world * wbytes / e2e_s / 1e9
        if echain.status() != 0:
            print(json.dumps({"error": "end-to-end chain reports a device timeout"}))
            sys.exit(3)

    if rank != 0:
        return
    # CPU baseline: the oracle on one whole layer (N = 1), rows split over
    # every host core, and single-threaded beside it.
    cpu = None
    if not args.no_cpu_baseline and world == 1 and part == "layer":
        import oracle
        oracle.build()
        mats = []
        for i, (role, qt, M, K) in enumerate(synth.LAYER):
            h = layers[0][role]
            w = h._w.cpu().numpy()
            sc = None if h._scales is None else h._scales.cpu().numpy()
            x = synth.activations(1, K, seed=0, stream=300 + i)
            mats.append((qt, w, M, K, np.arange(M), x, sc))
        cores = host_cores()
        t_all = oracle_rows_timed(mats, cores)
        t_one = oracle_rows_timed(mats, 1)
        cpu = {"value": round(wbytes / t_all / 1e9, 4), "unit": "GB/s", "cores": cores,
               "kind": "oracle",
               "sample": "one whole decode layer (7 matrices, 63.9 MB of weights), N=1, rows "
                         f"split over {cores} threads",
               "single_thread_value": round(wbytes / t_one / 1e9, 4)}

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
        "dtype": "f16",  # MMA operands (x, decoded weights); see "accumulate"
        "accumulate": "f32",
        "weights": "4-bit block formats (Q4_K, Q6_K in the decode layer)",
        "data": "synthetic",
        "config": {"workload": WORKLOAD if part == "layer" else WORKLOAD + ":" + part, "N": rows,
                   "layers_rotated": N_LAYERS,
                   "layer_api": {"chain": "qgemv_chain_run (a launch per call, PDL-chained)",
                                 "persistent": "qgemv_chain_run (one persistent launch)",
                                 "calls": "four entry-point calls"}[args.layer_api]
                   if part in ("layer", "prefill") else "one call",
                   "weight_bytes_per_step": wbytes,
                   "cold": ("6 copies of the matrix (478 MB) > L2; no flush needed"
                            if part == "nvfp4" else
                            "36 distinct layers (2.3 GB) > L2; no flush needed"),
                   "pct_of_nominal_8TBps": round(100 * value / world / 8000.0, 2),
                   "pct_of_measured_hbm": round(100 * value / world / peak, 2)},
        "roofline": roofline,
        "calls": calls,
        "sustained": sustained,
        "cpu_baseline": cpu,
        "e2e": None if e2e_val is None else {"value": round(e2e_val, 3), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "steps": e2e_steps,
                "how": "per step: qgemv_chain_run_host -- the step's inputs copied from "
                       "pinned host memory to the device, the layer's calls, all outputs "
                       "copied back to pinned host memory, stream synchronized"},
        "configs": configs,
        "device_status": 0,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
    }
    print(json.dumps(line))


def run_configs(args, torch, qg, synth, layers, side, e0, e1, peak, tpeak, dev):
    """The other workloads, each timed cold (rotating copies > 4x L2) with
    CUDA events over one graph replay: the single small GEMV, the skinny row
    sweeps, prefill chunks over the 36-layer set and the NVFP4 ~10 GB set."""
    f16 = torch.float16
    out = {}
    ncalls = N_LAYERS * 4

    # Single Q4_K GEMV 256 x 2560, N = 1: copies covering > 4x L2.
    c0 = synth.CONFIG0
    nb0 = c0["M"] * synth.row_bytes(c0["qtype"], c0["K"])
    copies = int(math.ceil(4 * 129e6 / nb0))
    hs0 = []
    for i in range(copies):
        w, sc, g = synth.device_weights(c0["qtype"], c0["M"], c0["K"], seed=0, stream=50000 + i,
                                        device=dev)
        hs0.append(qg.QGemv(c0["qtype"], c0["M"], c0["K"], w, sc, g, max_tokens=8))
    x0 = synth.device_activations(1, c0["K"], 0, 11, dev)
    y0 = torch.empty((1, c0["M"]), dtype=f16, device=dev)
    us = _graph_us(torch, side, copies, lambda i, s: qg.qgemv_run(
        hs0[i].h, x0.data_ptr(), 1, y0.data_ptr(), qg.OUT_F16, s), e0, e1)
    out["c0_q4k_256x2560_n1"] = dict(_bw(nb0, us, peak), copies=copies)
    del hs0

    # Skinny row sweeps: Q4_K 9728 x 2560 (the gate of each layer) and Q5_K
    # 2560 x 9728 (36 copies), N rows.
    hs5 = []
    for L in range(N_LAYERS):
        w, sc, g = synth.device_weights(synth.Q5_K, 2560, 9728, seed=0, stream=60000 + L,
                                        device=dev)
        hs5.append(qg.QGemv(synth.Q5_K, 2560, 9728, w, sc, g, max_tokens=32))
    sweeps = {}
    for name, hsel, M, K, qt in (
            ("q4k_9728x2560", lambda i: layers[i % N_LAYERS]["gate"], 9728, 2560, synth.Q4_K),
            ("q5k_2560x9728", lambda i: hs5[i % N_LAYERS], 2560, 9728, synth.Q5_K)):
        xs = synth.device_activations(32, K, 0, 12, dev)
        ys = torch.empty((32, M), dtype=f16, device=dev)
        nbytes = M * synth.row_bytes(qt, K)
        pts = []
        for n in synth.SWEEP_N:
            us = _graph_us(torch, side, ncalls, lambda i, s, n=n: qg.qgemv_run(
                hsel(i).h, xs.data_ptr(), n, ys.data_ptr(), qg.OUT_F16, s), e0, e1)
            pts.append(dict(_bw(nbytes, us, peak), N=n))
        sweeps[name] = pts
    out["c2_sweep"] = sweeps
    del hs5

    # Prefill chunks over the 36-layer Q4_K_M-mixed set: per layer the QKV
    # triple, Wo + residual, the gate/up pair and down at N tokens.
    layer_bytes = sum(M * synth.row_bytes(qt, K) for _, qt, M, K in synth.LAYER)
    layer_mk = sum(M * K for _, qt, M, K in synth.LAYER)
    pre = {}
    for n in synth.PREFILL_N:
        xq = synth.device_activations(n, 2560, 0, 13, dev)
        xo = synth.device_activations(n, 4096, 0, 14, dev)
        xd = synth.device_activations(n, 9728, 0, 15, dev)
        rr = synth.device_activations(n, 2560, 0, 16, dev)
        yb = {M: torch.empty((n, M), dtype=f16, device=dev) for M in (4096, 1024, 2560, 9728)}
        yb2 = {M: torch.empty((n, M), dtype=f16, device=dev) for M in (1024, 9728)}

        def layer_call(i, s, n=n, xq=xq, xo=xo, xd=xd, rr=rr, yb=yb, yb2=yb2):
            h = layers[i % N_LAYERS]
            qg.qgemv_triple_run(h["wq"].h, h["wk"].h, h["wv"].h, xq.data_ptr(), n,
                                yb[4096].data_ptr(), yb[1024].data_ptr(), yb2[1024].data_ptr(),
                                qg.OUT_F16, s)
            qg.qgemv_run_add(h["wo"].h, xo.data_ptr(), n, rr.data_ptr(), yb[2560].data_ptr(), s)
            qg.qgemv_pair_run(h["gate"].h, h["up"].h, xq.data_ptr(), n, yb[9728].data_ptr(),
                              yb2[9728].data_ptr(), qg.OUT_F16, s)
            qg.qgemv_run(h["down"].h, xd.data_ptr(), n, yb[2560].data_ptr(), qg.OUT_F16, s)

        us = _graph_us(torch, side, N_LAYERS, layer_call, e0, e1)
        tf = 2.0 * n * layer_mk / (us * 1e-6) / 1e12
        d = _bw(layer_bytes, us, peak)
        d = {"us_per_layer": d["us_per_call"], "GBps": d["GBps"],
             "frac_of_measured_hbm": d["frac_of_measured"], "TFLOPs": round(tf, 1),
             "frac_of_tensor_peak": round(tf / tpeak, 4),
             "us_36_layers": round(us * N_LAYERS, 1)}
        pre[f"N{n}"] = d
    out["c3_prefill_36_layers"] = pre

    # NVFP4 W4A16: 56 copies of {27648x5120, 5120x27648, 7168x5120} (~10 GB).
    sets = args.nvfp4_sets
    hs4 = []
    set_bytes = 0
    for M, K in synth.NVFP4_SHAPES:
        set_bytes += M * K // 2 + M * K // 16 + 4
    for c in range(sets):
        for j, (M, K) in enumerate(synth.NVFP4_SHAPES):
            w, sc, g = synth.device_weights(synth.NVFP4, M, K, seed=0, stream=70000 + 3 * c + j,
                                            device=dev)
            hs4.append(qg.QGemv(synth.NVFP4, M, K, w, sc, g, max_tokens=32))
    xs4 = {K: synth.device_activations(32, K, 0, 17, dev) for K in (5120, 27648)}
    ys4 = {M: torch.empty((32, M), dtype=f16, device=dev) for M in (27648, 5120, 7168)}
    nv = {"copies": sets, "bytes_per_pass": sets * set_bytes}
    for n in synth.NVFP4_N:
        us = _graph_us(torch, side, len(hs4), lambda i, s, n=n: qg.qgemv_run(
            hs4[i].h, xs4[hs4[i].K].data_ptr(), n, ys4[hs4[i].M].data_ptr(), qg.OUT_F16, s),
            e0, e1)
        total_us = us * len(hs4)
        d = _bw(sets * set_bytes, total_us, peak)
        nv[f"N{n}"] = {"us_per_pass": round(total_us, 1), "GBps": d["GBps"],
                       "frac_of_measured": d["frac_of_measured"],
                       "frac_of_8TBps": d["frac_of_8TBps"]}
    out["c4_nvfp4_set"] = nv
    bad = sum(1 for h in hs4 if h.device_status() != 0)
    del hs4
    torch.cuda.empty_cache()

    # FP8 block-scaled W8A16 (e4m3 + one bf16 scale per 128 x 128 block) on
    # the same three shapes: 8 copies (2.6 GB, > 4x L2).
    fsets = 8
    hs8 = []
    f_bytes = 0
    for M, K in synth.NVFP4_SHAPES:
        f_bytes += M * K + ((M + 127) // 128) * (K // 128) * 2
    for c in range(fsets):
        for j, (M, K) in enumerate(synth.NVFP4_SHAPES):
            w, sc, g = synth.device_weights(synth.FP8, M, K, seed=0, stream=80000 + 3 * c + j,
                                            device=dev)
            hs8.append(qg.QGemv(synth.FP8, M, K, w, sc, g, max_tokens=32))
    f8 = {"copies": fsets, "bytes_per_pass": fsets * f_bytes,
          "shapes": "27648x5120, 5120x27648, 7168x5120"}
    for n in synth.NVFP4_N:
        us = _graph_us(torch, side, len(hs8), lambda i, s, n=n: qg.qgemv_run(
            hs8[i].h, xs4[hs8[i].K].data_ptr(), n, ys4[hs8[i].M].data_ptr(), qg.OUT_F16, s),
            e0, e1)
        total_us = us * len(hs8)
        d = _bw(fsets * f_bytes, total_us, peak)
        f8[f"N{n}"] = {"us_per_pass": round(total_us, 1), "GBps": d["GBps"],
                       "frac_of_measured": d["frac_of_measured"],
                       "frac_of_8TBps": d["frac_of_8TBps"]}
    out["fp8_w8a16_set"] = f8
    bad += sum(1 for h in hs8 if h.device_status() != 0)
    bad += sum(1 for hs in layers for h in hs.values() if h.device_status() != 0)
    if bad:
        print(json.dumps({"error": f"{bad} handles report a device timeout (configs)"}))
        sys.exit(3)
    del hs8
    torch.cuda.empty_cache()
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3600)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the other workloads (single GEMV, sweeps, prefill, NVFP4 set)")
    ap.add_argument("--no-sweep", dest="no_configs", action="store_true",
                    help="same as --no-configs")
    ap.add_argument("--nvfp4-sets", type=int, default=56,
                    help="copies of the three NVFP4 shapes (56: ~10 GB)")
    ap.add_argument("--part", default="layer",
                    choices=["layer", "qkv", "wo", "pair", "down", "gate", "prefill", "nvfp4"],
                    help="time one call of the layer only (profiling); prefill: the whole layer "
                         "at --rows tokens; default: the whole layer at N = 1")
    ap.add_argument("--layer-api", default="chain", choices=["chain", "persistent", "calls"],
                    help="layer step through one decode chain call (qgemv_chain_run: one "
                         "launch per matrix call, PDL-chained), the same in one persistent "
                         "launch, or four separate entry-point calls")
    ap.add_argument("--rows", type=int, default=1,
                    help="N for --part gate (the gate matrix alone at N rows: the skinny and "
                         "prefill kernels) and --part prefill (for profiling)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
