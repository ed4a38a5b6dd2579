#!/usr/bin/env python
"""Benchmark of the GB300 Q4_K SwiGLU FFN (one JSON line on rank 0).

Workload: the LLaMA-7B-shaped decode FFN (hidden 4096, inter 11008, m = 1,
seeded Q4_K weights, float32 activations). A step is one full call of the
feed-forward block (all its kernels). The metric is weight bytes streamed per
second (GB/s) against the measured HBM copy bandwidth; a secondary object
reports the 27B-shaped long prefill (hidden 5120, inter 17408, m = 2048) in
int8-equivalent TOPS against the measured dense fp16/bf16 tensor peak.

Timing: W eager warm-up steps, then K steps replayed from a CUDA graph and
timed with CUDA events on the capture stream, bracketed by a barrier and a
device synchronisation on both sides. The weights rotate over enough replicas
that more than three times the L2 size is touched between two uses of one
replica, so every step streams its weights from HBM. nvidia-smi samples the
SM clock and throttle reasons during the timed region.

  python bench.py [--gpus N --steps K --warmup W]          this library
  python bench.py --impl reference [...]                   the CPU oracle
For N > 1 each rank runs an independent replica (the FFN does not shard here).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import multiprocessing as mp
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

L2_BYTES = 135_528_448
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--prefill-steps", type=int, default=120)
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--no-q8", action="store_true", help="skip the Q8_1-activation decode leg")
    ap.add_argument("--no-q6k", action="store_true", help="skip the Q6_K LM-head GEMV leg")
    ap.add_argument("--cpu-budget-s", type=float, default=12.0)
    return ap.parse_args()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def src_hash(*files) -> str:
    """Hash of the code that decides the profiled kernel's memory traffic: the GEMV
    kernel template and its CTA shapes in decode.cu, plus the named helper files,
    with comments and blank space removed (edits to comments or to other kernels
    keep a committed profile valid)."""
    import re
    h = hashlib.sha256()
    for f in files:
        text = open(os.path.join(ROOT, "q4_swiglu_ffn_gb300", "csrc", f)).read()
        if f == "decode.cu":
            a = text.index("template <bool GATEUP, int NT, int COMBOS, int TPW, int SLICES, int STAGES, int CPS>")
            b = text.index("constexpr size_t gemv_smem()")
            text = text[a:b]
        text = re.sub(r"//[^\n]*", "", text)
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        h.update(re.sub(r"\s+", "", text).encode())
    return h.hexdigest()[:16]


def profiled_traffic(name: str, sha: str):
    """DRAM bytes per launch from a committed ncu summary, if taken on the current source."""
    path = os.path.join(ROOT, "profiles", name)
    if not os.path.exists(path):
        return None
    for line in open(path):
        if line.startswith("BENCH_TRAFFIC "):
            d = json.loads(line[len("BENCH_TRAFFIC "):])
            if d.get("src_sha") == sha:
                return d.get("dram_bytes_per_launch")
    return None


# --------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: str):
        self.samples = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", gpu_index], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        win = [p for (t, p) in self.samples if t0 <= t <= t1] or [p for (_, p) in self.samples[-3:]]
        if not win:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = sorted(float(p[1]) for p in win if p[1].replace(".", "").isdigit())
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for p in win for n, v in zip(names, p[5:9]) if v.lower().startswith("active")})
        return {"sm_mhz": sm[len(sm) // 2] if sm else None, "sm_max_mhz": float(win[0][2]),
                "reasons": reasons, "samples": len(win)}


# --------------------------------------------------------------------------- CPU baseline (oracle)
def _cpu_decode_worker(budget_s: float, q):
    import numpy as np
    import oracle
    import workloads
    cfg = workloads.LLAMA7B_DECODE
    wg, wu, wd = workloads.weights(cfg)
    x, _ = workloads.activations(cfg)
    reps, t_total = 0, 0.0
    while t_total < budget_s and reps < 50:
        t = time.perf_counter()
        oracle.ffn_decode(x, wg, wu, wd)
        t_total += time.perf_counter() - t
        reps += 1
    q.put({"reps": reps, "seconds": t_total, "bytes": cfg.weight_bytes() * reps})


def cpu_baseline(budget_s: float):
    """The oracle (numpy float64, unmodified) on the host cores, in a spawned process."""
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    p = ctx.Process(target=_cpu_decode_worker, args=(budget_s, q))
    p.start()
    r = q.get()
    p.join()
    cores = os.cpu_count()
    return {"value": r["bytes"] / r["seconds"] / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{r['reps']} full LLaMA-7B-shaped decode FFN call(s) (m=1) of the numpy float64 oracle, "
                      f"{r['seconds']:.1f} s; BLAS matvecs multi-threaded, per-block dequantisation "
                      f"single-threaded"}


# --------------------------------------------------------------------------- GPU side
def gpu_decode(args, rank, world, dist, path="f32"):
    """Times the decode FFN call: `path` "f32" is ffn_q4k_swiglu (float32 activations),
    "q8_1" is ffn_q4k_swiglu_q8_1 (activations quantized to Q8_1, integer dot products)."""
    import numpy as np
    import torch
    import workloads
    import q4_swiglu_ffn_gb300 as q

    cfg = workloads.LLAMA7B_DECODE
    dev = torch.device("cuda", torch.cuda.current_device())
    wbytes = cfg.weight_bytes()
    R = max(2, math.ceil(3 * L2_BYTES / wbytes))
    host = [workloads.weights(cfg), workloads.weights(cfg, seed=cfg.seed + 1000)]
    reps = [tuple(torch.from_numpy(a).to(dev) for a in host[r % 2]) for r in range(R)]
    x_np, _ = workloads.activations(cfg)
    x = torch.from_numpy(x_np).to(dev)
    y = torch.empty_like(x)
    stream = torch.cuda.Stream()
    torch.cuda.set_stream(stream)

    if path == "q8_1":
        ws = torch.empty(q.ffn_q4k_q8_1_workspace_bytes(cfg.m, cfg.hidden, cfg.inter), dtype=torch.uint8,
                         device=dev)

        def step(i):
            wg, wu, wd = reps[i % R]
            q.ffn_q4k_swiglu_q8_1(x, wg, wu, wd, ws, y=y)
    else:
        def step(i):
            wg, wu, wd = reps[i % R]
            q.ffn_q4k_swiglu(x, wg, wu, wd, y=y)

    for i in range(max(3, args.warmup)):
        step(i)
    torch.cuda.synchronize()
    G = R * max(1, 64 // R)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for i in range(G):
            step(i)
    graph.replay()
    torch.cuda.synchronize()
    n_rep = max(1, math.ceil(args.steps / G))
    K = n_rep * G

    gpu_index = os.environ.get("CUDA_VISIBLE_DEVICES", str(dev.index)).split(",")[dev.index if world == 1 else 0]
    sampler = ClockSampler(gpu_index.strip())
    time.sleep(0.5)
    # an event after every replay of G steps: the spread of per-step times
    evr = [torch.cuda.Event(enable_timing=True) for _ in range(n_rep + 1)]
    for e in evr:
        e.record(stream)  # torch creates the CUDA event on first record
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    evr[0].record(stream)
    for i in range(n_rep):
        graph.replay()
        evr[i + 1].record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    if dist:
        dist.barrier()
    sampler.stop()
    ms = evr[0].elapsed_time(evr[-1])
    per_step = sorted(evr[i].elapsed_time(evr[i + 1]) / G for i in range(n_rep))
    pct = {q: per_step[min(n_rep - 1, int(q / 100 * n_rep))] for q in (10, 50, 90)}
    clocks = sampler.summary(t0, t1)

    # per-kernel durations (events around each kernel of the call; serialises them)
    nk = 5
    P = 300
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2 * nk)] for _ in range(P)]
    for ev in evs:
        for e in ev:
            e.record(stream)  # torch creates the CUDA event on first record
    torch.cuda.synchronize()
    for i in range(P):
        q.q4k_set_profile_events(evs[i])
        step(i)
    q.q4k_set_profile_events(None)
    torch.cuda.synchronize()
    kern_ms = [sum(evs[i][2 * k].elapsed_time(evs[i][2 * k + 1]) for i in range(P)) / P for k in range(nk)]

    # end to end, every step through the C ABI with host buffers and a stream sync:
    # (a) x and y in page-locked host memory, read and written by the kernels across
    #     the host link (no separate copies); (b) explicit copies: pinned x -> device,
    #     the call, device y -> pinned host.
    xh = torch.from_numpy(x_np).pin_memory()
    yh = torch.empty(x_np.shape, dtype=torch.float32).pin_memory()
    E = min(K, 2000) if path == "f32" else 0

    def host_step(i):
        wg, wu, wd = reps[i % R]
        q.ffn_q4k_swiglu(xh, wg, wu, wd, y=yh)

    e2e_ms = e2e_copy_ms = 0.0
    if E:
        for i in range(3):
            host_step(i)
        torch.cuda.synchronize()
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        f0.record(stream)
        for i in range(E):
            host_step(i)
            stream.synchronize()
        f1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = f0.elapsed_time(f1)
        f0.record(stream)
        for i in range(E):
            x.copy_(xh, non_blocking=True)
            step(i)
            yh.copy_(y, non_blocking=True)
            stream.synchronize()
        f1.record(stream)
        torch.cuda.synchronize()
        e2e_copy_ms = f0.elapsed_time(f1)
    assert q.q4k_check_device_error() == 0
    step(0)
    launches = q.q4k_last_call_kernels()
    return {"ms": ms, "K": K, "clocks": clocks, "kern_ms": kern_ms, "e2e_ms": e2e_ms, "e2e_copy_ms": e2e_copy_ms,
            "E": E, "R": R,
            "wbytes": wbytes, "xbytes": x_np.nbytes, "launches_per_step": launches, "pct": pct, "G": G}


def gpu_q6k(args):
    """The Q6_K LM-head GEMV (LLaMA-7B output projection, m = 1), graph-replayed like the decode."""
    import torch
    import workloads
    import q4_swiglu_ffn_gb300 as q

    c = workloads.LMHEADS[1]
    dev = torch.device("cuda", torch.cuda.current_device())
    wbytes = c.weight_bytes()
    R = max(2, math.ceil(3 * L2_BYTES / wbytes))
    base = workloads.lmhead_weights(c)
    reps = [torch.from_numpy(base).to(dev) for _ in range(R)]
    x = torch.from_numpy(workloads.lmhead_x(c)).to(dev)
    y = torch.empty((c.m, c.n), dtype=torch.float32, device=dev)
    ws = torch.empty(q.q6k_gemv_workspace_bytes(c.m, c.n, c.k), dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream()
    torch.cuda.set_stream(stream)

    def step(i):
        q.q6k_gemv(x, reps[i % R], ws, y=y)

    for i in range(max(3, args.warmup)):
        step(i)
    torch.cuda.synchronize()
    G = R * max(1, 64 // R)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for i in range(G):
            step(i)
    graph.replay()
    torch.cuda.synchronize()
    n_rep = max(3, math.ceil(args.steps / 4 / G))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(n_rep):
        graph.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / (n_rep * G)
    P = 200
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(P)]
    for ev in evs:
        for e in ev:
            e.record(stream)
    torch.cuda.synchronize()
    for i in range(P):
        q.q4k_set_profile_events(evs[i])
        step(i)
    q.q4k_set_profile_events(None)
    torch.cuda.synchronize()
    kern_ms = [sum(evs[i][2 * k].elapsed_time(evs[i][2 * k + 1]) for i in range(P)) / P for k in range(2)]
    assert q.q4k_check_device_error() == 0
    return {"cfg": c, "ms": ms, "K": n_rep * G, "kern_ms": kern_ms, "wbytes": wbytes, "R": R}


def gpu_prefill(args):
    import torch
    import workloads
    import q4_swiglu_ffn_gb300 as q

    cfg = workloads.LONG_PREFILL_27B
    dev = torch.device("cuda", torch.cuda.current_device())
    wg, wu, wd = (torch.from_numpy(a).to(dev) for a in workloads.weights(cfg))
    _, xb = workloads.activations(cfg)
    import numpy as np
    x = torch.from_numpy(xb.view(np.int16)).to(dev).view(torch.bfloat16)
    m, H, I = cfg.m, cfg.hidden, cfg.inter
    ws = torch.zeros(q.ffn_q4k_workspace_bytes(m, H, I), dtype=torch.uint8, device=dev)
    y = torch.empty((m, H), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        q.ffn_q4k_swiglu_ex(x, wg, wu, wd, ws, y=y)

    for _ in range(3):
        step()
    torch.cuda.synchronize()
    gpu_index = os.environ.get("CUDA_VISIBLE_DEVICES", str(dev.index)).split(",")[0]
    sampler = ClockSampler(gpu_index.strip())
    time.sleep(0.3)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.time()
    e0.record(stream)
    for _ in range(args.prefill_steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    sampler.stop()
    clocks = sampler.summary(t0, t1)
    ms = e0.elapsed_time(e1) / args.prefill_steps
    nk = 5
    P = 10
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2 * nk)] for _ in range(P)]
    for ev in evs:
        for e in ev:
            e.record(stream)  # torch creates the CUDA event on first record
    torch.cuda.synchronize()
    for i in range(P):
        q.q4k_set_profile_events(evs[i])
        step()
    q.q4k_set_profile_events(None)
    torch.cuda.synchronize()
    kern_ms = [sum(evs[i][2 * k].elapsed_time(evs[i][2 * k + 1]) for i in range(P)) / P for k in range(nk)]
    assert q.q4k_check_device_error() == 0
    return {"ms": ms, "kern_ms": kern_ms, "ops": cfg.int8_ops(), "cfg": cfg, "clocks": clocks}


def whole_job(ms_local: float, units_local: float, dist=None):
    """Max over ranks of the timed region (ms) and the whole-job rate: units summed
    over all ranks (each rank does the same work) divided by that time."""
    ms, world = ms_local, 1
    if dist is not None and dist.is_initialized():
        import torch
        world = dist.get_world_size()
        dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
        t = torch.tensor([ms_local], dtype=torch.float64, device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    return ms, units_local * world / (ms * 1e-3)


def main():
    args = parse()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    import workloads
    cfg = workloads.LLAMA7B_DECODE
    metric = "Q4_K SwiGLU FFN: decode weight GB/s vs HBM peak; prefill int8 TOPS vs peak"
    workload = {"workload": cfg.name, "hidden": cfg.hidden, "inter": cfg.inter, "m": cfg.m,
                "weights": "seeded Q4_K (d, dmin ~ U[0.001, 0.05] fp16, 6-bit scales/mins, 4-bit quants uniform)",
                "x": "float32 N(0,1)"}

    if args.impl == "reference":
        if rank != 0:
            return
        cb = cpu_baseline(args.cpu_budget_s)
        v = cb["value"]
        line = {"impl": "reference", "metric": metric, "value": v, "unit": "GB/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": cfg.weight_bytes() / (v * 1e9) * 1e3,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": workload, "cpu_baseline": cb,
                "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    import torch
    dist = None
    if world > 1:
        import torch.distributed as tdist
        tdist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
        dist = tdist
    torch.cuda.set_device(local)
    try:
        import q4_swiglu_ffn_gb300  # noqa: F401
    except ImportError:
        import __graft_entry__
        __graft_entry__.build()

    r = gpu_decode(args, rank, world, dist)
    ms, rate = whole_job(r["ms"], r["wbytes"] * r["K"], dist)
    value = rate / 1e9
    pk, pk_kind = peaks()

    r8 = None
    if not args.no_q8 and rank == 0:
        r8 = gpu_decode(args, rank, 1, None, path="q8_1")

    r6 = None
    if not args.no_q6k and rank == 0:
        r6 = gpu_q6k(args)

    pre = None
    if not args.no_prefill and rank == 0:
        pre = gpu_prefill(args)
    cb = cpu_baseline(args.cpu_budget_s) if (rank == 0 and world == 1) else None

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return
    # dominant kernel: gate+up GEMV (2/3 of the weight bytes)
    k1_bytes = 2 * cfg.inter * (cfg.hidden // 256) * 144
    k1_ms = r["kern_ms"][1]
    ach = k1_bytes / (k1_ms * 1e-3) / 1e9
    sha = src_hash("decode.cu", "common.cuh")
    roof = {"kernel": "gemv_kernel<gate/up> (K1)", "bound": "hbm", "achieved": ach, "peak": pk["hbm_gbs"],
            "unit": "GB/s", "frac": ach / pk["hbm_gbs"], "peak_kind": f"{pk_kind} copy bandwidth",
            "traffic": profiled_traffic("decode_gateup_llama7b_m1.txt", sha),
            "algorithmic_bytes_per_launch": k1_bytes, "avg_launch_ms": k1_ms,
            "step_frac": (r["wbytes"] / (ms / r["K"] * 1e-3) / 1e9) / pk["hbm_gbs"]}
    e2e_val = r["wbytes"] * r["E"] / (r["e2e_ms"] * 1e-3) / 1e9
    line = {"metric": metric, "value": value, "unit": "GB/s", "n_gpus": world, "steps": r["K"],
            "warmup": args.warmup, "ms_per_step": ms / r["K"],
            "ms_per_step_p10_p50_p90": [r["pct"][10], r["pct"][50], r["pct"][90]],
            "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f16",
            "data": "synthetic",
            "config": dict(workload, l2=f"rotating {r['R']} weight replicas ({r['R'] * r['wbytes'] / 1e6:.0f} MB "
                                        f"> 3x the {L2_BYTES / 1e6:.0f} MB L2)", graph="CUDA graph replay",
                           parallelism=f"replicas x{world}"),
            "roofline": roof,
            "kernels_ms": dict(zip(["prep_x", "gate_up", "swiglu_frag_h", "down", "down_chunk_sum"],
                                   r["kern_ms"][:r["launches_per_step"]])),
            "cpu_baseline": cb,
            "e2e": {"value": e2e_val, "unit": "GB/s", "h2d_bytes_per_step": r["xbytes"],
                    "d2h_bytes_per_step": r["xbytes"], "steps": r["E"],
                    "note": "every step: the C-ABI call with x and y in page-locked host memory (the kernels "
                            "read x and write y across NVLink-C2C), then a stream sync",
                    "with_copies": {"value": r["wbytes"] * r["E"] / (r["e2e_copy_ms"] * 1e-3) / 1e9,
                                    "note": "pinned x -> device copy, the call, device y -> pinned host copy, "
                                            "stream sync, every step"}},
            "gpu_launches": r["launches_per_step"] * r["K"] * world,
            "clocks": r["clocks"]}
    if r8 is not None:
        k1q_ms = r8["kern_ms"][1]
        ach8 = k1_bytes / (k1q_ms * 1e-3) / 1e9
        line["decode_q8_1"] = {
            "workload": cfg.name, "value": r8["wbytes"] * r8["K"] / (r8["ms"] * 1e-3) / 1e9, "unit": "GB/s",
            "ms_per_step": r8["ms"] / r8["K"],
            "ms_per_step_p10_p50_p90": [r8["pct"][10], r8["pct"][50], r8["pct"][90]],
            "step_frac": (r8["wbytes"] / (r8["ms"] / r8["K"] * 1e-3) / 1e9) / pk["hbm_gbs"],
            "dtype": "int8 x u4 (dp4a), f32 scales",
            "numerics": "activations quantized to Q8_1 (x once for gate and up, h before down): "
                        "not the float32-activation contract of the headline value",
            "kernels_ms": dict(zip(["q8_1_x", "gate_up", "swiglu_q8_1_h", "down", "down_chunk_sum"],
                                   r8["kern_ms"][:r8["launches_per_step"]])),
            "roofline": {"kernel": "gemv_q8_kernel<gate/up> (K1)", "bound": "hbm", "achieved": ach8,
                         "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": ach8 / pk["hbm_gbs"],
                         "peak_kind": f"{pk_kind} copy bandwidth", "algorithmic_bytes_per_launch": k1_bytes,
                         "avg_launch_ms": k1q_ms},
            "gpu_launches": r8["launches_per_step"] * r8["K"],
            "clocks": r8["clocks"]}
    if r6 is not None:
        c6 = r6["cfg"]
        ach6 = r6["wbytes"] / (r6["kern_ms"][1] * 1e-3) / 1e9
        line["lmhead_q6k"] = {
            "workload": c6.name, "value": r6["wbytes"] / (r6["ms"] * 1e-3) / 1e9, "unit": "GB/s",
            "ms_per_step": r6["ms"], "steps": r6["K"], "dtype": "f16 (x as fp16 hi + lo), f32 accumulate",
            "kernels_ms": dict(zip(["x_fragments", "q6k_gemv"], r6["kern_ms"])),
            "roofline": {"kernel": "q6k_gemv_kernel", "bound": "hbm", "achieved": ach6, "peak": pk["hbm_gbs"],
                         "unit": "GB/s", "frac": ach6 / pk["hbm_gbs"], "peak_kind": f"{pk_kind} copy bandwidth",
                         "algorithmic_bytes_per_launch": r6["wbytes"], "avg_launch_ms": r6["kern_ms"][1]},
            "step_frac": (r6["wbytes"] / (r6["ms"] * 1e-3) / 1e9) / pk["hbm_gbs"],
            "l2": f"rotating {r6['R']} weight replicas"}
    if pre is not None:
        c = pre["cfg"]
        gu_ops = 2 * c.m * c.hidden * c.inter * 2
        gu_ms = pre["kern_ms"][2]
        peak_t = pk["bf16_tflops_sustained"]  # a long run of back-to-back calls, as the sustained GEMM
        line["prefill"] = {
            "workload": c.name, "value": pre["ops"] / (pre["ms"] * 1e-3) / 1e12, "unit": "TOPS (int8-equivalent)",
            "ms_per_step": pre["ms"],
            "kernels_ms": dict(zip(["q8_1_x", "expand_x", "gate_up_mmq", "expand_h", "down_mmq"], pre["kern_ms"])),
            "roofline": {"kernel": "mmq_kernel<gate+up> (tcgen05 kind::f16)", "bound": "tensor",
                         "achieved": gu_ops / (gu_ms * 1e-3) / 1e12, "peak": peak_t, "unit": "TFLOP/s",
                         "frac": gu_ops / (gu_ms * 1e-3) / 1e12 / peak_t,
                         "peak_kind": f"{pk_kind} sustained dense bf16 (same tensor rate as fp16)",
                         "executed_fp16_frac": 2 * gu_ops / (gu_ms * 1e-3) / 1e12 / peak_t,
                         "note": "achieved counts the algorithmic int8-equivalent ops; the kernel executes 2x "
                                 "that in fp16 (activations split into hi+lo)"},
            "clocks": pre["clocks"],
            "int8_mma_sync_peak_tops": 151.7}
    print(json.dumps(line))
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
