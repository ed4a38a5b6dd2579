#!/usr/bin/env python
"""Benchmark of the GB300 Q4_K SwiGLU FFN (one JSON line on rank 0).

Headline workload: the LLaMA-7B-shaped decode FFN (hidden 4096, inter 11008,
m = 1, seeded Q4_K weights, float32 activations). A step is one full call of
the feed-forward block (all its kernels). The metric is weight bytes streamed
per second (GB/s) against the measured HBM copy bandwidth. Further objects on
the same line report the other workloads of the method: the tiny decode (256 x
768), the 13B-shaped batched decode (m = 8, outlier channels), the 8B-shaped
prefill (m = 512) and the 27B-shaped long prefill (m = 2048), the prefills in
int8-equivalent TOPS against the measured dense fp16/bf16 tensor peak (burst
and sustained) and against the int8 mma.sync rate measured in this run; plus
the Q8_1-activation decode and the Q6_K LM-head GEMV.

Timing: W eager warm-up steps, then exactly K steps replayed from CUDA graphs
and timed with CUDA events on the capture stream, bracketed by a barrier and a
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
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--prefill-steps", type=int, default=120)
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--no-q8", action="store_true", help="skip the Q8_1-activation decode leg")
    ap.add_argument("--no-q6k", action="store_true", help="skip the Q6_K LM-head GEMV leg")
    ap.add_argument("--no-configs", action="store_true", help="skip the tiny, 13B batched and 8B prefill legs")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end host-buffer loops")
    ap.add_argument("--quick", action="store_true",
                    help="short counts everywhere (no clock lead-in, 64-step secondary legs, 20 profiled calls): "
                         "for launch-list captures")
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
            a = text.find("template <bool GATEUP, int NT, int COMBOS, int TPW, int SLICES, int STAGES, int CPS")
            b = text.find("constexpr size_t gemv_smem()")
            if 0 <= a < b:
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
def _oracle_call_args(frac_blocks: int | None):
    """The LLaMA-7B-shaped decode FFN's inputs, or (frac_blocks = b) the same FFN restricted to the
    first b 256-wide blocks of the intermediate dimension: a sub-problem of the same computation
    whose cost scales with b (a bounded sample of one call)."""
    import workloads
    cfg = workloads.LLAMA7B_DECODE
    wg, wu, wd = workloads.weights(cfg)
    x, _ = workloads.activations(cfg)
    if frac_blocks is None:
        return (x, wg, wu, wd), cfg.weight_bytes()
    b = frac_blocks
    wg, wu, wd = wg[:256 * b], wu[:256 * b], wd[:, :b]
    return (x, wg, wu, wd), (wg.nbytes + wu.nbytes + wd.nbytes)


def _cpu_decode_worker(budget_s: float, q):
    import oracle
    args, nbytes = _oracle_call_args(None)
    reps, t_total = 0, 0.0
    while t_total < budget_s and reps < 50:
        t = time.perf_counter()
        oracle.ffn_decode(*args)
        t_total += time.perf_counter() - t
        reps += 1
    q.put({"reps": reps, "seconds": t_total, "bytes": nbytes * reps})


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


def _reference_worker(steps: int, warmup: int, budget_s: float, q):
    """`--impl reference`: exactly `warmup` untimed and `steps` timed oracle calls. Each step is one
    full call when all of them fit in the budget; otherwise each step is the same bounded sample
    (the FFN restricted to a leading block range of the intermediate dimension)."""
    import oracle
    args, nbytes = _oracle_call_args(None)
    t = time.perf_counter()
    oracle.ffn_decode(*args)
    t_call = time.perf_counter() - t
    blocks = 43                                # 11008 / 256: the whole call
    if (steps + warmup) * t_call > budget_s:
        blocks = max(1, int(43 * budget_s / ((steps + warmup) * t_call)))
        args, nbytes = _oracle_call_args(blocks)
    for _ in range(max(0, warmup - 1)):
        oracle.ffn_decode(*args)
    t0 = time.perf_counter()
    for _ in range(steps):
        oracle.ffn_decode(*args)
    sec = time.perf_counter() - t0
    q.put({"steps": steps, "seconds": sec, "bytes": nbytes * steps, "blocks": blocks})


def reference_arm(steps: int, warmup: int, budget_s: float = 240.0):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    p = ctx.Process(target=_reference_worker, args=(steps, warmup, budget_s, q))
    p.start()
    r = q.get()
    p.join()
    return r


# --------------------------------------------------------------------------- GPU side
class Steps:
    """Exactly K calls of `step(i)` (i = 0..K-1, replica i % R) recorded into CUDA graphs: as many
    replays of a G-step graph as fit, then one graph of the K mod G remaining steps."""

    def __init__(self, step, K: int, R: int, stream):
        import torch
        self.K = K
        self.G = max(1, min(K, R * max(1, 64 // R)))
        self.full, rem = divmod(K, self.G)
        self.stream = stream

        def capture(n):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for i in range(n):
                    step(i)
            return g
        self.g_full = capture(self.G) if self.full else None
        self.g_rem = capture(rem) if rem else None
        self.rem = rem

    def replay_all(self, events=None):
        """Enqueues the K steps; events (full + 2 of them) are recorded before, after each full replay and at the end."""
        if events:
            events[0].record(self.stream)
        for i in range(self.full):
            self.g_full.replay()
            if events:
                events[i + 1].record(self.stream)
        if self.g_rem is not None:
            self.g_rem.replay()
        if events:
            events[-1].record(self.stream)


def _events(n):
    import torch
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    for e in ev:
        e.record()  # torch creates the CUDA event on first record
    return ev


QUICK = False


def _kernel_ms(q, step, P: int, nk: int):
    """Mean duration of each of the call's kernels over P calls (events around each kernel;
    they serialise the kernels, so these are per-kernel, not per-call, figures)."""
    import torch
    P = min(P, 20) if QUICK else P
    evs = [_events(2 * nk) for _ in range(P)]
    torch.cuda.synchronize()
    for i in range(P):
        q.q4k_set_profile_events(evs[i])
        step(i)
    q.q4k_set_profile_events(None)
    torch.cuda.synchronize()
    return [sum(evs[i][2 * k].elapsed_time(evs[i][2 * k + 1]) for i in range(P)) / P for k in range(nk)]


def _gpu_index(dev, world):
    return os.environ.get("CUDA_VISIBLE_DEVICES", str(dev.index)).split(",")[dev.index if world == 1 else 0].strip()


def gpu_decode(cfg, K, warmup, rank, world, dist, path="f32", e2e=False):
    """Times K decode FFN calls on `cfg`: `path` "f32" is ffn_q4k_swiglu (float32 activations),
    "q8_1" is ffn_q4k_swiglu_q8_1 (activations quantized to Q8_1)."""
    import torch
    import workloads
    import q4_swiglu_ffn_gb300 as q

    dev = torch.device("cuda", torch.cuda.current_device())
    wbytes = cfg.weight_bytes()
    R = min(64, max(2, math.ceil(3 * L2_BYTES / wbytes)))
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

    for i in range(max(3, warmup)):
        step(i)
    torch.cuda.synchronize()
    runs = Steps(step, K, R, stream)
    runs.replay_all()
    torch.cuda.synchronize()

    sampler = ClockSampler(_gpu_index(dev, world))
    time.sleep(0.3)
    # a long untimed lead-in keeps the clocks at their loaded value into the timed region
    lead = Steps(step, max(K, 2000), R, stream) if (K < 2000 and not QUICK) else runs
    ev = _events(runs.full + 2)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    lead.replay_all()
    runs.replay_all(ev)
    torch.cuda.synchronize()
    t1 = time.time()
    if dist:
        dist.barrier()
    ms = ev[0].elapsed_time(ev[-1])
    per_step = sorted(ev[i].elapsed_time(ev[i + 1]) / runs.G for i in range(runs.full)) or [ms / K]
    n = len(per_step)
    pct = {p: per_step[min(n - 1, int(p / 100 * n))] for p in (10, 50, 90)}
    # a longer timed run beside the K steps: many steps, so the spread and clocks mean something
    long_ms, long_K = None, 0
    if lead is not runs:
        ev2 = _events(lead.full + 2)
        lead.replay_all(ev2)
        torch.cuda.synchronize()
        long_ms, long_K = ev2[0].elapsed_time(ev2[-1]), lead.K
    t2 = time.time()
    sampler.stop()
    clocks = sampler.summary(t0, t2)
    kern_ms = _kernel_ms(q, step, 300, 5)

    e2e_ms = e2e_copy_ms = 0.0
    E = min(max(K, 200), 2000) if e2e else 0
    xh = torch.from_numpy(x_np).pin_memory()
    yh = torch.empty(x_np.shape, dtype=torch.float32).pin_memory()
    if E:
        # end to end, every step through the C ABI with host buffers and a stream sync:
        # (a) x and y in page-locked host memory, read and written by the kernels across
        #     the host link (no separate copies); (b) explicit copies: pinned x -> device,
        #     the call, device y -> pinned host.
        def host_step(i):
            wg, wu, wd = reps[i % R]
            q.ffn_q4k_swiglu(xh, wg, wu, wd, y=yh)

        for i in range(3):
            host_step(i)
        torch.cuda.synchronize()
        f0, f1 = _events(2)
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
    torch.cuda.synchronize()
    torch.cuda.set_stream(torch.cuda.default_stream())
    return {"cfg": cfg, "path": path, "ms": ms, "K": K, "clocks": clocks, "kern_ms": kern_ms, "e2e_ms": e2e_ms,
            "e2e_copy_ms": e2e_copy_ms, "E": E, "R": R, "wbytes": wbytes, "xbytes": x_np.nbytes,
            "launches_per_step": launches, "pct": pct, "G": runs.G, "long_ms": long_ms, "long_K": long_K}


def gpu_q6k(K):
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

    for i in range(3):
        step(i)
    torch.cuda.synchronize()
    runs = Steps(step, K, R, stream)
    runs.replay_all()
    ev = _events(runs.full + 2)
    runs.replay_all(ev)
    torch.cuda.synchronize()
    ms = ev[0].elapsed_time(ev[-1]) / K
    kern_ms = _kernel_ms(q, step, 200, 2)
    assert q.q4k_check_device_error() == 0
    torch.cuda.set_stream(torch.cuda.default_stream())
    return {"cfg": c, "ms": ms, "K": K, "kern_ms": kern_ms, "wbytes": wbytes, "R": R}


def gpu_prefill(cfg, steps, world):
    import numpy as np
    import torch
    import workloads
    import q4_swiglu_ffn_gb300 as q

    dev = torch.device("cuda", torch.cuda.current_device())
    wg, wu, wd = (torch.from_numpy(a).to(dev) for a in workloads.weights(cfg))
    _, xb = workloads.activations(cfg)
    x = torch.from_numpy(xb.view(np.int16)).to(dev).view(torch.bfloat16)
    m, H, I = cfg.m, cfg.hidden, cfg.inter
    ws = torch.zeros(q.ffn_q4k_workspace_bytes(m, H, I), dtype=torch.uint8, device=dev)
    y = torch.empty((m, H), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def step(i=0):
        q.ffn_q4k_swiglu_ex(x, wg, wu, wd, ws, y=y)

    for _ in range(3):
        step()
    torch.cuda.synchronize()
    sampler = ClockSampler(_gpu_index(dev, world))
    time.sleep(0.3)
    e0, e1 = _events(2)
    t0 = time.time()
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    sampler.stop()
    clocks = sampler.summary(t0, t1)
    ms = e0.elapsed_time(e1) / steps
    kern_ms = _kernel_ms(q, step, 30, len(PREFILL_KERNELS))
    step()
    launches = q.q4k_last_call_kernels()
    assert q.q4k_check_device_error() == 0
    return {"ms": ms, "kern_ms": kern_ms, "ops": cfg.int8_ops(), "cfg": cfg, "clocks": clocks, "steps": steps,
            "launches_per_step": launches, "timed_s": t1 - t0}


def gpu_fp8_gemm(cfg, reps=20):
    """The FP8 tensor-path Q4_K x Q8_1 GEMM (tcgen05 kind::f8f6f4) on the gate projection of `cfg`:
    Q8_1 activations [m, hidden] x W_gate [inter rows] -> [m, inter] float32; CUDA events over `reps`
    back-to-back calls (two kernels each: operand planes, GEMM) and around the GEMM kernel alone."""
    import numpy as np
    import torch
    import workloads
    import q4_swiglu_ffn_gb300 as q
    dev = torch.device("cuda", torch.cuda.current_device())
    m, k, n = cfg.m, cfg.hidden, cfg.inter
    wg = torch.from_numpy(workloads.weights(cfg)[0]).to(dev)
    xf, _ = workloads.activations(cfg)
    xq8 = torch.empty(q.q8_1_bytes(m, k), dtype=torch.uint8, device=dev)
    q.q8_1_quantize_act(torch.from_numpy(xf).to(dev), xq8)
    ws = torch.empty(q.q4k_mmq_fp8_workspace_bytes(m, k), dtype=torch.uint8, device=dev)
    out = torch.empty((m, n), dtype=torch.float32, device=dev)
    for _ in range(3):
        q.q4k_mmq_fp8(xq8, m, k, wg, workspace=ws, out=out)
    torch.cuda.synchronize()
    e0, e1 = _events(2)
    e0.record()
    for _ in range(reps):
        q.q4k_mmq_fp8(xq8, m, k, wg, workspace=ws, out=out)
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / reps
    assert q.q4k_check_device_error() == 0
    ops = 2 * m * k * n
    return {"cfg": cfg, "ms": ms, "ops": ops, "reps": reps}


def gpu_int8_peak(world):
    """The int8 tensor rate of this part (mma.sync m16n8k32 s8), measured now: best of 5 launches."""
    import torch
    import q4_swiglu_ffn_gb300 as q
    dev = torch.device("cuda", torch.cuda.current_device())
    iters = 512 if QUICK else 8192
    for _ in range(2):
        q.q4k_bench_int8_mma(iters)
    torch.cuda.synchronize()
    sampler = ClockSampler(_gpu_index(dev, world))
    time.sleep(0.3)
    best = None
    t0 = time.time()
    for _ in range(5):
        e0, e1 = _events(2)
        e0.record()
        ops = q.q4k_bench_int8_mma(iters)
        e1.record()
        torch.cuda.synchronize()
        tops = ops / (e0.elapsed_time(e1) * 1e-3) / 1e12
        best = tops if best is None else max(best, tops)
    t1 = time.time()
    sampler.stop()
    assert q.q4k_check_device_error() == 0
    return {"tops": best, "instruction": "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32",
            "how": "best of 5 launches, 4 CTAs x 8 warps per SM, 8 independent MMA chains per warp, CUDA events",
            "clocks": sampler.summary(t0, t1)}


def gpu_tcgen05_issue():
    """Cycles per tcgen05.mma kind::f16 (M 128, K 16) from one issuing thread per CTA at
    N 64, 128 and 256, and from two threads at N 64 and 128: the issue cost behind the prefill
    MMQ's one N = 256 MMA per K step (the tensor pipe takes 4096 multiply-adds per cycle), and
    the floor of about 64 cycles per MMA of one issuing thread that narrow N does not lower."""
    import q4_swiglu_ffn_gb300 as q
    iters = 256 if QUICK else 2048
    out = {}
    for n, k in ((64, 1), (128, 1), (256, 1), (64, 2), (128, 2)):
        q.q4k_bench_tcgen05_issue(n, k, 16)
        c = q.q4k_bench_tcgen05_issue(n, k, iters)
        out[f"n{n}_issuers{k}"] = {"cycles_per_mma": c, "pipe_fraction": k * 128 * n * 16 / c / 4096}
    assert q.q4k_check_device_error() == 0
    return {"per_issuing_thread": out,
            "how": f"one CTA per SM, {iters} rounds of 4 MMAs per issuing thread, A in tensor memory, one commit "
                   "per round; cycles of one issuing thread from its first MMA to its last MMA's completion"}


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


DECODE_KERNELS = ["prep_x", "gate_up", "swiglu_frag_h", "down", "down_chunk_sum"]
Q8_KERNELS = ["q8_1_x", "gate_up", "swiglu_q8_1_h", "down", "down_chunk_sum"]
PREFILL_KERNELS = ["quant_expand_x", "gate_up_mmq", "expand_h", "down_mmq_and_sums"]
DECODE_DTYPE = "f16 hi+lo x (~22-bit), exact f16 q*scale weights, f32 accumulate"


def _kernel_slots(r):
    """The profiling slots (K0, K1, K1b, K2, K3) a decode call used: with x in device memory one
    token on the float32 entry, and one or two on the Q8_1 entry, have no K0 (the gate/up GEMV
    takes x itself)."""
    slots = [0, 1, 2, 3, 4]
    if (r.get("path") == "f32" and r["cfg"].m == 1) or (r.get("path") == "q8_1" and r["cfg"].m <= 2):
        slots = slots[1:]  # no K0: the gate/up GEMV takes x itself
    return slots[:r["launches_per_step"]]


def decode_object(r, pk, pk_kind, names, dtype, kernel_label):
    """The JSON object of one decode leg: rate, per-kernel times and the roofline of the gate/up GEMV."""
    c = r["cfg"]
    k1_bytes = 2 * c.inter * (c.hidden // 256) * 144
    k1_ms = r["kern_ms"][1]
    ach = k1_bytes / (k1_ms * 1e-3) / 1e9
    step_ms = r["ms"] / r["K"]
    o = {"workload": c.name, "hidden": c.hidden, "inter": c.inter, "m": c.m,
         "value": r["wbytes"] / (step_ms * 1e-3) / 1e9, "unit": "GB/s", "steps": r["K"], "ms_per_step": step_ms,
         "step_frac": (r["wbytes"] / (step_ms * 1e-3) / 1e9) / pk["hbm_gbs"], "dtype": dtype,
         "kernels_ms": {names[i]: r["kern_ms"][i] for i in _kernel_slots(r)},
         "roofline": {"kernel": kernel_label, "bound": "hbm", "achieved": ach, "peak": pk["hbm_gbs"],
                      "unit": "GB/s", "frac": ach / pk["hbm_gbs"], "peak_kind": f"{pk_kind} copy bandwidth",
                      "algorithmic_bytes_per_launch": k1_bytes, "avg_launch_ms": k1_ms},
         "l2": f"rotating {r['R']} weight replicas ({r['R'] * r['wbytes'] / 1e6:.1f} MB)"
               + (" > 3x the L2" if r["R"] * r["wbytes"] > 3 * L2_BYTES else ", L2-resident: launch-bound size"),
         "gpu_launches": r["launches_per_step"] * r["K"], "clocks": r["clocks"]}
    if r["long_ms"]:
        o["long_run"] = {"steps": r["long_K"], "ms_per_step": r["long_ms"] / r["long_K"],
                         "value": r["wbytes"] * r["long_K"] / (r["long_ms"] * 1e-3) / 1e9}
    return o


def prefill_object(pre, pk, pk_kind, int8):
    c = pre["cfg"]
    gu_ops = 2 * c.m * c.hidden * c.inter * 2
    gu_ms = pre["kern_ms"][PREFILL_KERNELS.index("gate_up_mmq")]
    ach = gu_ops / (gu_ms * 1e-3) / 1e12
    burst, sus = pk["bf16_tflops"], pk["bf16_tflops_sustained"]
    o = {"workload": c.name, "hidden": c.hidden, "inter": c.inter, "m": c.m,
         "value": pre["ops"] / (pre["ms"] * 1e-3) / 1e12, "unit": "TOPS (int8-equivalent)",
         "ms_per_step": pre["ms"], "steps": pre["steps"], "timed_s": pre["timed_s"],
         "dtype": "f16 tcgen05 (exact f16 q*scale weights, Q8_1 activations as f16 hi+lo), f32 accumulate",
         "kernels_ms": dict(zip(PREFILL_KERNELS, pre["kern_ms"])),
         "roofline": {"kernel": "mmq_kernel<gate+up> (tcgen05 kind::f16)", "bound": "tensor",
                      "achieved": ach, "peak": burst, "unit": "TFLOP/s", "frac": ach / burst,
                      "peak_kind": f"{pk_kind} burst dense bf16 (the fp16 tensor rate is the same)",
                      "frac_sustained": ach / sus, "peak_sustained": sus,
                      "executed_fp16_frac": 2 * ach / burst, "avg_launch_ms": gu_ms,
                      "algorithmic_ops_per_launch": gu_ops,
                      "note": "achieved counts the algorithmic int8-equivalent ops; the kernel executes 2x "
                              "that in fp16 (activations split into hi+lo)"},
         "gpu_launches": pre["launches_per_step"] * pre["steps"], "clocks": pre["clocks"]}
    if int8 is not None:
        o["vs_int8_mma_sync"] = {"int8_peak_tops": int8["tops"], "call_frac": o["value"] / int8["tops"],
                                 "gate_up_frac": ach / int8["tops"]}
    return o


def main():
    global QUICK
    args = parse()
    QUICK = args.quick
    legK = 64 if QUICK else 2000
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
        r = reference_arm(args.steps, args.warmup)
        v = r["bytes"] / r["seconds"] / 1e9
        whole = r["blocks"] == 43
        sample = (f"{r['steps']} timed calls of the numpy float64 oracle on the whole LLaMA-7B-shaped decode FFN "
                  f"(m=1), {args.warmup} untimed" if whole else
                  f"{r['steps']} timed calls of the numpy float64 oracle, each on the same bounded sample of the "
                  f"LLaMA-7B-shaped decode FFN: intermediate rows 0..{256 * r['blocks'] - 1} of 11008")
        line = {"impl": "reference", "metric": metric, "value": v, "unit": "GB/s", "n_gpus": world,
                "steps": r["steps"], "warmup": args.warmup, "ms_per_step": r["seconds"] / r["steps"] * 1e3,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": workload,
                "cpu_baseline": {"value": v, "unit": "GB/s", "cores": os.cpu_count(), "kind": "oracle",
                                 "sample": sample},
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

    K = max(1, args.steps)
    r = gpu_decode(cfg, K, args.warmup, rank, world, dist, e2e=not args.no_e2e)
    ms, rate = whole_job(r["ms"], r["wbytes"] * r["K"], dist)
    value = rate / 1e9
    pk, pk_kind = peaks()
    lead = rank == 0

    r8 = gpu_decode(cfg, legK, 3, rank, 1, None, path="q8_1") if (lead and not args.no_q8) else None
    r6 = gpu_q6k(legK // 2) if (lead and not args.no_q6k) else None
    others = {}
    if lead and not args.no_configs:
        others["decode_tiny_h256_i768_m1"] = gpu_decode(workloads.TINY_DECODE, legK, 3, rank, 1, None)
        others["decode_13b_h5120_i13824_m8"] = gpu_decode(workloads.BATCHED_13B_DECODE, legK, 3, rank, 1, None)
    int8 = gpu_int8_peak(1) if (lead and not args.no_prefill) else None
    tc_issue = gpu_tcgen05_issue() if (lead and not args.no_prefill) else None
    pre = {}
    if lead and not args.no_prefill:
        if not args.no_configs:
            pre["prefill_8b_h4096_i14336_m512"] = gpu_prefill(workloads.PREFILL_8B,
                                                              (4 if QUICK else 4 * args.prefill_steps), 1)
        pre["prefill_27b_h5120_i17408_m2048"] = gpu_prefill(workloads.LONG_PREFILL_27B,
                                                              (4 if QUICK else args.prefill_steps), 1)
    f8 = gpu_fp8_gemm(workloads.LONG_PREFILL_27B, 4 if QUICK else 20) if (lead and not args.no_prefill) else None
    cb = cpu_baseline(args.cpu_budget_s) if (lead and world == 1) else None

    if not lead:
        if dist:
            dist.destroy_process_group()
        return
    head = decode_object(r, pk, pk_kind, DECODE_KERNELS, DECODE_DTYPE, "gemv_kernel<gate/up> (K1)")
    roof = dict(head["roofline"])
    roof["traffic"] = profiled_traffic("decode_gateup_llama7b_m1.txt", src_hash("decode.cu", "common.cuh"))
    roof["step_frac"] = head["step_frac"]
    e2e_val = r["wbytes"] * r["E"] / (r["e2e_ms"] * 1e-3) / 1e9 if r["E"] else None
    line = {"metric": metric, "value": value, "unit": "GB/s", "n_gpus": world, "steps": r["K"],
            "warmup": args.warmup, "ms_per_step": ms / r["K"],
            "ms_per_step_p10_p50_p90": [r["pct"][10], r["pct"][50], r["pct"][90]],
            "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": DECODE_DTYPE,
            "data": "synthetic",
            "config": dict(workload, l2=head["l2"], graph="CUDA graph replay", parallelism=f"replicas x{world}"),
            "roofline": roof,
            "kernels_ms": head["kernels_ms"],
            "cpu_baseline": cb,
            "e2e": {"value": e2e_val, "unit": "GB/s", "h2d_bytes_per_step": r["xbytes"],
                    "d2h_bytes_per_step": r["xbytes"], "steps": r["E"],
                    "note": "every step: the C-ABI call with x and y in page-locked host memory (the kernels "
                            "read x and write y across NVLink-C2C), then a stream sync",
                    "with_copies": {"value": r["wbytes"] * r["E"] / (r["e2e_copy_ms"] * 1e-3) / 1e9 if r["E"] else None,
                                    "note": "pinned x -> device copy, the call, device y -> pinned host copy, "
                                            "stream sync, every step"}},
            "gpu_launches": r["launches_per_step"] * r["K"] * world,
            "clocks": r["clocks"]}
    if r["long_ms"]:
        line["long_run"] = head["long_run"]
    for key, ro in others.items():
        line[key] = decode_object(ro, pk, pk_kind, DECODE_KERNELS, DECODE_DTYPE, "gemv_kernel<gate/up> (K1)")
    if r8 is not None:
        o = decode_object(r8, pk, pk_kind, Q8_KERNELS, "Q8_1 activations: int8 x u4 dp4a (m <= 2), f32 scales",
                          "gemv_q8_kernel<gate/up> (K1)")
        o["numerics"] = ("activations quantized to Q8_1 (x once for gate and up, h before down): "
                         "not the float32-activation contract of the headline value")
        line["decode_q8_1"] = o
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
    if int8 is not None:
        line["int8_tensor_peak"] = int8
    if tc_issue is not None:
        line["tcgen05_mma_issue"] = tc_issue
    for key, p in pre.items():
        line[key] = prefill_object(p, pk, pk_kind, int8)
    if f8 is not None:
        c = f8["cfg"]
        ach = f8["ops"] / (f8["ms"] * 1e-3) / 1e12
        fp8_peak = 2.0 * pk["bf16_tflops"]
        o = {"workload": f"{c.name} gate projection only (m {c.m}, k {c.hidden}, n {c.inter})",
             "value": ach, "unit": "TOPS (int8-equivalent)", "ms_per_call": f8["ms"], "calls": f8["reps"],
             "dtype": "e4m3 x e4m3 tcgen05 kind::f8f6f4, exact integer products, f32 scales per sub-block",
             "roofline": {"kernel": "mmq_fp8_kernel (tcgen05 kind::f8f6f4)", "bound": "tensor", "achieved": ach,
                          "peak": fp8_peak, "unit": "TFLOP/s", "frac": ach / fp8_peak,
                          "peak_kind": f"{pk_kind} burst dense bf16 x 2 (the nominal fp8/bf16 ratio)",
                          "note": "the call includes the operand-plane kernel; per op it executes 2 MMAs (hi, lo)"}}
        gp = pre.get("prefill_27b_h5120_i17408_m2048")
        if gp is not None:
            gu_ops = 2 * c.m * c.hidden * c.inter * 2
            gu_ms = gp["kern_ms"][PREFILL_KERNELS.index("gate_up_mmq")]
            o["fp16_mmq_gate_up_tops_same_run"] = gu_ops / (gu_ms * 1e-3) / 1e12
        line["prefill_fp8_gemm_prototype"] = o
    print(json.dumps(line))
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
