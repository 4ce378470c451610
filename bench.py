"""Throughput of the fused attention hot path on GB300: one JSON line.

Default (our arm): ``python bench.py [--gpus N --steps K --warmup W]``.
A step is one pass of the hot path over one batch of the headline workload
(B=4, Hq=Hkv=16, N=4096, d=128, non-causal, bf16, synthetic N(0,1) inputs):
the forward kernel, then (once built) the backward chain (preprocess,
main kernel, dQ postprocess) on the same batch.  FLOPs credited:
4*B*Hq*N^2*d for the forward, 2.5x that for the backward.

Timing: W untimed steps, then K steps bracketed by a barrier and
torch.cuda.synchronize(), timed with CUDA events on the launching stream; the
inputs (Q, K, V, dO: 64 MiB each) exceed the 126 MB L2, so no flush is done
between steps.  Per-kernel durations come from CUDA events recorded between
the launches of every timed step.  SM clocks and throttle reasons are sampled
with nvidia-smi during the timed region.

``--impl reference`` times the CPU oracle (float64, the machine's host cores) on a
bounded sample of the same workload and prints the same line with
"impl": "reference".  Under torchrun every rank runs the workload on its own
GPU (replicas; attention has no exchange step) and rank 0 prints the line.
"""
import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "attention fwd/bwd TFLOPs/s (BF16, d=128) and % of 2.25 PFLOPS dense peak"
PEAK_NOMINAL_TFLOPS = 2250.0
WORKLOAD = "large"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-bwd", action="store_true", help="time the forward only")
    ap.add_argument("--workload", default=WORKLOAD,
                    help="large (default), tiny, causal, varlen, causal_bwd, large_d64, causal_bwd_d64, "
                         "large_d256, causal_d256, varlen_d256")
    ap.add_argument("--deterministic", action="store_true", help="backward in deterministic mode")
    ap.add_argument("--exp2-emu", type=int, default=0, help="forward: sixteenths of exp2 on the FMA pipe (0-4)")
    ap.add_argument("--tau", type=float, default=8.0, help="forward: conditional-rescale threshold (log2 units)")
    ap.add_argument("--bwd-kernel", type=int, default=0,
                    help="backward main kernel: 0 one CTA per 128-key tile, 1 CTA pairs per 256-key block")
    ap.add_argument("--fwd-kernel", type=int, default=2, choices=[0, 2],
                    help="forward kernel: 0 ping-pong 128x128, 2 CTA pairs with 256-key blocks")
    ap.add_argument("--e2e-steps", type=int, default=100,
                    help="end-to-end steps timed (the first upload and the last download are not overlapped)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="CPU baseline sample budget")
    return ap.parse_args()


def dist_init(n):
    rank, world = int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if os.environ.get("FA_BENCH_BACKEND", "nccl") == "nccl" else "gloo"
        dist.init_process_group(backend=backend)
    return rank, world


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world, device=None):
    """Largest x over all ranks (the slowest rank's time); x itself at N=1."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    if device is None or dist.get_backend() == "gloo":
        device = "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_tflops(flops_per_step, steps, world, ms_max):
    """Whole-job throughput: every rank runs the same per-GPU workload
    (replicas), so the job processed world * steps steps in the slowest
    rank's time."""
    return flops_per_step * steps * world / (ms_max / 1e3) / 1e12


class ClockSampler:
    """nvidia-smi SM clock / throttle-reason samples taken in a thread."""

    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.samples = []
        self.proc = None
        self.index = index

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q, "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()
        t0 = time.time()
        while not self.samples and time.time() - t0 < 5:
            time.sleep(0.01)

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 7:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        def num(s):
            try:
                return float(s)
            except ValueError:
                return None
        win = [p for (t, p) in self.samples if t0 <= t <= t1] or [p for (_, p) in self.samples[-3:]]
        if not win:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [num(p[0]) for p in win if num(p[0]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in win for i in range(4) if p[3 + i].strip() == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": num(win[0][1]),
                "power_w_max": max((num(p[2]) or 0.0) for p in win), "reasons": reasons, "samples": len(win)}


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f)
    except (OSError, ValueError):
        return None


def tile_budget(kind, M=128, N=128, d=128, mma_flop_per_clk=8192, exp_per_clk=16, smem_bytes_per_clk=128,
                pair=False, ds_t_in_tmem=True, tma_writes=False):
    """Per-SM cycles one M x N (query x key) tile costs each resource alone:
    the feeds-and-speeds model of the FA4 blog ("Feeds and speeds") and the
    FA4 paper summary (Tables 1 and 3), with B200's rates as defaults.

    tensor core: 2 products of 2 M N d FLOP forward, 5 backward;
    exponential unit: M N exponentials;
    shared memory: the bytes the tensor core reads as operands, plus what
    threads or copies move through it:
      forward  -- Q, K and V tiles (P is read from tensor memory);
      backward -- S^T = K Q^T reads K and Q, dP^T = V dO^T reads V and dO,
                  dV += P^T dO reads dO (P^T from tensor memory), dK += dS^T Q
                  reads Q (and dS^T unless it sits in tensor memory), dQ = dS K
                  reads dS and K; the dS tile is stored, and the fp32 dQ tile
                  is written to and read back from shared memory for its
                  reduction.
    pair: on CTA pairs each CTA stages half of every B operand (K in the
    forward's S, V in P V; Q, dO, dO, Q, K in the backward's five products);
    the dQ tile's round trip is counted whole, as the paper summary's Table 3
    counts it.
    tma_writes=True gives this build's one-CTA backward (dK reads dS^T from
    tensor memory; the Q and dO copies land in shared memory)."""
    b = 2  # bf16 bytes
    if kind == "fwd":
        mma = 4 * M * N * d / mma_flop_per_clk
        q, k, v = M * d * b, N * d * b, N * d * b
        if pair:
            k, v = k / 2, v / 2
        smem = q + k + v + (q + k + v if tma_writes else 0)
    elif kind == "bwd":
        mma = 10 * M * N * d / mma_flop_per_clk
        q = do = M * d * b
        k = v = N * d * b
        ds = M * N * b
        half = 0.5 if pair else 1.0
        reads = (k + q * half) + (v + do * half) + do * half + (q * half + (0 if ds_t_in_tmem else ds)) \
            + (ds + k * half)
        dq = M * d * 4
        smem = reads + ds + 2 * dq + ((q + do) if tma_writes else 0)
    else:
        raise ValueError(kind)
    return {"mma": mma, "exp": M * N / exp_per_clk, "smem": smem / smem_bytes_per_clk}


def kernel_traffic(name, workload):
    """dram bytes per launch from the committed ncu summary, or None when the
    counters were taken on another workload or the kernel's sources changed
    since."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        rec = json.load(open(path)).get(name)
    except (OSError, ValueError):
        return None
    if not rec or rec.get("workload", "").split(":")[0] != workload:
        return None
    h = hashlib.sha256()
    try:
        for src in rec["sources"]:
            h.update(open(os.path.join(ROOT, src), "rb").read())
    except (OSError, KeyError):
        return None
    return rec["dram_bytes_per_launch"] if h.hexdigest()[:16] == rec["sources_sha"] else None


def traffic_key(args, w, kernel):
    """Record name in profiles/dram_traffic.json for a step kernel."""
    if w.d != 128:   # the records are taken at d = 128
        return "%s_d%d" % (kernel, w.d)
    if kernel == "bwd":
        return "bwd" if args.bwd_kernel == 0 else "bwd_pair"
    if kernel != "fwd":
        return kernel
    if args.fwd_kernel == 0:
        return "fwd_pingpong"
    return "fwd_pair"


def _slice(inp, w, b):
    """Rows of sequence b: (q, k, v, do) float64 arrays [L, H, d]."""
    import numpy as np
    cu = inp["cu_seqlens"]
    out = []
    for n in ("q", "k", "v", "do"):
        t = inp[n]
        t = t[b] if cu is None else t[int(cu[b]):int(cu[b + 1])]
        out.append(t.float().numpy().astype(np.float64))
    return out


def cpu_baseline(w, inp, with_bwd, budget_s):
    """The float64 oracle, as it stands, on whole (sequence, head) slices of
    the same workload until ``budget_s`` seconds have been spent (at least one)."""
    from attention_blackwell_gb300 import workloads as W
    from oracle import attention as A

    g = w.Hq // w.Hkv
    done, flops, t0 = 0, 0.0, time.perf_counter()
    while True:
        b, h = divmod(done % (w.B * w.Hq), w.Hq)
        q, k, v, do = _slice(inp, w, b)
        L = q.shape[0]
        A.head_forward(q[:, h], k[:, h // g], v[:, h // g], w.alpha, w.causal)
        flops += W.attention_flops(1, [L], w.causal, d=w.d)
        if with_bwd:
            A.head_backward(q[:, h], k[:, h // g], v[:, h // g], do[:, h], w.alpha, w.causal)
            flops += W.attention_flops(1, [L], w.causal, d=w.d, backward=True)
        done += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": "%d (sequence, head) slices of the %s workload (%d in total), %s, float64 NumPy, %.1f s"
                      % (done, w.name, w.B * w.Hq, "forward+backward" if with_bwd else "forward", dt)}


def build_step(fa, w, dev_t, has_bwd, deterministic):
    """[(name, launch callable, credited FLOPs, launches)] for one step."""
    from attention_blackwell_gb300 import workloads as W
    q, k, v, o, lse = dev_t["q"], dev_t["k"], dev_t["v"], dev_t["o"], dev_t["lse"]
    cu, ms, lens = dev_t["cu"], dev_t["max_seqlen"], dev_t["lengths"]
    ks = [("fwd", lambda: fa.fwd(q, k, v, causal=w.causal, cu_seqlens=cu, max_seqlen=ms, out=o, lse=lse),
           W.attention_flops(w.Hq, lens, w.causal, d=w.d), 1)]
    if has_bwd:
        do, dq, dk, dv, ws = dev_t["do"], dev_t["dq"], dev_t["dk"], dev_t["dv"], dev_t["ws"]

        def stage(s):
            return lambda: fa.bwd(q, k, v, o, lse, do, causal=w.causal, cu_seqlens=cu, max_seqlen=ms,
                                  deterministic=deterministic, workspace=ws, dq=dq, dk=dk, dv=dv, stages=s)
        # status reset + preprocess (+ the varlen work-list plan)
        ks.append(("bwd_pre", stage(1), 0.0, 2 + (cu is not None)))
        ks.append(("bwd", stage(2), W.attention_flops(w.Hq, lens, w.causal, d=w.d, backward=True), 1))
        ks.append(("bwd_post", stage(4), 0.0, 1))
    return ks


def run_ours(args, rank, world):
    import torch

    import attention_blackwell_gb300 as fa
    from attention_blackwell_gb300 import workloads as W

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = W.WORKLOADS[args.workload]
    fa.set_tuning(args.exp2_emu, args.tau)
    fa.set_fwd_kernel(args.fwd_kernel)
    fa.set_bwd_kernel(args.bwd_kernel)
    has_bwd = hasattr(fa, "bwd") and not args.no_bwd
    inp = W.make_inputs(w, with_grad=True)
    t = {n: inp[n].to(dev) for n in ("q", "k", "v", "do")}
    t["o"] = torch.empty_like(t["q"])
    t["lengths"] = inp["lengths"]
    if w.varlen:
        t["cu"], t["max_seqlen"] = inp["cu_seqlens"].to(dev), max(inp["lengths"])
        t["lse"] = torch.empty((w.Hq, inp["T"]), dtype=torch.float32, device=dev)
        n_rows = inp["T"]
    else:
        t["cu"], t["max_seqlen"] = None, None
        t["lse"] = torch.empty((w.B, w.Hq, w.N), dtype=torch.float32, device=dev)
        n_rows = w.N
    if has_bwd:
        t["dq"], t["dk"], t["dv"] = torch.empty_like(t["q"]), torch.empty_like(t["k"]), torch.empty_like(t["v"])
        t["ws"] = fa.bwd_workspace(w.B, w.Hq, n_rows, deterministic=args.deterministic, varlen=w.varlen, d=w.d,
                                   device=dev)
    kernels = build_step(fa, w, t, has_bwd, args.deterministic)
    stream = torch.cuda.current_stream()

    def step(ev=None):
        for i, (_, fn, _, _) in enumerate(kernels):
            if ev is not None:
                ev[i][0].record(stream)
            fn()
            if ev is not None:
                ev[i][1].record(stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    if fa.device_status(t.get("ws")) != 0:
        raise RuntimeError("device status reported a timeout during warm-up")

    K = args.steps
    evs = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in kernels]
           for _ in range(K)]
    clocks = ClockSampler(local) if rank == 0 else None
    if clocks:
        clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    wall0 = time.time()
    t_start.record(stream)
    for s in range(K):
        step(evs[s])
    t_end.record(stream)
    torch.cuda.synchronize()
    wall1 = time.time()
    barrier(world)
    if clocks:
        clocks.stop()
    if fa.device_status(t.get("ws")) != 0:
        raise RuntimeError("device status reported a timeout in the timed region")
    ms_local = t_start.elapsed_time(t_end)
    ms = max_over_ranks(ms_local, world, dev)
    per_kernel = []
    for i, (name, _, fl, nl) in enumerate(kernels):
        d = [evs[s][i][0].elapsed_time(evs[s][i][1]) for s in range(K)]
        per_kernel.append({"kernel": name, "avg_ms": sum(d) / K, "flops": fl, "launches_per_step": nl})
    flops_step = sum(k[2] for k in kernels)
    value = aggregate_tflops(flops_step, K, world, ms)

    # End to end through the public API with host buffers: every step copies
    # its inputs from pinned host memory to the device, runs and copies its
    # results back to pinned host memory.  As in a serving or training loop,
    # consecutive steps overlap: step s's inputs go up on one copy stream
    # while step s-1 computes and step s-2's results come down on another;
    # two device buffer sets alternate, ordered by events.
    ins = ["q", "k", "v"] + (["do"] if has_bwd else [])
    outs = ["o", "lse"] + (["dq", "dk", "dv"] if has_bwd else [])
    host = {n: inp[n].pin_memory() for n in ins}
    host_out = [{n: torch.empty(t[n].shape, dtype=t[n].dtype, pin_memory=True) for n in outs} for _ in range(2)]
    h2d = sum(host[n].numel() * host[n].element_size() for n in ins)
    d2h = sum(host_out[0][n].numel() * host_out[0][n].element_size() for n in outs)
    t2 = dict(t)
    for n in ins + outs:
        t2[n] = torch.empty_like(t[n])
    if has_bwd:
        t2["ws"] = fa.bwd_workspace(w.B, w.Hq, n_rows, deterministic=args.deterministic, varlen=w.varlen, d=w.d,
                                    device=dev)
    sets = [t, t2]
    kern = [kernels, build_step(fa, w, t2, has_bwd, args.deterministic)]
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev_in, ev_comp, ev_out = ([torch.cuda.Event() for _ in range(2)] for _ in range(3))
    E = max(3, args.e2e_steps)

    def e2e_run(nsteps):
        for s in range(nsteps):
            b = s & 1
            T = sets[b]
            with torch.cuda.stream(s_in):
                if s >= 2:
                    s_in.wait_event(ev_comp[b])      # step s-2 has finished with these inputs
                for n in ins:
                    T[n].copy_(host[n], non_blocking=True)
                ev_in[b].record(s_in)
            stream.wait_event(ev_in[b])
            if s >= 2:
                stream.wait_event(ev_out[b])         # step s-2's results have been read back
            for _, fn, _, _ in kern[b]:
                fn()
            ev_comp[b].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_comp[b])
                for n in outs:
                    host_out[b][n].copy_(T[n], non_blocking=True)
                ev_out[b].record(s_out)
        torch.cuda.synchronize()

    e2e_run(2)
    if fa.device_status(t2.get("ws")) != 0:
        raise RuntimeError("device status reported a timeout in the end-to-end warm-up")
    barrier(world)
    e0 = time.perf_counter()
    e2e_run(E)
    e2e_ms = max_over_ranks((time.perf_counter() - e0) * 1e3, world, dev)
    e2e_value = aggregate_tflops(flops_step, E, world, e2e_ms)
    return locals()


def bwd_pairs_resident():
    import attention_blackwell_gb300 as fa
    return fa.bwd_pairs_resident()


def fa_pairs_resident():
    import attention_blackwell_gb300 as fa
    return fa.fwd_pairs_resident()


def describe(w, inp):
    head = "%s: B=%d Hq=%d Hkv=%d d=%d %s" % (w.name, w.B, w.Hq, w.Hkv, w.d, "causal" if w.causal else "non-causal")
    if w.varlen:
        return head + " varlen T=%d lengths U[%d,%d] seed %d" % (inp["T"], w.len_range[0], w.len_range[1], 4)
    return head + " N=%d" % w.N


def emit(line):
    print(json.dumps(line), flush=True)


def main_ours(args):
    rank, world = dist_init(args.gpus)
    r = run_ours(args, rank, world)
    if rank != 0:
        return
    w, K, kernels, per_kernel = r["w"], r["K"], r["kernels"], r["per_kernel"]
    peaks = measured_peaks()
    dom = max(per_kernel, key=lambda p: p["avg_ms"] * p["launches_per_step"])
    achieved = dom["flops"] / (dom["avg_ms"] / 1e3) / 1e12 if dom["flops"] else None
    if peaks and peaks.get("bf16_tflops"):
        peak, peak_src = float(peaks["bf16_tflops"]), "measured burst cuBLAS bf16 (MEASURED_PEAKS.json)"
    else:
        peak, peak_src = 1900.0, "fallback 1.9 PFLOP/s bf16"
    clk = r["clocks"].summary(r["wall0"], r["wall1"]) if r["clocks"] else None
    step_name = "+".join(p["kernel"] for p in per_kernel)
    line = {
        "metric": METRIC,
        "value": round(r["value"], 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": K,
        "warmup": max(3, args.warmup),
        "ms_per_step": round(r["ms"] / K, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": describe(w, r["inp"]),
            "step": step_name, "global_batch": w.B * world, "seq_len": w.N or max(r["inp"]["lengths"]),
            "deterministic_bwd": bool(args.deterministic), "exp2_emu_sixteenths": args.exp2_emu, "tau": args.tau,
            "fwd_kernel": ("one 128-row tile, 64-key blocks (d = 256)" if w.d == 256 else
                           "ping-pong 2x128" if w.d != 128 or args.fwd_kernel == 0 else
                           "CTA pairs, 256-key blocks"),
            "fwd_pairs_resident": fa_pairs_resident(),
            "bwd_kernel": ("128-key tile per head-dim half, 64-row query steps (d = 256)" if w.d == 256 else
                           "one CTA per 128-key tile" if args.bwd_kernel == 0 or w.d != 128
                           else "CTA pairs per 256-key block"),
            "bwd_pairs_resident": bwd_pairs_resident(),
            "parallelism": "replicas" if world > 1 else "single",
            "l2": "no flush: the step's inputs (%.0f MiB) exceed the 126 MB L2" % (
                sum(r["t"][n].numel() * 2 for n in ("q", "k", "v", "do")) / 2 ** 20)},
        "pct_of_2.25PF": round(100.0 * r["value"] / PEAK_NOMINAL_TFLOPS, 2),
        "breakdown": [{"kernel": p["kernel"], "avg_ms": round(p["avg_ms"], 4),
                       "tflops": round(p["flops"] / (p["avg_ms"] / 1e3) / 1e12, 1) if p["flops"] else None}
                      for p in per_kernel],
        "roofline": {"kernel": dom["kernel"], "bound": "tensor",
                     "achieved": round(achieved, 1) if achieved else None, "peak": peak,
                     "unit": "TFLOP/s", "frac": round(achieved / peak, 4) if achieved else None,
                     "peak_source": peak_src,
                     "frac_of_sustained": round(achieved / float(peaks["bf16_tflops_sustained"]), 4)
                     if achieved and peaks and peaks.get("bf16_tflops_sustained") else None,
                     "traffic": kernel_traffic(traffic_key(args, w, dom["kernel"]), w.name)},
        "e2e": {"value": round(r["e2e_value"], 2), "unit": "TFLOP/s", "h2d_bytes_per_step": r["h2d"],
                "d2h_bytes_per_step": r["d2h"], "steps": r["E"],
                "note": "public API, pinned host buffers, copies of step s overlap compute of step s-1; "
                        "the timed steps include the first upload and the last download"},
        "gpu_launches": K * sum(p["launches_per_step"] for p in per_kernel),
        "clocks": clk,
    }
    line["cpu_baseline"] = cpu_baseline(w, r["inp"], r["has_bwd"], args.cpu_seconds)
    emit(line)


def main_reference(args):
    """The CPU oracle as the reference arm (rank 0 only)."""
    rank, world = int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1"))
    if rank != 0:
        return
    import numpy as np

    from attention_blackwell_gb300 import workloads as W
    from oracle import attention as A

    w = W.WORKLOADS[args.workload]
    with_bwd = not args.no_bwd   # the same step as ours
    inp = W.make_inputs(w, with_grad=True)

    def step(s):  # one (sequence, head) slice of the workload per step
        b, h = divmod(s % (w.B * w.Hq), w.Hq)
        hk = h // (w.Hq // w.Hkv)
        q, k, v, do = _slice(inp, w, b)
        L = q.shape[0]
        A.head_forward(q[:, h], k[:, hk], v[:, hk], w.alpha, w.causal)
        f = W.attention_flops(1, [L], w.causal, d=w.d)
        if with_bwd:
            A.head_backward(q[:, h], k[:, hk], v[:, hk], do[:, h], w.alpha, w.causal)
            f += W.attention_flops(1, [L], w.causal, d=w.d, backward=True)
        return f

    for s in range(max(1, args.warmup)):
        step(s)
    t0 = time.perf_counter()
    flops = sum(step(s) for s in range(args.steps))
    dt = time.perf_counter() - t0
    value = flops / dt / 1e12
    sample = "one (sequence, head) slice of the %s workload per step (%s), float64 NumPy" % (
        w.name, "forward+backward" if with_bwd else "forward")
    emit({"impl": "reference", "metric": METRIC, "value": round(value, 5), "unit": "TFLOP/s", "n_gpus": world,
          "steps": args.steps, "warmup": max(1, args.warmup), "ms_per_step": round(dt * 1e3 / args.steps, 2),
          "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
          "config": {"workload": describe(w, inp), "step": "oracle slice"},
          "cpu_baseline": {"value": round(value, 5), "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
                           "sample": sample},
          "e2e": {"value": round(value, 5), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}})


if __name__ == "__main__":
    a = parse()
    if a.impl == "reference":
        main_reference(a)
    else:
        main_ours(a)
