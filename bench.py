#!/usr/bin/env python
"""Attention forward+backward throughput on GB300, all three numerical modes.

One step = fa_fwd + fa_bwd in the baseline, stabilised and FP32-output modes
on the GPT-2-small attention training shape (B=8, H=12, N=1024, d=64, causal,
scale 1/8; seeded synthetic BF16 inputs with 5% planted tied-max rows).
Throughput counts 12*d algorithmic FLOP per visible (query, key) pair per mode
(4d forward: QK^T and PV; 8d backward: dP, dV, dK, dQ; the backward's
recomputation of S is not counted).  The timed steps run as one launch of a
CUDA graph captured from the fa_fwd / fa_bwd_noalloc calls (fa_bwd where the
no-alloc scratch is too small; the L2 flush and the step and mode events are
graph nodes too); the end-to-end figure runs fa_fwd / fa_bwd call by call
with the host copies.  --workload selects another input set for profiling
(gpt2m, long, ties); the headline is gpt2s.

Prints one JSON line.  ``--impl reference`` times the CPU FP64 oracle instead
(the only reference implementation of this method available), on a bounded
sample of the same workload.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
For N > 1 launch with torch.distributed.run; each rank runs the full workload
on its own GPU (weak scaling, no collective on the data path).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "attention fwd+bwd TFLOPS/s on 1 GB300 (% of dense BF16 peak), per mode"
WORKLOAD = "gpt2-small attention training shape: B=8 H=12 N=1024 d=64 causal, fwd+bwd x 3 modes"
MODES = [("baseline", 0), ("stabilised", 1), ("fp32_out", 2)]
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# files whose contents define the backward / forward kernels (for the traffic record)
KERNEL_SOURCES = {
    "bwd_main": ["precision_flash_attention_attn_gb300/csrc/fa_bwd.cu",
                 "precision_flash_attention_attn_gb300/csrc/fa_ptx.cuh",
                 "precision_flash_attention_attn_gb300/csrc/fa_internal.h"],
    "fwd": ["precision_flash_attention_attn_gb300/csrc/fa_fwd.cu",
            "precision_flash_attention_attn_gb300/csrc/fa_ptx.cuh",
            "precision_flash_attention_attn_gb300/csrc/fa_internal.h"],
}
# algorithmic FLOP per visible pair of each timed kernel (per launch = x pairs)
KERNEL_FLOP_PER_PAIR_D = {"fwd": 4, "bwd_main": 8}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=600)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target CPU time of the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", default="gpt2s", choices=["gpt2s", "gpt2m", "long", "ties"],
                    help="input set of the GPU arm (the headline is gpt2s; the others are for profiling)")
    return ap.parse_args()


def workload_name(case) -> str:
    if case.spec.name == "gpt2s":
        return WORKLOAD
    kind = "causal" if case.causal else "full"
    return f"{case.spec.name} attention: B={case.B} H={case.H} N={case.N} d={case.d} {kind}, fwd+bwd x 3 modes"


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(x: float, dist=None, device="cpu") -> float:
    """Maximum of a per-rank float over all ranks (identity without a group)."""
    if dist is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def visible_pairs(B, H, N, causal):
    return B * H * (N * (N + 1) // 2 if causal else N * N)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def sources_sha(kernel):
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES.get(kernel, []):
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def recorded_traffic(kernel, workload="gpt2s"):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current sources of that kernel and on the same workload."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        rec = json.load(f).get(kernel)
    if not rec or rec.get("source_sha256") != sources_sha(kernel) or rec.get("workload") != workload:
        return None
    return rec.get("dram_bytes_per_launch")


# ---------------------------------------------------------------- clocks ----

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "50"]
        if self.gpu_index is not None:
            cmd += ["-i", str(self.gpu_index)]
        try:
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(cmd, stdout=self.out, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        self.t0 = time.time()

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.close()
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                    power.append(float(parts[3]))
                except ValueError:
                    continue
                for nm, val in zip(names, parts[5:9]):
                    if val.lower().startswith("active"):
                        reasons.add(nm)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# ------------------------------------------------------------ CPU oracle ----

def oracle_sample(case, heads, modes):
    """Run the FP64 oracle forward+backward on whole heads; returns seconds."""
    from oracle import oracle as orc
    BH = case.B * case.H
    arr = {n: case.f64(n).reshape(BH, case.N, case.d).astype("float32") for n in ("q", "k", "v", "do")}
    t0 = time.perf_counter()
    for h in heads:
        sl = slice(h, h + 1)
        for _mode in modes:
            f = orc.fwd(arr["q"][sl], arr["k"][sl], arr["v"][sl], case.causal, case.scale, _mode,
                        dout=arr["do"][sl])
            orc.bwd(arr["q"][sl], arr["k"][sl], arr["v"][sl], arr["do"][sl], case.causal, case.scale,
                    lse=f["lse"], delta=f["delta"])
    return time.perf_counter() - t0


def cpu_baseline(case, target_s):
    from oracle import oracle as orc
    orc.build()
    flop_head = 12 * case.d * (case.N * (case.N + 1) // 2 if case.causal else case.N * case.N)
    modes = [m for _, m in MODES]
    oracle_sample(case, [0], [0])                      # warm (page-in, thread pool)
    spent, heads = 0.0, 0
    BH = case.B * case.H
    while heads < BH and (spent < target_s or heads == 0):
        spent += oracle_sample(case, [heads], modes)
        heads += 1
    flops = flop_head * len(modes) * heads
    return {"value": flops / spent / 1e12, "unit": "TFLOP/s", "cores": orc.num_threads(),
            "kind": "oracle",
            "sample": f"{heads} of {BH} heads x 3 modes, full fwd+bwd in FP64 ({spent:.1f} s)"}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    from precision_flash_attention_attn_gb300.inputs import make_case
    from oracle import oracle as orc
    orc.build()
    case = make_case("gpt2s")
    modes = [m for _, m in MODES]
    flop_head = 12 * case.d * (case.N * (case.N + 1) // 2)
    for s in range(args.warmup):
        oracle_sample(case, [s % (case.B * case.H)], modes)
    times = []
    for s in range(args.steps):
        times.append(oracle_sample(case, [(args.warmup + s) % (case.B * case.H)], modes))
    total = sum(times)
    flops = flop_head * len(modes) * args.steps
    value = flops / total / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": WORKLOAD + " (oracle: one head per step)", "B": case.B, "H": case.H,
                   "N": case.N, "d": case.d, "causal": True},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": orc.num_threads(), "kind": "oracle",
                         "sample": "one of 96 heads per step, 3 modes, full fwd+bwd in FP64"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ GPU -----

def run_ours(args):
    import numpy as np
    import torch

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        dist = None
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())

    import __graft_entry__
    __graft_entry__.build()
    from precision_flash_attention_attn_gb300 import fa
    from precision_flash_attention_attn_gb300.inputs import make_case

    case = make_case(args.workload)
    B, H, N, d, causal, scale = case.B, case.H, case.N, case.d, case.causal, case.scale
    pairs = visible_pairs(B, H, N, causal)
    flop_mode = 12 * d * pairs
    flop_step = flop_mode * len(MODES)

    def to_dev(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)

    q, k, v, do = (to_dev(getattr(case, n)) for n in ("q", "k", "v", "do"))
    outs = {}
    for name, m in MODES:
        outs[m] = dict(
            o=torch.empty((B, H, N, d), device=dev, dtype=torch.float32 if m == 2 else torch.bfloat16),
            lse=torch.empty((B, H, N), device=dev, dtype=torch.float32),
            dq=torch.empty_like(q), dk=torch.empty_like(q), dv=torch.empty_like(q))
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)   # 2x the 129 MB L2

    def one_mode(m, qq=q, kk=k, vv=v, gg=do, st=stream, bwd=fa.fa_bwd):
        b = outs[m]
        fa.fa_fwd(qq, kk, vv, b["o"], b["lse"], B, H, N, d, causal, scale, m, st)
        bwd(qq, kk, vv, b["o"], b["lse"], gg, b["dq"], b["dk"], b["dv"], B, H, N, d, causal, scale, m, st)

    # the allocation-free backward where its static scratch holds the workspace
    ws_bytes = B * H * N * d * 4 + 2 * B * H * ((N + 127) // 128 * 128) * 4
    bwd_timed = fa.fa_bwd_noalloc if ws_bytes <= fa.NOALLOC_SCRATCH_BYTES else fa.fa_bwd
    bwd_name = "fa_bwd_noalloc" if bwd_timed is fa.fa_bwd_noalloc else "fa_bwd"
    for _ in range(args.warmup):
        for _, m in MODES:
            flush.zero_()
            one_mode(m, bwd=bwd_timed)
    torch.cuda.synchronize()
    if fa.fa_device_status() != 0:
        raise RuntimeError("kernel timeout during warm-up")

    # The K timed steps are captured, with the L2 flush between steps and an
    # event at every mode boundary, into one CUDA graph that is launched once:
    # a step enqueued call by call costs more host time than its GPU time.
    # An event-record node between two kernels costs about 3 us, so the
    # per-kernel events (library profiling) go into a second graph of the same
    # K steps, launched once right after; it gives the per-kernel durations.
    # Where capture is unavailable the steps are launched call by call.
    def capture(kernel_events):
        evs = [[torch.cuda.Event(enable_timing=True, external=True) for _ in range(2 * len(MODES))]
               for _ in range(args.steps)]
        g = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream()
        if kernel_events:
            fa.fa_profile_start()
        try:
            with torch.cuda.graph(g, stream=cap):
                for s in range(args.steps):
                    for i, (_, m) in enumerate(MODES):
                        flush.zero_()       # every mode starts with a cold L2
                        evs[s][2 * i].record(cap)
                        one_mode(m, st=cap, bwd=bwd_timed)
                        evs[s][2 * i + 1].record(cap)
        except Exception:
            if kernel_events:
                fa.fa_profile_stop()
            raise
        return g, evs

    graph = graph_k = ev_k = None
    timing = (f"one CUDA graph launch of the {args.steps} steps (captured fa_fwd + {bwd_name} calls); "
              "per-kernel durations from a second launch with an event pair per kernel")
    try:
        graph, ev = capture(False)
        # its profiling session stays open until after its launch; the graph's
        # event-record nodes need their events alive as long as the graph
        graph_k, ev_k = capture(True)
    except Exception as exc:  # noqa: BLE001 - any capture failure falls back to eager launches
        graph = graph_k = ev_k = None
        timing = f"eager launches (graph capture unavailable: {type(exc).__name__})"
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2 * len(MODES))] for _ in range(args.steps)]
    torch.cuda.synchronize()
    gpu_index = None
    cvd = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    ids = [x for x in cvd.split(",") if x.strip()]
    if ids:
        gpu_index = ids[dev.index] if dev.index < len(ids) else None
    else:
        gpu_index = dev.index
    sampler = ClockSampler(gpu_index)
    sampler.start()
    time.sleep(0.3)
    if graph is None:
        fa.fa_profile_start()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    if graph is not None:
        # Untimed launches of the same graph for about half a second first, so
        # that the clock sampler sees the GPU under this load (the timed launch
        # itself can be shorter than the sampling interval); the timed launch
        # below overwrites every event these record.
        t_pre = time.time()
        while time.time() - t_pre < 0.5:
            graph.replay()
            torch.cuda.synchronize()
        for _, m in MODES:                  # every output must come from the graph launch
            for kname in ("dq", "dk", "dv"):
                outs[m][kname].fill_(float("nan"))
        graph.replay()
        wrote = all(bool(torch.isfinite(outs[m][kname]).all()) for _, m in MODES for kname in ("dq", "dk", "dv"))
        if not wrote:
            raise RuntimeError("the graph launch left gradient buffers unwritten")
        graph_k.replay()                    # the same K steps with an event pair per kernel
    else:
        for s in range(args.steps):
            e = ev[s]
            for i, (_, m) in enumerate(MODES):
                flush.zero_()                   # L2 flushed before every mode, outside the events
                e[2 * i].record(stream)
                one_mode(m, bwd=bwd_timed)
                e[2 * i + 1].record(stream)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    prof = fa.fa_profile_stop()
    clocks = sampler.stop()
    if fa.fa_device_status() != 0:
        raise RuntimeError("kernel timeout during the timed region")

    # The timed launches computed what the same calls compute eagerly (the
    # calls the parity tests check): O, LSE, dK and dV bit for bit, dQ up to
    # the order of the FP32 reduce-adds into its accumulator.
    same_as_eager = True
    for _, m in MODES:
        got = outs[m]
        ref = {kname: torch.empty_like(t) for kname, t in got.items()}
        fa.fa_fwd(q, k, v, ref["o"], ref["lse"], B, H, N, d, causal, scale, m, stream)
        bwd_timed(q, k, v, ref["o"], ref["lse"], do, ref["dq"], ref["dk"], ref["dv"], B, H, N, d, causal, scale,
                  m, stream)
        torch.cuda.synchronize()
        exact = all(torch.equal(got[kname], ref[kname]) for kname in ("o", "lse", "dk", "dv"))
        dq_diff = float((got["dq"].float() - ref["dq"].float()).norm())
        dq_norm = float(ref["dq"].float().norm())
        dq_rel = dq_diff / dq_norm if dq_norm > 0 else dq_diff   # dQ is all zero where each row sees one key
        if not exact or not dq_rel <= 1e-4:
            same_as_eager = False
    if not same_as_eager:
        raise RuntimeError("the timed launches' outputs differ from the same calls made eagerly")

    per_mode_ms = [0.0] * len(MODES)
    for e in ev:
        for i in range(len(MODES)):
            per_mode_ms[i] += e[2 * i].elapsed_time(e[2 * i + 1])
    graph = graph_k = None                  # release the graphs before the events they record
    total_ms = max_over_ranks(sum(per_mode_ms), dist, dev)
    ms_step = total_ms / args.steps
    value = world * flop_step * args.steps / (total_ms * 1e-3) / 1e12

    # ---------------------------------------------------------- end to end --
    pin = {n: torch.from_numpy(np.ascontiguousarray(getattr(case, n)).view(np.int16)).pin_memory()
           for n in ("q", "k", "v", "do")}
    dq_in = {n: torch.empty((B, H, N, d), device=dev, dtype=torch.bfloat16) for n in pin}
    host_out = {m: {kname: torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for kname, t in outs[m].items()}
                for _, m in MODES}
    h2d = sum(t.numel() * t.element_size() for t in pin.values())
    d2h = sum(t.numel() * t.element_size() for m in host_out for t in host_out[m].values())
    e2e_ms = 0.0
    e2e_steps = max(3, args.steps // 4)
    if dist is not None:
        dist.barrier()
    # Each mode's outputs go to the host on a copy stream while the next mode
    # computes; the step ends when the last copy has landed.
    copy_stream = torch.cuda.Stream()
    for s in range(e2e_steps + 2):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for n in pin:
            dq_in[n].view(torch.int16).copy_(pin[n], non_blocking=True)
        for _, m in MODES:
            one_mode(m, dq_in["q"], dq_in["k"], dq_in["v"], dq_in["do"])
            done = torch.cuda.Event()
            done.record(stream)
            copy_stream.wait_event(done)
            with torch.cuda.stream(copy_stream):
                for kname, t in outs[m].items():
                    host_out[m][kname].copy_(t, non_blocking=True)
        stream.wait_stream(copy_stream)
        b.record(stream)
        b.synchronize()
        if s >= 2:
            e2e_ms += a.elapsed_time(b)
    e2e_ms = max_over_ranks(e2e_ms, dist, dev)
    e2e_value = world * flop_step * e2e_steps / (e2e_ms * 1e-3) / 1e12

    # The same copies alone, back to back on the stream (best of 3).  A step
    # cannot end before its inputs are in, its first mode has run and every
    # output is out, so these give the end-to-end number's own bound.
    def copies_ms(issue):
        best = None
        for _ in range(3):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            issue()
            b.record(stream)
            b.synchronize()
            best = a.elapsed_time(b) if best is None else min(best, a.elapsed_time(b))
        return best

    def issue_h2d():
        for n in pin:
            dq_in[n].view(torch.int16).copy_(pin[n], non_blocking=True)

    def issue_d2h():
        for _, m in MODES:
            for kname, t in outs[m].items():
                host_out[m][kname].copy_(t, non_blocking=True)

    h2d_ms, d2h_ms = copies_ms(issue_h2d), copies_ms(issue_d2h)
    e2e_bound_ms = h2d_ms + per_mode_ms[0] / args.steps + d2h_ms

    # ------------------------------------------- fa_bwd against fa_bwd_noalloc --
    # The same backward through both entry points, called eagerly one by one
    # (fa_bwd allocates its workspace from the stream's pool, clears its
    # barrier words and frees it; fa_bwd_noalloc uses the static scratch),
    # each bracketed by events right after a forward keeps the GPU busy.
    alloc_cmp = None
    if ws_bytes <= fa.NOALLOC_SCRATCH_BYTES:
        tot = {"fa_bwd": 0.0, "fa_bwd_noalloc": 0.0}
        n_cmp = max(5, args.steps // 2)
        for s in range(n_cmp + 2):
            for bname, bfn in (("fa_bwd", fa.fa_bwd), ("fa_bwd_noalloc", fa.fa_bwd_noalloc)):
                for _, m in MODES:
                    b = outs[m]
                    flush.zero_()
                    fa.fa_fwd(q, k, v, b["o"], b["lse"], B, H, N, d, causal, scale, m, stream)
                    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    a0.record(stream)
                    bfn(q, k, v, b["o"], b["lse"], do, b["dq"], b["dk"], b["dv"], B, H, N, d, causal, scale, m,
                        stream)
                    a1.record(stream)
                    a1.synchronize()
                    if s >= 2:
                        tot[bname] += a0.elapsed_time(a1)
        alloc_cmp = {"fa_bwd_ms": tot["fa_bwd"] / (n_cmp * len(MODES)),
                     "fa_bwd_noalloc_ms": tot["fa_bwd_noalloc"] / (n_cmp * len(MODES)),
                     "ratio": tot["fa_bwd"] / tot["fa_bwd_noalloc"], "calls_each": n_cmp * len(MODES),
                     "how": "eager calls after a forward, events around the backward call, L2 flushed first"}
    if fa.fa_device_status() != 0:
        raise RuntimeError("kernel timeout or non-finite output after the timed region")

    # ------------------------------------------------------------ roofline --
    peaks, peak_src = load_peaks()
    timed = {kname: v for kname, v in prof.items() if v[0] > 0}
    dom = max(timed, key=lambda kk: timed[kk][1])
    launches, dom_ms = timed[dom]
    avg_ms = dom_ms / launches
    per_pair = KERNEL_FLOP_PER_PAIR_D.get(dom)
    roof = None
    if per_pair is not None:
        flop_launch = per_pair * d * pairs
        achieved = flop_launch / (avg_ms * 1e-3) / 1e12
        peak = float(peaks["bf16_tflops"])
        roof = {"kernel": dom, "bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": recorded_traffic(dom, args.workload),
                "flop_per_launch": flop_launch, "avg_launch_ms": avg_ms,
                "peak_source": f"bf16_tflops (burst) of {peak_src}"}
    kernel_share = {kname: {"launches": v[0], "total_ms": v[1], "share": v[1] / sum(x[1] for x in timed.values())}
                    for kname, v in timed.items()}
    gpu_launches = sum(v[0] for v in timed.values())

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": workload_name(case), "B": B, "H": H, "N": N, "d": d, "causal": causal, "scale": scale,
                   "modes": [n for n, _ in MODES], "planted_tie_rows": 0.05,
                   "flop_per_step": flop_step, "flop_convention": "12*d per visible pair per mode",
                   "l2": "flushed before every mode's fwd+bwd (256 MiB write, outside the timed events)",
                   "timing": timing},
        "frac_of_peak": value / world / float(peaks["bf16_tflops"]),
        "peak_source": f"bf16_tflops {peaks['bf16_tflops']} ({peak_src})",
        "per_mode": {n: {"ms": per_mode_ms[i] / args.steps,
                         "tflops": flop_mode / (per_mode_ms[i] / args.steps * 1e-3) / 1e12}
                     for i, (n, _) in enumerate(MODES)},
        "stabilised_overhead": per_mode_ms[1] / per_mode_ms[0] - 1.0,
        "bwd_alloc_vs_noalloc": alloc_cmp,
        "roofline": roof,
        "kernels": kernel_share,
        "gpu_launches": gpu_launches,
        "outputs_match_eager_calls": same_as_eager,
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps": e2e_steps, "ms_per_step": e2e_ms / e2e_steps,
                "copy_bound": {"h2d_ms": h2d_ms, "d2h_ms": d2h_ms,
                               "h2d_gbs": h2d / (h2d_ms * 1e-3) / 1e9, "d2h_gbs": d2h / (d2h_ms * 1e-3) / 1e9,
                               "bound_ms_per_step": e2e_bound_ms,
                               "frac": e2e_bound_ms / (e2e_ms / e2e_steps),
                               "how": "inputs in, then the first mode, then every output out, each timed "
                                      "alone (copies best of 3, pinned host memory)"}},
        "clocks": clocks,
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(case, args.cpu_seconds)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def main():
    args = parse_args()
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
