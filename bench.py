"""Throughput of causal linear attention (phi = elu + 1) on one GB300 per rank.

Default workload: causal forward + backward, bf16 inputs with fp32
accumulation, B=2 H=16 N=65536 Dk=Dv=128 (Q, K ~ N(0,1)/sqrt(128), V, dO ~
N(0,1), seed 5).  One step = la_causal_fwd + la_causal_bwd_after_fwd over that
batch (feature map, intra-chunk products, chunk-state scan; the backward takes
the per-segment forward states from the forward's workspace and recomputes
everything per position).  The inputs (2.1 GB) are far larger than L2, so consecutive steps
cannot reuse cached data.

Printed on rank 0 as one JSON line:
  value       tokens/s (B*N*ranks / step time), inputs resident in HBM; the timed
              region holds the K steps and two CUDA events, nothing else
  e2e         the same through the C ABI with host buffers (la_causal_step_host):
              pinned-host q, k, v, dO in and o, dq, dk, dv out inside the timed
              region, transfers overlapped with the kernels over groups of heads
  roofline    the dominant kernel against the measured HBM copy bandwidth, its
              duration from a separate instrumented pass of the same steps
  decode      recurrent step at B=64 H=8 D=32, 3072 and 784 steps, and at B=8000
              (state larger than L2), CUDA graphs of single-step launches
  noncausal   the non-causal forward and backward at B=4 H=8 N=1024 D=64 bf16, and at
              B=2 H=16 N=65536 D=128 bf16
  sweep       causal fwd+bwd at B=1 H=8 D=64 bf16 for N = 2^9 .. 2^16: time,
              tokens/s and peak device memory per N
  cpu_baseline  the fp64 oracle on a bounded sample of the same workload

`--impl reference` times the fp64 CPU oracle on the same workload instead
(the only reference that exists for this method: it is not a GPU program).
Multi-GPU (torchrun): every rank runs its own replica of the batch (heads are
independent), no collective on the data path; time is the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from causal_linear_attention_phi_gb300 import workloads as W  # noqa: E402

PEAKS_PATH = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_PATH = os.path.join(ROOT, "profiles", "tc_kernels_B1_H16_N32768_D128_dram_traffic.json")
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


# ------------------------------------------------------------------ helpers
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x: float) -> float:
    """Max of a per-rank float over the process group (identity when not distributed).
    Uses a CUDA tensor under NCCL and a CPU tensor under gloo."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_value(tokens_per_rank_step: int, world: int, ms_per_step_max: float) -> float:
    """Whole-job throughput: every rank processes its own batch; time is the slowest rank's."""
    return tokens_per_rank_step * world / (ms_per_step_max / 1e3)


def peaks():
    try:
        with open(PEAKS_PATH) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []   # (arrival time, csv line)
        self.t_start = None
        self.t_stop = None

    def mark_start(self):
        self.t_start = time.perf_counter()

    def mark_stop(self):
        self.t_stop = time.perf_counter()

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line.strip()))

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        lines = self.lines
        if self.t_start is not None and self.t_stop is not None:
            # the samples taken while the timed region ran (plus the one just after it, which
            # covers its last 20 ms); all of them if none arrived in that window
            inside = [x for x in lines if self.t_start <= x[0] <= self.t_stop + 0.03]
            lines = inside or lines
        for _, l in lines:
            parts = [x.strip() for x in l.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# The sources of the tensor-core kernels that the committed DRAM-traffic figures describe
# (kernels, shared device code and the headers they include): any change to these makes
# the figures stale; changes to other kernels (the scans, the CUDA-core path) do not.
TC_KERNEL_SOURCES = ("tc_fwd.cu", "tc_bwd.cu", "tc_retention.cu", "tc_apply.cu", "tc_noncausal_bwd.cu",
                     "tc_common.cuh", "sm100.cuh", "la_internal.cuh")


def kernel_sources_sha():
    h = hashlib.sha256()
    for name in TC_KERNEL_SOURCES:
        with open(os.path.join(ROOT, "causal_linear_attention_phi_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str):
    """DRAM bytes per launch from a committed ncu summary, if taken on the current kernels."""
    try:
        with open(TRAFFIC_PATH) as f:
            t = json.load(f)
    except Exception:
        return None
    if t.get("sources_sha") != kernel_sources_sha():
        return None
    k = t.get("kernels", {}).get(kernel)
    return None if k is None else float(k["dram_bytes_per_launch"])


# Compulsory HBM bytes per launch of each kernel (its own inputs and outputs,
# each counted once), for the long bf16 workload.  units = token-heads.
def kernel_algorithmic_bytes(name: str, B, H, N, Dk, Dv, sz):
    T = B * H * N
    table = {
        "segment_sums": T * (Dk + Dv) * sz,                       # read k, v
        "causal_fwd_out": T * (2 * Dk + 2 * Dv) * sz,             # read q, k, v; write o
        "causal_fwd_fused": T * (2 * Dk + 2 * Dv) * sz,           # read q, k, v; write o (the second read of
                                                                  # k, v for the segment sums is not counted)
        "bwd_forward_sweep": T * ((2 * Dk + 2 * Dv) * sz + Dk * sz + 8),   # read q,k,v,dO; write dq, (den,g)
        "bwd_reverse_sweep": T * ((2 * Dk + 2 * Dv) * sz + 8 + (Dk + Dv) * sz),  # read q,k,v,dO,(den,g); write dk,dv
    }
    for key, val in table.items():
        if key in name:
            return val
    return None


# ------------------------------------------------------------------ our implementation
def run_ours(args):
    import causal_linear_attention_phi_gb300 as la

    ws_n, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if ws_n > 1:
        import datetime
        import torch.distributed as dist
        dist.init_process_group("nccl", timeout=datetime.timedelta(minutes=10))
    la.build.build_library()
    la.library()
    la.clear_error()
    # the decode step first, on a fresh device allocator (it is independent of the main
    # workload, whose 8 GB of buffers would otherwise shape where its small buffers land)
    decode = bench_decode(la, dev, peaks()[0]) if (rank == 0 and not args.skip_extras) else None
    ret_step = bench_retention_step(la, dev) if (rank == 0 and not args.skip_extras) else None

    w = W.LONG_BF16
    if args.workload == "profile":
        # same recipe, half the heads and half the length (inputs 0.5 GB, still far above L2)
        import dataclasses
        w = dataclasses.replace(w, name="causal fwd+bwd bf16 B=1 H=16 N=32768 Dk=Dv=128", B=1, N=32768)
    B, H, N, Dk, Dv = w.B, w.H, w.N, w.Dk, w.Dv
    q, k, v, dO = W.make_inputs(w, with_grad=True)
    qd, kd, vd, dOd = (t.to(dev) for t in (q, k, v, dO))
    o = torch.empty_like(vd)
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    ws_f = torch.empty(la.workspace_bytes(la.OP_CAUSAL_FWD, B, H, N, Dk, Dv, w.dtype), dtype=torch.uint8, device=dev)
    ws_b = torch.empty(la.workspace_bytes(la.OP_CAUSAL_BWD, B, H, N, Dk, Dv, w.dtype), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        la.causal_fwd(qd, kd, vd, out=o, workspace=ws_f)
        la.causal_bwd(qd, kd, vd, dOd, dq=dq, dk=dk, dv=dv, workspace=ws_b, fwd_workspace=ws_f)

    def barrier():
        if ws_n > 1:
            import torch.distributed as dist
            dist.barrier()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert la.last_error() == 0

    # ---- timed region: device events on the launch stream around K steps, nothing else
    # recorded inside it
    barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        time.sleep(0.1)  # the sampler's first reading lands before the timed region starts
        clk.mark_start()
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
        clk.mark_stop()
    barrier()
    # ---- per-kernel split from a separate pass of the same steps with the library's
    # per-launch events on (outside the timed region)
    inst_steps = min(args.steps, 10)
    la.timing_reset()
    la.timing_enable(True)
    for _ in range(inst_steps):
        step()
    torch.cuda.synchronize()
    la.timing_enable(False)
    ktimes = la.timing_read()
    if args.workload == "profile":
        # two one-launch causal forwards, two retention forwards, two non-causal forwards and two
        # non-causal backwards at the same shape, outside the timed region, so that one small
        # command also covers their kernels in an ncu capture
        gam = W.retention_gammas(H).to(dev)
        for _ in range(2):
            la.causal_fwd(qd, kd, vd, out=o, one_launch=True)
        for _ in range(2):
            la.retention_fwd(qd, kd, vd, gam, out=o)
        for _ in range(2):
            la.noncausal_fwd(qd, kd, vd, out=o)
        for _ in range(2):
            la.noncausal_bwd(qd, kd, vd, dOd, dq=dq, dk=dk, dv=dv)
        torch.cuda.synchronize()
    ms_total = max_over_ranks(e0.elapsed_time(e1))
    ms_step = ms_total / args.steps
    tokens_per_step = B * N * ws_n
    value = weak_scaling_value(B * N, ws_n, ms_step)
    launches_per_step = sum(c for c, _ in ktimes.values()) / inst_steps
    launches = int(round(launches_per_step * args.steps))
    assert la.last_error() == 0

    # ---- roofline of the dominant kernel
    hbm, tc_peak, peak_kind = peaks()
    dom = max(ktimes.items(), key=lambda kv: kv[1][1])
    dom_name, (dom_n, dom_ms) = dom
    avg_ms = dom_ms / dom_n
    alg = kernel_algorithmic_bytes(dom_name, B, H, N, Dk, Dv, 2)
    achieved = alg / (avg_ms / 1e3) / 1e9 if alg else None
    traffic = ncu_traffic(dom_name)
    roofline = {"kernel": dom_name, "bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                "frac": (achieved / hbm) if achieved else None, "traffic": traffic,
                "peak_source": peak_kind + " (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured" else peak_kind,
                "algorithmic_bytes_per_launch": alg, "avg_launch_ms": avg_ms}
    step_alg_bytes = B * H * N * ((2 * Dk + 2 * Dv) + (4 * Dk + 3 * Dv)) * 2
    step_roof = {"algorithmic_bytes": step_alg_bytes,
                 "achieved_gbs": step_alg_bytes / (ms_step / 1e3) / 1e9,
                 "frac": step_alg_bytes / (ms_step / 1e3) / 1e9 / hbm}

    result = {
        "metric": "causal lin-attn fwd+bwd tokens/s @N=64K; decode steps/s; % of roofline",
        "value": value, "unit": "tokens/s", "n_gpus": ws_n, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic (seeded N(0,1) inputs, no dataset)",
        "config": {"workload": w.name, "B": B, "H": H, "N": N, "Dk": Dk, "Dv": Dv,
                   "global_batch": B * ws_n, "seq_len": N, "parallelism": "replicas over heads/batch (dp%d)" % ws_n,
                   "l2": "inputs (2.1 GB) larger than L2; no flush needed"},
        "kernel_times_ms": {n: {"launches": c, "total_ms": round(t, 4), "avg_ms": round(t / c, 5)}
                            for n, (c, t) in ktimes.items()},
        "kernel_times_from": "a separate pass of %d steps with per-launch CUDA events, after the timed region "
                             "(the timed region itself carries no instrumentation)" % inst_steps,
        "gpu_launches": launches,
        "roofline": roofline,
        "step_roofline": step_roof,
        "clocks": clk.summary(),
    }

    # ---- end to end through the C ABI with host buffers (pinned host in, host out):
    # la_causal_step_host pipelines the transfers and the kernels over groups of heads
    if not args.skip_e2e:
        host_in = [t.pin_memory() for t in (q, k, v, dO)]
        host_out = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in (v, q, k, v)]  # o, dq, dk, dv
        h2d = sum(t.numel() * t.element_size() for t in host_in)
        d2h = sum(t.numel() * t.element_size() for t in host_out)
        group = 2
        dev_buf = torch.empty(la.host_step_bytes(B, H, N, Dk, Dv, w.dtype, group), dtype=torch.uint8, device=dev)

        def e2e_step():
            la.causal_step_host(*host_in, *host_out, group_heads=group, dev_buf=dev_buf)

        e2e_steps = max(2, min(args.steps, 5))
        e2e_step()
        torch.cuda.synchronize()
        barrier()
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        for _ in range(e2e_steps):
            e2e_step()
        a1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(a0.elapsed_time(a1) / e2e_steps)
        result["e2e"] = {"value": tokens_per_step / (e2e_ms / 1e3), "unit": "tokens/s",
                         "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                         "how": "la_causal_step_host: pinned host q, k, v, dO in and o, dq, dk, dv out, transfers "
                                "and kernels pipelined over groups of %d heads" % group}
        del host_in, host_out, dev_buf

    # ---- decode and non-causal sub-measurements (rank 0 only, not part of value)
    if rank == 0 and not args.skip_extras:
        result["decode"] = decode
        result["noncausal"] = bench_noncausal(la, dev)
        result["retention"] = bench_retention(la, dev)
        result["retention"]["step"] = ret_step
        result["forward_forms"] = bench_forward_forms(la, dev)
        result["sweep"] = {"workload": "causal fwd+bwd bf16 B=1 H=8 Dk=Dv=64, N = 2^9 .. 2^16 (seed 3)",
                           "l2": "flushed before every timed step", "steps_per_n": 10,
                           "peak": "torch.cuda.max_memory_allocated above the flush buffer: inputs, outputs, "
                                   "workspaces", "rows": length_sweep(la, dev, 10, 3)}
    if rank == 0 and not args.skip_cpu:
        result["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
    assert la.last_error() == 0
    if ws_n > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(result))


def _decode_graph_us(la, wd, B, T, dev, reps=5):
    """CUDA graph of T single-step launches of the recurrent step at batch B (heads H, D of
    the decode workload), replayed `reps` times: microseconds per step."""
    g_in = torch.Generator(device="cpu")
    g_in.manual_seed(wd.seed)
    q, k, v = (torch.randn(T, B, wd.H, d, generator=g_in).to(dev) for d in (wd.Dk, wd.Dk, wd.Dv))
    S = torch.zeros(B, wd.H, wd.Dk, wd.Dv, device=dev)
    z = torch.zeros(B, wd.H, wd.Dk, device=dev)
    outs = torch.empty(T, B, wd.H, wd.Dv, device=dev)
    s = torch.cuda.Stream(dev)
    s.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(s):
        for t in range(3):  # warm-up outside capture
            la.recurrent_step(q[t], k[t], v[t], S, z, out=outs[t])
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for t in range(T):
            la.recurrent_step(q[t], k[t], v[t], S, z, out=outs[t])
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / (reps * T)
    del q, k, v, S, z, outs, g
    return us


def bench_decode(la, dev, hbm):
    """Steps/s of the recurrent step (CUDA-graph replay of single-step launches): at the decode
    workload (B=64 H=8 D=32, whose 2 MiB state stays in L2 between steps), and at
    B=8000, where the state (262 MB) is larger than L2 and every step moves it through HBM."""
    out = {}
    wd0 = W.DECODE_CIFAR
    bytes_per_head = 2 * wd0.Dk * wd0.Dv * 4 + 2 * wd0.Dk * 4 + (2 * wd0.Dk + 2 * wd0.Dv) * 4
    for wd in (W.DECODE_CIFAR, W.DECODE_MNIST):
        us_step = _decode_graph_us(la, wd, wd.B, wd.steps, dev)
        bytes_step = wd.B * wd.H * bytes_per_head
        out["steps_%d" % wd.steps] = {
            "steps_per_s": 1e6 / us_step, "us_per_step": us_step, "tokens_per_s": wd.B * 1e6 / us_step,
            "bytes_per_step": bytes_step,
            "achieved_gbs": bytes_step / (us_step * 1e-6) / 1e9,
            "frac_of_hbm": bytes_step / (us_step * 1e-6) / 1e9 / hbm,
            "launch_floor_us": 0.51,
            "note": "S (2 MiB) stays in L2 across steps, so the step is bound by launch and L2 latency, not HBM; "
                    "launch_floor_us is a CUDA-graph replay of an empty kernel of the same grid with "
                    "programmatic dependent launch, measured on this GPU type; graph of %d single-step launches"
                    % wd.steps}
    B_big, T_big = 8000, 64  # B*H = 64000 heads (the library takes up to 65535)
    us_big = _decode_graph_us(la, wd0, B_big, T_big, dev)
    bytes_big = B_big * wd0.H * bytes_per_head
    out["large_batch"] = {
        "workload": "recurrent decode f32 B=%d H=%d Dk=Dv=%d, CUDA graph of %d single-step launches"
                    % (B_big, wd0.H, wd0.Dk, T_big),
        "us_per_step": us_big, "steps_per_s": 1e6 / us_big, "tokens_per_s": B_big * 1e6 / us_big,
        "bytes_per_step": bytes_big, "achieved_gbs": bytes_big / (us_big * 1e-6) / 1e9,
        "frac_of_hbm": bytes_big / (us_big * 1e-6) / 1e9 / hbm,
        "note": "S is 262 MB, larger than L2: each step reads and writes it from HBM"}
    return out


def bench_noncausal(la, dev):
    w = W.FWD_BF16
    q, k, v = (t.to(dev) for t in W.make_inputs(w))
    o = torch.empty_like(v)
    ws = torch.empty(la.workspace_bytes(la.OP_NONCAUSAL_FWD, w.B, w.H, w.N, w.Dk, w.Dv, w.dtype),
                     dtype=torch.uint8, device=dev)
    oc = torch.empty_like(v)
    wsc = torch.empty(la.workspace_bytes(la.OP_CAUSAL_FWD, w.B, w.H, w.N, w.Dk, w.Dv, w.dtype),
                      dtype=torch.uint8, device=dev)
    g = torch.Generator(device="cpu")
    g.manual_seed(12)
    dO = torch.randn(v.shape, generator=g).to(w.dtype).to(dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    wsb = torch.empty(la.workspace_bytes(la.OP_NONCAUSAL_BWD, w.B, w.H, w.N, w.Dk, w.Dv, w.dtype),
                      dtype=torch.uint8, device=dev)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    res = {}
    for name, fn in (("noncausal_fwd", lambda: la.noncausal_fwd(q, k, v, out=o, workspace=ws)),
                     ("noncausal_bwd", lambda: la.noncausal_bwd(q, k, v, dO, dq=dq, dk=dk, dv=dv, workspace=wsb)),
                     ("causal_fwd", lambda: la.causal_fwd(q, k, v, out=oc, workspace=wsc))):
        for _ in range(3):
            fn()
        times = []
        for _ in range(20):
            flush.zero_()  # evict L2 (inputs are only 16.8 MB)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            times.append(e0.elapsed_time(e1))
        ms = statistics.median(times)
        res[name] = {"ms": ms, "tokens_per_s": w.B * w.N / (ms / 1e3),
                     "workload": "%s bf16 B=%d H=%d N=%d Dk=Dv=%d" % (name.replace("_", " "), w.B, w.H, w.N, w.Dk),
                     "l2": "flushed"}
    del q, k, v, o, ws, oc, wsc, dO, dq, dk, dv, wsb, flush
    # the non-causal forward and backward at the long-context shape (inputs larger than L2)
    wl = W.LONG_BF16
    q, k, v, dO = (t.to(dev) for t in W.make_inputs(wl, with_grad=True))
    o = torch.empty_like(v)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(la.workspace_bytes(la.OP_NONCAUSAL_FWD, wl.B, wl.H, wl.N, wl.Dk, wl.Dv, wl.dtype),
                     dtype=torch.uint8, device=dev)
    wsb = torch.empty(la.workspace_bytes(la.OP_NONCAUSAL_BWD, wl.B, wl.H, wl.N, wl.Dk, wl.Dv, wl.dtype),
                      dtype=torch.uint8, device=dev)
    for name, fn in (("noncausal_fwd_long", lambda: la.noncausal_fwd(q, k, v, out=o, workspace=ws)),
                     ("noncausal_bwd_long",
                      lambda: la.noncausal_bwd(q, k, v, dO, dq=dq, dk=dk, dv=dv, workspace=wsb))):
        for _ in range(3):
            fn()
        times = []
        for _ in range(10):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            times.append(e0.elapsed_time(e1))
        ms = statistics.median(times)
        res[name] = {"ms": ms, "tokens_per_s": wl.B * wl.N / (ms / 1e3),
                     "workload": "noncausal " + name.split("_")[1] + " bf16 B=2 H=16 N=65536 Dk=Dv=128",
                     "l2": "inputs larger than L2"}
    return res


def bench_forward_forms(la, dev):
    """The causal forward as three launches (la_causal_fwd: segment sums, scan, outputs) and as
    one launch with a chained scan (la_causal_fwd_fused), median of 10 calls each, at the
    long-context shape (inputs larger than L2) and at shorter shapes (L2 flushed before each
    call)."""
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    shapes = [(W.LONG_BF16, None), (W.FWD_BF16, None), (W.sweep(512), None), (W.sweep(2048), None)]
    out = {}
    for w, _ in shapes:
        q, k, v = (t.to(dev) for t in W.make_inputs(w))
        o = torch.empty_like(v)
        ws = torch.empty(la.workspace_bytes(la.OP_CAUSAL_FWD, w.B, w.H, w.N, w.Dk, w.Dv, w.dtype),
                         dtype=torch.uint8, device=dev)
        row = {}
        for form, one in (("three_launches", False), ("one_launch", True)):
            for _ in range(3):
                la.causal_fwd(q, k, v, out=o, workspace=ws, one_launch=one)
            times = []
            for _ in range(10):
                if w.N < 65536:
                    flush.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                la.causal_fwd(q, k, v, out=o, workspace=ws, one_launch=one)
                e1.record()
                torch.cuda.synchronize()
                times.append(e0.elapsed_time(e1))
            row[form + "_ms"] = statistics.median(times)
        out["causal fwd bf16 B=%d H=%d N=%d Dk=Dv=%d" % (w.B, w.H, w.N, w.Dk)] = row
        del q, k, v, o, ws
    del flush
    return out


def bench_retention_step(la, dev):
    """Retention decode, S <- gamma S + k v^T and out = S^T q, at the decode shape: a CUDA
    graph of single-step launches replayed as for the causal decode step."""
    wd = W.DECODE_CIFAR
    T = wd.steps
    qd, kd, vd = (t.to(dev) for t in W.make_decode_inputs(wd))
    gd = W.retention_gammas(wd.H).to(dev)
    S = torch.zeros(wd.B, wd.H, wd.Dk, wd.Dv, device=dev)
    outs = torch.empty(T, wd.B, wd.H, wd.Dv, device=dev)
    s = torch.cuda.Stream(dev)
    s.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(s):
        for t in range(3):
            la.retention_step(qd[t], kd[t], vd[t], gd, S, out=outs[t])
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for t in range(T):
            la.retention_step(qd[t], kd[t], vd[t], gd, S, out=outs[t])
    g.replay()
    torch.cuda.synchronize()
    reps = 5
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    us_step = e0.elapsed_time(e1) * 1e3 / (reps * T)
    return {"us_per_step": us_step, "steps_per_s": 1e6 / us_step,
            "workload": "retention decode f32 B=%d H=%d Dk=Dv=%d, CUDA graph of %d single-step launches" %
            (wd.B, wd.H, wd.Dk, T)}


def bench_retention(la, dev):
    """Retention (constant decay per head) forward at the long-context shape."""
    w = W.RETENTION_BF16
    q, k, v = (t.to(dev) for t in W.make_inputs(w))  # 805 MB of inputs: larger than L2
    gam = W.retention_gammas(w.H).to(dev)
    o = torch.empty_like(v)
    ws = torch.empty(la.workspace_bytes(la.OP_RETENTION_FWD, w.B, w.H, w.N, w.Dk, w.Dv, w.dtype),
                     dtype=torch.uint8, device=dev)
    for _ in range(3):
        la.retention_fwd(q, k, v, gam, out=o, workspace=ws)
    times = []
    la.timing_reset()
    la.timing_enable(True)
    for _ in range(5):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        la.retention_fwd(q, k, v, gam, out=o, workspace=ws)
        e1.record()
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    la.timing_enable(False)
    kern = {n: ms / c for n, (c, ms) in la.timing_read().items()}
    ms = statistics.median(times)
    res = {"fwd": {"ms": ms, "tokens_per_s": w.B * w.N / (ms / 1e3), "workload": w.name,
                   "kernel_ms": kern, "l2": "inputs larger than L2"}}
    del q, k, v, o, ws
    return res


# ------------------------------------------------------------------ CPU baseline (the fp64 oracle)
def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def cpu_baseline(seconds_hint: float = 15.0):
    """The fp64 oracle (recurrent forward + reverse-recurrence backward) on a
    bounded sample of the long bf16 workload: `heads` whole heads, first
    `n_pos` positions each.  Throughput is scaled to the workload's unit:
    tokens/s = (heads * n_pos / H) / seconds."""
    import oracle
    cores = cpu_cores()
    os.environ.setdefault("OMP_NUM_THREADS", str(cores))
    w = W.LONG_BF16
    heads = cores
    # calibrate the sample size on a small probe so the run lasts about `seconds_hint`
    n_probe = 1024
    q, k, v, dO = W.make_inputs(w, with_grad=True, B=1, H=heads, N=n_probe)
    t0 = time.perf_counter()
    oracle.causal_recurrent(q, k, v)
    oracle.causal_bwd_recurrent(q, k, v, dO)
    dt = time.perf_counter() - t0
    n_pos = int(min(w.N, max(n_probe, n_probe * seconds_hint / max(dt, 1e-6))))
    if n_pos == w.N:  # whole heads already: take more of them (up to all B*H) to fill the time
        per_head = dt / n_probe * w.N
        heads = int(min(w.B * w.H, max(heads, cores * round(seconds_hint / max(per_head, 1e-6)))))
    q, k, v, dO = W.make_inputs(w, with_grad=True, B=1, H=heads, N=n_pos)
    t0 = time.perf_counter()
    oracle.causal_recurrent(q, k, v)
    oracle.causal_bwd_recurrent(q, k, v, dO)
    dt = time.perf_counter() - t0
    tps = heads * n_pos / w.H / dt
    return {"value": tps, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": "%d heads x %d positions of B=2 H=16 N=65536 D=128 (fp64 recurrent fwd + reverse-recurrence "
                      "bwd, OpenMP over heads), %.1f s" % (heads, n_pos, dt),
            "seconds": dt}


def run_reference(args):
    ws_n, rank, local = dist_env()
    if rank != 0:
        return
    step_seconds = max(1.0, args.cpu_seconds / max(1, args.steps))
    for _ in range(args.warmup):
        cpu_baseline(min(step_seconds, 2.0))
    vals = []
    t0 = time.perf_counter()
    for _ in range(args.steps):
        vals.append(cpu_baseline(step_seconds))
    total = time.perf_counter() - t0
    value = statistics.mean(v["value"] for v in vals)
    w = W.LONG_BF16
    res = {"impl": "reference", "metric": "causal lin-attn fwd+bwd tokens/s @N=64K; decode steps/s; % of roofline",
           "value": value, "unit": "tokens/s", "n_gpus": ws_n, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded, no dataset)",
           "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "Dk": w.Dk, "Dv": w.Dv},
           "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": vals[0]["cores"], "kind": "oracle",
                            "sample": vals[0]["sample"]},
           "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(res))


def length_sweep(la, dev, steps: int, warmup: int):
    """fwd+bwd time, tokens/s and peak device memory per N for the length sweep (bf16,
    B=1 H=8 D=64, N = 2^9 .. 2^16), L2 flushed before every timed step; a list of dicts."""
    rows = []
    hbm = peaks()[0]
    for N in W.SWEEP_NS:
        w = W.sweep(N)
        q, k, v, dO = W.make_inputs(w, with_grad=True)
        torch.cuda.empty_cache()
        torch.cuda.reset_peak_memory_stats()
        base = torch.cuda.memory_allocated()
        qd, kd, vd, dOd = (t.to(dev) for t in (q, k, v, dO))
        o = torch.empty_like(vd)
        dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
        wsf = torch.empty(la.workspace_bytes(la.OP_CAUSAL_FWD, w.B, w.H, N, w.Dk, w.Dv, w.dtype), dtype=torch.uint8,
                          device=dev)
        wsb = torch.empty(la.workspace_bytes(la.OP_CAUSAL_BWD, w.B, w.H, N, w.Dk, w.Dv, w.dtype), dtype=torch.uint8,
                          device=dev)
        flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)

        def step():
            la.causal_fwd(qd, kd, vd, out=o, workspace=wsf)
            la.causal_bwd(qd, kd, vd, dOd, dq=dq, dk=dk, dv=dv, workspace=wsb, fwd_workspace=wsf)

        for _ in range(warmup):
            step()
        times = []
        for _ in range(steps):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            step()
            e1.record()
            torch.cuda.synchronize()
            times.append(e0.elapsed_time(e1))
        ms = statistics.median(times)
        peak = torch.cuda.max_memory_allocated() - base - flush.numel()
        alg = w.B * w.H * N * ((2 * w.Dk + 2 * w.Dv) + (4 * w.Dk + 3 * w.Dv)) * 2
        rows.append({"N": N, "ms": ms, "tokens_per_s": w.B * N / (ms / 1e3), "peak_bytes": int(peak),
                     "workspace_bytes": int(wsf.numel() + wsb.numel()),
                     "io_bytes": int(8 * w.B * w.H * N * w.Dk * 2),
                     "frac_of_hbm": alg / (ms / 1e3) / 1e9 / hbm})
        del qd, kd, vd, dOd, o, dq, dk, dv, wsf, wsb, flush
    return rows


def run_sweep(args):
    """The length sweep alone, one JSON line per N."""
    import causal_linear_attention_phi_gb300 as la
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    la.build.build_library()
    for row in length_sweep(la, dev, args.steps, args.warmup):
        print(json.dumps(dict(sweep="causal fwd+bwd bf16 B=1 H=8 D=64", l2="flushed between steps", **row)))


def run_decode_profile(args):
    """Five eager decode steps at B=64 H=8 D=32 (state in L2) and five at B=8000 (state in
    HBM): a short, fixed launch sequence for ncu captures of the recurrent step."""
    import causal_linear_attention_phi_gb300 as la
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    la.build.build_library()
    wd = W.DECODE_CIFAR
    for B in (wd.B, 8000):
        q, k, v = (torch.randn(B, wd.H, d, device=dev) for d in (wd.Dk, wd.Dk, wd.Dv))
        S = torch.zeros(B, wd.H, wd.Dk, wd.Dv, device=dev)
        z = torch.zeros(B, wd.H, wd.Dk, device=dev)
        for _ in range(5):
            la.recurrent_step(q, k, v, S, z)
        torch.cuda.synchronize()
    assert la.last_error() == 0
    print(json.dumps({"decode_profile": "5 steps at B=64 and 5 at B=8000, H=8 Dk=Dv=32 fp32"}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--skip-cpu", action="store_true")
    ap.add_argument("--skip-e2e", action="store_true")
    ap.add_argument("--skip-extras", action="store_true")
    ap.add_argument("--sweep", action="store_true", help="length sweep N=2^9..2^16 (time, peak memory)")
    ap.add_argument("--decode-profile", action="store_true",
                    help="only 5 decode steps at B=64 and 5 at B=8000 (H=8 D=32), for ncu captures")
    ap.add_argument("--workload", choices=("long", "profile"), default="long",
                    help="long: B=2 H=16 N=65536 D=128 (the benchmark); profile: B=1 H=16 N=32768, plus two "
                         "one-launch causal forwards, two retention forwards, two non-causal forwards and two "
                         "non-causal backwards of that shape after the timed steps (ncu captures)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.gpus != world:
        # one process per GPU: N GPUs need N ranks, started by torch.distributed.run
        sys.exit("bench.py --gpus %d needs %d ranks (python -m torch.distributed.run --nproc-per-node %d "
                 "bench.py --gpus %d); this launch has WORLD_SIZE=%d" % (args.gpus, args.gpus, args.gpus,
                                                                         args.gpus, world))
    if args.decode_profile:
        run_decode_profile(args)
    elif args.sweep:
        run_sweep(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
