"""Benchmark of the exact-attention hot path on one GB300 (or N, one process each).

A step is one pass of the whole path over one batch of synthetic input:
fa_fwd, then fa_bwd on the forward's O and LSE (the backward's kernels:
D = rowsum(dO*O), the main pass, the dQ conversion).  The step's
workload is B=4, H=16,
N=4096, d=128, bf16, non-causal, with inputs larger than L2 (Q, K, V, O, dO:
5 x 67 MB).

Printed (rank 0, one JSON line): whole-job TFLOPS (forward 4*B*H*N^2*d plus
backward 2.5x that, per step time; the median over the timed steps), the
roofline of the dominant kernel (the backward's main kernel, its time per
launch isolated with CUPTI kernel records) against the measured peaks, an
end-to-end figure through the Python API with pinned host buffers, SM clocks
sampled during the timed region, every stated workload timed on its own
("configs": the tiny case, B4 H16 N4096 in both masks and both passes, the
16k-token sequence sweep, the rescaling stress case, the causal N8192
backward in both reduction orders, the d = 64 backward on single CTAs and on
CTA pairs) with the forward gate at N >= 8k, and the
fp64 CPU oracle timed on a bounded sample (cpu_baseline).

``--impl reference`` times the oracle instead (host cores, bounded sample per
step) and prints the same line shape with "impl": "reference".
Under torchrun (N > 1) every rank runs its own copy of the workload (weak
scaling over independent (batch, head) problems; no data-path collective).
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
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import fa_inputs  # noqa: E402

METRIC = "attention fwd/bwd TFLOPS (bf16, d=128) and % of GB300 dense BF16 peak"
LAUNCHES_PER_STEP = 4      # fa_fwd: one kernel; fa_bwd: prep, main, convert
WORKLOAD = fa_inputs.WORKLOADS["fwd_4k"]          # B4 H16 N4096 d128, non-causal


# ----------------------------------------------------------------- helpers

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def rank_workload(w: fa_inputs.Workload, rank: int) -> fa_inputs.Workload:
    """Each rank owns an independent copy of the workload (its own seed)."""
    return w.with_(seed=w.seed + 1000 * rank)


def max_over_ranks(value: float, pg, device) -> float:
    """The largest `value` over all ranks (a single process returns its own)."""
    if pg is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"bf16_tflops": p["bf16_tflops"], "bf16_tflops_sustained": p["bf16_tflops_sustained"],
                "hbm_gbs": p["hbm_gbs"], "source": "measured"}
    return {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0,
            "source": "fallback"}


def kernel_source_hash(name: str) -> str:
    path = os.path.join(ROOT, "exact_attention_74_gb300", "csrc", name)
    if not os.path.exists(path):
        return ""
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def ncu_traffic(name: str):
    """DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) from
    the committed ncu summary profiles/traffic.json, for a call ("fa_fwd",
    "fa_bwd") or one kernel (by name prefix), or None once the kernel sources
    the capture was taken with have changed."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        t = json.load(f)
    for call, entry in t.items():
        if not isinstance(entry, dict) or "source_hashes" not in entry:
            continue
        stale = any(kernel_source_hash(src) != h for src, h in entry["source_hashes"].items())
        if call == name:
            return None if stale else entry.get("bytes_per_launch")
        for kname, kv in entry.get("kernels", {}).items():
            if kname.startswith(name):
                return None if stale else kv["dram_read"] + kv["dram_write"]
    return None


def gpu_selector(local: int) -> str:
    """The nvidia-smi -i argument for torch device `local`: its UUID.

    torch numbers only the devices CUDA_VISIBLE_DEVICES leaves visible, while
    nvidia-smi numbers every GPU of the machine, so the index alone can name
    another GPU; the UUID names this one.  Falls back to mapping the index
    through CUDA_VISIBLE_DEVICES."""
    try:
        import torch
        u = str(torch.cuda.get_device_properties(local).uuid)
        if u:
            return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        pass
    vis = [x.strip() for x in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if x.strip()]
    return vis[local] if local < len(vis) else str(local)


class ClockSampler:
    """nvidia-smi clocks and throttle reasons of one GPU, sampled every 200 ms."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, selector: str):
        self.selector = selector
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.selector, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "gpu": self.selector}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm), "gpu": self.selector}


# ------------------------------------------------------------ CPU oracle leg

def oracle_sample(w: fa_inputs.Workload, budget_s: float, with_bwd: bool):
    """Time the fp64 oracle on whole heads of the workload until budget_s passes.

    Returns (flops done, seconds, heads, threads).
    """
    import oracle
    threads = len(os.sched_getaffinity(0))
    one = w.with_(B=1, H=1)
    flops_head = one.fwd_flops() + (one.bwd_flops() if with_bwd else 0.0)
    done, heads, secs = 0.0, 0, 0.0
    while heads == 0 or secs < budget_s:
        h = one.with_(seed=w.seed + 17 * heads)
        qb, kb, vb = fa_inputs.make_qkv(h)
        q, k, v = (fa_inputs.bf16_bits_to_f64(x)[0, 0] for x in (qb, kb, vb))
        do = fa_inputs.bf16_bits_to_f64(fa_inputs.make_dout(h))[0, 0] if with_bwd else None
        t1 = time.perf_counter()          # input generation stays outside the timing
        oracle.head_forward(q, k, v, causal=w.causal, scale=w.scale)
        if with_bwd:
            oracle.head_backward(q, k, v, do, causal=w.causal, scale=w.scale)
        secs += time.perf_counter() - t1
        done += flops_head
        heads += 1
    return done, secs, heads, threads


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    w = WORKLOAD
    steps_t = []
    for i in range(args.warmup + args.steps):
        flops, secs, heads, threads = oracle_sample(w, args.ref_budget, with_bwd=True)
        if i >= args.warmup:
            steps_t.append((flops, secs, heads))
    flops = sum(f for f, _, _ in steps_t)
    secs = sum(s for _, s, _ in steps_t)
    value = flops / secs / 1e12
    heads = steps_t[0][2]
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOPS",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": secs / len(steps_t) * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"B{w.B} H{w.H} N{w.N_q} d{w.d} non-causal, fwd+bwd",
                   "sample_per_step": f"{heads} whole heads (B=1,H=1,N={w.N_q},d={w.d})"},
        "cpu_baseline": {"value": value, "unit": "TFLOPS", "cores": threads, "kind": "oracle",
                         "sample": f"{heads} whole heads of the workload per step, fwd+bwd, fp64 numpy"},
        "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ GPU leg

def event_times(torch, stream, fn, reps, warmup=3):
    """Per-call device times (ms) of fn, CUDA events recorded on `stream`
    around each call, after `warmup` untimed calls."""
    for _ in range(warmup):
        fn()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    torch.cuda.synchronize()
    for a, b in evs:
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


_KERNELS = ("fwd_kernel", "fwd64_kernel", "fwd256p_kernel", "prep_kernel", "main_kernel", "main64_kernel",
            "pair_kernel", "convert_kernel", "fwd8_kernel", "fwd8_256_kernel", "quant_qk_kernel", "quant_v_kernel")


def _short_kernel_name(name: str) -> str:
    return name.split("(")[0].replace("void ", "").replace("fa::", "").strip()


def cupti_kernel_split(torch, fn, reps=10):
    """Per-launch device time of each of this library's kernels over `reps`
    calls of fn, from CUPTI kernel records (torch.profiler): (split, note),
    split None when the profiler recorded none of them (note says why).
    Run outside the timed region."""
    try:
        from torch.profiler import ProfilerActivity, profile
        fn()
        torch.cuda.synchronize()
        with profile(activities=[ProfilerActivity.CPU, ProfilerActivity.CUDA]) as prof:
            for _ in range(reps):
                fn()
            torch.cuda.synchronize()
        acc = {}

        def add(name, dur_us):
            if any(k in name for k in _KERNELS):
                n, t = acc.get(_short_kernel_name(name), (0, 0.0))
                acc[_short_kernel_name(name)] = (n + 1, t + dur_us)

        events = list(prof.events())
        for e in events:        # device-side kernel events
            if "cuda" in str(getattr(e, "device_type", "")).lower():
                add(e.name, getattr(e, "device_time", 0.0) or getattr(e, "cuda_time", 0.0))
        if not acc:             # else the kernels attached to host-side launch events
            for e in events:
                for kern in getattr(e, "kernels", []) or []:
                    add(kern.name, kern.duration)
        if not acc:
            return None, (f"no kernel records of this library; {len(events)} profiler events: "
                          f"{sorted({e.name for e in events})[:8]}")
        out = {k: {"launches_per_call": n / reps, "ms_per_launch": t / n / 1e3} for k, (n, t) in acc.items()}
        return out, "CUPTI kernel records (torch.profiler)"
    except Exception as ex:   # the profiler is optional here
        return None, f"torch.profiler unavailable: {type(ex).__name__}: {ex}"


def launch_list_share(kernel_prefix: str):
    """Fallback split: the kernel's share of the backward call in the committed
    launch list of the bench step (cold-cache ncu times), or None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        t = json.load(f).get("fa_bwd", {})
    times = t.get("kernel_us", {})
    tot = sum(times.values())
    for k, v in times.items():
        if k.startswith(kernel_prefix) and tot > 0:
            return v / tot
    return None


def run_gpu(args):
    import torch
    import exact_attention_74_gb300 as fa

    rank, world, local = dist_env()
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
        pg = dist
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = rank_workload(WORKLOAD, rank)
    B, H, N, d = w.B, w.H, w.N_q, w.d
    qb, kb, vb = fa_inputs.make_qkv(w)
    dob = fa_inputs.make_dout(w)

    def to_dev(bits):
        return torch.from_numpy(bits.view(np.int16)).to(dev).view(torch.bfloat16)

    q, k, v, do = (to_dev(x) for x in (qb, kb, vb, dob))
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws_bytes = fa.fa_bwd_workspace_bytes(B, H, N, N, d)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    causal = int(w.causal)

    def fwd():
        st = fa.fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                       B, H, N, N, d, causal, w.scale, sh)
        if st != fa.FA_OK:
            raise fa.FAError(st, "fa_fwd")

    def bwd():
        st = fa.fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(),
                       lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                       B, H, N, N, d, causal, w.scale, ws.data_ptr(), ws_bytes, sh)
        if st != fa.FA_OK:
            raise fa.FAError(st, "fa_bwd")

    def step():
        fwd()
        bwd()

    step()
    torch.cuda.synchronize(dev)
    # this library's kernels per step and their per-launch times (CUPTI records,
    # outside the timed region)
    split, split_note = cupti_kernel_split(torch, step)
    launches_per_step = round(sum(x["launches_per_call"] for x in split.values())) if split else None

    # warm-up
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    clocks = ClockSampler(gpu_selector(local))
    clocks.__enter__()
    try:
        if pg:
            pg.barrier()
        torch.cuda.synchronize(dev)
        t_wall = time.perf_counter()
        for i in range(args.steps):
            ev[i][0].record(stream)
            fwd()
            ev[i][1].record(stream)
            bwd()
            ev[i][2].record(stream)
        torch.cuda.synchronize(dev)
        wall = time.perf_counter() - t_wall
        if pg:
            pg.barrier()
        st = fa.fa_get_last_device_status(sh)
        if st != fa.FA_OK:
            raise fa.FAError(st, "device status after timed region")
        t_fwd = [e[0].elapsed_time(e[1]) for e in ev]
        t_bwd = [e[1].elapsed_time(e[2]) for e in ev]
        ms_step = max_over_ranks(statistics.median(a + b for a, b in zip(t_fwd, t_bwd)), pg, dev)

        flops_step = w.fwd_flops() + w.bwd_flops()
        value = flops_step * world / (ms_step * 1e-3) / 1e12

        e2e = end_to_end(torch, fa, w, dev, stream, ws, ws_bytes, qb, kb, vb, dob, args.steps, pg)

        peaks = measured_peaks()
        peak = peaks["bf16_tflops"]
        med_fwd, med_bwd = statistics.median(t_fwd), statistics.median(t_bwd)

        # ---- roofline of the dominant kernel: the backward's main kernel
        main_name = next((n for n in (split or {}) if "main_kernel" in n), None)
        if main_name is not None:
            main_ms = split[main_name]["ms_per_launch"]
            time_source = "CUPTI kernel records (torch.profiler), 10 steps outside the timed region"
        else:
            share = launch_list_share("main_kernel")
            main_ms = med_bwd * share if share else med_bwd
            main_name = "bwd::main_kernel<128, false>"
            time_source = ("the backward call's event time x the kernel's share of the committed ncu "
                           "launch list" if share else "the backward call's event time (no split available)")
        achieved = w.bwd_flops() / (main_ms * 1e-3) / 1e12
        roofline = {"bound": "tensor", "kernel": main_name, "achieved": achieved, "peak": peak,
                    "unit": "TFLOP/s", "frac": achieved / peak, "traffic": ncu_traffic("main_kernel"),
                    "ms_per_launch": main_ms, "time_source": time_source,
                    "peak_source": f"{peaks['source']} (burst bf16 GEMM)",
                    "frac_of_sustained": achieved / peaks["bf16_tflops_sustained"],
                    "call": {"what": "fa_bwd (prep + main + convert), CUDA events in the timed region",
                             "achieved": w.bwd_flops() / (med_bwd * 1e-3) / 1e12,
                             "frac": w.bwd_flops() / (med_bwd * 1e-3) / 1e12 / peak,
                             "traffic": ncu_traffic("fa_bwd")}}

        line = {
            "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": f"B{B} H{H} N{N} d{d} non-causal, fwd+bwd",
                       "l2": "inputs larger than L2 (5 x 67 MB), no flush",
                       "parallelism": f"{world} independent replica(s), no collective",
                       "ms_per_step": "median of the per-step CUDA-event times"},
            "pct_of_peak": value / world / peak * 100.0,
            "kernels_ms": {"fa_fwd": med_fwd, "fa_bwd": med_bwd},
            "kernel_split": split, "kernel_split_source": split_note,
            "fwd_tflops": w.fwd_flops() / (med_fwd * 1e-3) / 1e12,
            "bwd_tflops": w.bwd_flops() / (med_bwd * 1e-3) / 1e12,
            "roofline": roofline,
            "e2e": e2e,
            "gpu_launches": (launches_per_step or LAUNCHES_PER_STEP) * args.steps,
            "wall_s_timed_region": wall,
        }
        line["bwd_deterministic_tflops"] = deterministic_bwd_tflops(torch, fa, w, q, k, v, o, do, lse,
                                                                    dq, dk, dv, ws, ws_bytes, stream)
        line["fwd_fp8_tflops"] = fp8_fwd_tflops(torch, fa, w, q, k, v, stream)
        del q, k, v, do, o, lse, dq, dk, dv, ws
        if not args.no_configs:
            configs = time_configs(torch, fa, dev, stream, peak)
            line["configs"] = configs
            line["gate"] = forward_gate(configs)
        if args.extras:
            line["extras"] = sweep_fp8(torch, fa, dev, stream)
    finally:
        clocks.__exit__(None, None, None)
    line["clocks"] = clocks.summary()
    line["clocks"]["window"] = "the timed steps and every timing after them (end to end, configs)"
    if rank == 0 and not args.no_cpu_baseline:
        flops, secs, heads, threads = oracle_sample(WORKLOAD, args.cpu_budget, with_bwd=True)
        line["cpu_baseline"] = {"value": flops / secs / 1e12, "unit": "TFLOPS", "cores": threads,
                                "kind": "oracle",
                                "sample": f"{heads} whole heads (B=1,H=1,N={N},d={d}) fwd+bwd, fp64 numpy, "
                                          f"{secs:.1f} s"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if pg:
        pg.destroy_process_group()
    return 0


def end_to_end(torch, fa, w, dev, stream, ws, ws_bytes, qb, kb, vb, dob, steps, pg):
    """The step through the Python API with pinned host buffers: every step's
    host-to-device copy of Q, K, V, dO and device-to-host copy of O, dQ, dK,
    dV, LSE inside the timed region."""
    B, H, N, d = w.B, w.H, w.N_q, w.d
    host_in = [torch.from_numpy(x.view(np.int16)).pin_memory() for x in (qb, kb, vb, dob)]
    host_out = [torch.empty(x.shape, dtype=torch.int16).pin_memory() for x in (qb, qb, kb, vb)]
    host_lse = torch.empty((B, H, N), dtype=torch.float32).pin_memory()
    h2d = sum(x.numel() * 2 for x in host_in)
    d2h = sum(x.numel() * 2 for x in host_out) + host_lse.numel() * 4

    def e2e_step():
        qq, kk, vv, dd = (h.to(dev, non_blocking=True).view(torch.bfloat16) for h in host_in)
        oo, ll = fa.forward(qq, kk, vv, causal=w.causal, scale=w.scale)
        outs = [oo] + list(fa.backward(qq, kk, vv, oo, dd, ll, causal=w.causal, scale=w.scale, workspace=ws))
        for hbuf, t in zip(host_out, outs):
            hbuf.copy_(t.view(torch.int16), non_blocking=True)
        host_lse.copy_(ll, non_blocking=True)

    # (a) serial: every step uploads, computes and downloads on one stream
    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ms_serial = max_over_ranks(e0.elapsed_time(e1) / steps, pg, dev)

    # (b) pipelined, as a serving loop runs: uploads, compute and downloads on
    # three streams with two device buffer sets, so that step k+1's inputs
    # upload and step k-1's outputs download while step k computes.  Every
    # step's own copies are inside the timed region (first upload to last
    # download).
    s_up, s_down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    s_cmp = stream
    dev_in = [[torch.empty(h.shape, dtype=torch.int16, device=dev) for h in host_in] for _ in range(2)]
    dev_out = [[torch.empty(h.shape, dtype=torch.int16, device=dev) for h in host_out] +
               [torch.empty((B, H, N), dtype=torch.float32, device=dev)] for _ in range(2)]
    ev_in, ev_cmp, ev_out = ([torch.cuda.Event() for _ in range(2)] for _ in range(3))

    def e2e_step_pipelined(i):
        b = i & 1
        with torch.cuda.stream(s_up):
            if i >= 2:
                s_up.wait_event(ev_cmp[b])             # step i-2 has read this input set
            for d_, h_ in zip(dev_in[b], host_in):
                d_.copy_(h_, non_blocking=True)
            ev_in[b].record(s_up)
        s_cmp.wait_event(ev_in[b])
        if i >= 2:
            s_cmp.wait_event(ev_out[b])                # step i-2's outputs have left this set
        qq, kk, vv, dd = (x.view(torch.bfloat16) for x in dev_in[b])
        oo, dq_, dk_, dv_ = (x.view(torch.bfloat16) for x in dev_out[b][:4])
        ll = dev_out[b][-1]
        fa.forward(qq, kk, vv, causal=w.causal, scale=w.scale, out=oo, lse=ll, stream=s_cmp)
        st_ = fa.fa_bwd(qq.data_ptr(), kk.data_ptr(), vv.data_ptr(), oo.data_ptr(), dd.data_ptr(),
                        ll.data_ptr(), dq_.data_ptr(), dk_.data_ptr(), dv_.data_ptr(), B, H, N, N, d,
                        int(w.causal), w.scale, ws.data_ptr(), ws_bytes, s_cmp.cuda_stream)
        if st_ != fa.FA_OK:
            raise fa.FAError(st_, "fa_bwd")
        ev_cmp[b].record(s_cmp)
        with torch.cuda.stream(s_down):
            s_down.wait_event(ev_cmp[b])
            for h_, d_ in zip(host_out, dev_out[b][:4]):
                h_.copy_(d_, non_blocking=True)
            host_lse.copy_(dev_out[b][-1], non_blocking=True)
            ev_out[b].record(s_down)

    for i in range(2):
        e2e_step_pipelined(i)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_up)
    for i in range(steps):
        e2e_step_pipelined(i)
    e1.record(s_down)
    torch.cuda.synchronize(dev)
    ms_e2e = max_over_ranks(e0.elapsed_time(e1) / steps, pg, dev)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    flops_step = w.fwd_flops() + w.bwd_flops()
    return {"value": flops_step * world / (ms_e2e * 1e-3) / 1e12, "unit": "TFLOPS",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ms_e2e,
            "mode": "pipelined: copies of neighbouring steps overlap the compute (3 streams)",
            "serial": {"value": flops_step * world / (ms_serial * 1e-3) / 1e12, "ms_per_step": ms_serial}}


def deterministic_bwd_tflops(torch, fa, w, q, k, v, o, do, lse, dq, dk, dv, ws, ws_bytes, stream, reps=20):
    """Backward TFLOPS of fa_bwd_ex in its fixed-order (bit-reproducible) mode."""
    sh = stream.cuda_stream

    def call():
        st = fa.fa_bwd_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(),
                          lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), w.B, w.H, w.N_q,
                          w.N_kv, w.d, int(w.causal), w.scale, 1, ws.data_ptr(), ws_bytes, sh)
        if st != fa.FA_OK:
            raise fa.FAError(st, "fa_bwd_ex")

    ms = statistics.median(event_times(torch, stream, call, reps))
    return w.bwd_flops() / (ms * 1e-3) / 1e12


FP8_SIGNS = (0x9E3779B9, 0x7F4A7C15, 0x2545F491, 0x4F6CDD1D, 0x85EBCA6B, 0xC2B2AE35, 0x27D4EB2F, 0x165667B1)


def fp8_fwd_tflops(torch, fa, w, q, k, v, stream, reps=20):
    """The same forward through fa_fwd_fp8 (e4m3 operands, quantisation
    included in the timed call): plain block quantisation and with
    incoherent processing.  Same flop count as the bf16 forward."""
    sh = stream.cuda_stream
    o8 = torch.empty_like(q)
    lse8 = torch.empty((w.B, w.H, w.N_q), dtype=torch.float32, device=q.device)
    ws_bytes = fa.fa_fwd_fp8_workspace_bytes(w.B, w.H, w.N_q, w.N_kv, w.d)
    ws8 = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
    out = {}
    for name, signs in (("plain", None), ("incoherent", FP8_SIGNS[:w.d // 32])):
        def call():
            st = fa.fa_fwd_fp8(q.data_ptr(), k.data_ptr(), v.data_ptr(), o8.data_ptr(), lse8.data_ptr(), w.B, w.H,
                               w.N_q, w.N_kv, w.d, int(w.causal), w.scale, signs, ws8.data_ptr(), ws_bytes, sh)
            if st != fa.FA_OK:
                raise fa.FAError(st, "fa_fwd_fp8")
        ms = statistics.median(event_times(torch, stream, call, reps))
        out[name] = w.fwd_flops() / (ms * 1e-3) / 1e12
    return out


def _config_workloads():
    """(label, workload, passes) for every stated workload, then the extra
    head dimensions.  Passes: "fwd", "bwd" (unordered dQ), "bwd_det" (fixed
    order), "bwd_pair" (fa_bwd_pair: pairs of CTAs sharing products, d = 64)."""
    W = fa_inputs.WORKLOADS
    out = [("1 tiny", W["tiny"], ("fwd",)), ("1 tiny", W["tiny_causal"], ("fwd",)),
           ("2", W["fwd_4k"], ("fwd", "bwd", "bwd_det")), ("2", W["fwd_4k_causal"], ("fwd", "bwd"))]
    out += [("3 sweep", x, ("fwd",)) for x in fa_inputs.sweep_workloads(False) + fa_inputs.sweep_workloads(True)]
    out += [("4 stress", W["stress_8k"], ("fwd",)), ("5 backward", W["bwd_8k"], ("fwd", "bwd", "bwd_det"))]
    out += [("extra d=64", W["hdim64_8k"], ("fwd", "bwd", "bwd_pair")),
            ("extra d=64", W["hdim64_8k"].with_(name="hdim64_8k_causal", causal=True), ("fwd", "bwd", "bwd_pair")),
            ("extra d=256", W["hdim256_8k"], ("fwd",)), ("extra d=256", W["hdim256_8k_causal"], ("fwd",))]
    return out


def time_configs(torch, fa, dev, stream, peak, reps=10):
    """Median CUDA-event time per call of every stated workload (and the extra
    head dimensions), each at its full size, with TFLOPS and the fraction of
    the measured bf16 peak.  Inputs are the seeded recipes of fa_inputs."""
    sh = stream.cuda_stream
    out = []
    cache = {}
    for label, w, passes in _config_workloads():
        key = (w.B, w.H, w.N_q, w.N_kv, w.d, w.seed, w.kind)
        if key not in cache:
            cache.clear()
            qb, kb, vb = fa_inputs.make_qkv(w)
            cache[key] = [torch.from_numpy(x.view(np.int16)).to(dev).view(torch.bfloat16) for x in (qb, kb, vb)]
        q, k, v = cache[key]
        o = torch.empty_like(q)
        lse = torch.empty((w.B, w.H, w.N_q), dtype=torch.float32, device=dev)

        def fwd():
            st = fa.fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                           w.B, w.H, w.N_q, w.N_kv, w.d, int(w.causal), w.scale, sh)
            if st != fa.FA_OK:
                raise fa.FAError(st, f"fa_fwd {w.name}")

        fwd()
        rec = {"config": label, "workload": w.name, "B": w.B, "H": w.H, "N": w.N_q, "d": w.d,
               "causal": w.causal, "kind": w.kind}
        if "fwd" in passes:
            ms = statistics.median(event_times(torch, stream, fwd, reps))
            tf = w.fwd_flops() / (ms * 1e-3) / 1e12
            out.append({**rec, "pass": "fwd", "ms": ms, "tflops": tf, "frac": tf / peak})
        bwd_passes = [p for p in passes if p.startswith("bwd")]
        if bwd_passes:
            do = torch.from_numpy(fa_inputs.make_dout(w).view(np.int16)).to(dev).view(torch.bfloat16)
            dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
            wsb = fa.fa_bwd_workspace_bytes(w.B, w.H, w.N_q, w.N_kv, w.d)
            ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
            for p in bwd_passes:
                det = 1 if p == "bwd_det" else 0
                args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(), lse.data_ptr(),
                        dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), w.B, w.H, w.N_q, w.N_kv, w.d, int(w.causal),
                        w.scale)

                def bwd():
                    if p == "bwd_pair":
                        st = fa.fa_bwd_pair(*args, ws.data_ptr(), wsb, sh)
                    else:
                        st = fa.fa_bwd_ex(*args, det, ws.data_ptr(), wsb, sh)
                    if st != fa.FA_OK:
                        raise fa.FAError(st, f"{p} {w.name}")

                ms = statistics.median(event_times(torch, stream, bwd, reps))
                tf = w.bwd_flops() / (ms * 1e-3) / 1e12
                name = {"bwd": "bwd", "bwd_det": "bwd fixed order", "bwd_pair": "bwd cta pair"}[p]
                out.append({**rec, "pass": name, "ms": ms, "tflops": tf, "frac": tf / peak})
            del do, dq, dk, dv, ws
        del o, lse
    torch.cuda.synchronize(dev)
    st = fa.fa_get_last_device_status(sh)
    if st != fa.FA_OK:
        raise fa.FAError(st, "device status after the configs")
    cache.clear()
    return out


def forward_gate(configs):
    """The forward gate: every d = 128 bf16 forward at N >= 8k (the sequence
    sweep's 8k, 16k and 32k in both masks, and the stress workload) at >= 60%
    of the measured peak."""
    rows = [c for c in configs if c["pass"] == "fwd" and c["d"] == 128 and c["N"] >= 8192
            and c["config"] in ("3 sweep", "4 stress")]
    if not rows:
        return None
    worst = min(rows, key=lambda c: c["frac"])
    return {"criterion": "d=128 bf16 forward at N >= 8k, >= 0.60 of the measured burst bf16 peak",
            "workloads": [c["workload"] for c in rows], "min_frac": worst["frac"],
            "min_workload": worst["workload"], "max_frac": max(c["frac"] for c in rows),
            "pass": worst["frac"] >= 0.60}


def sweep_fp8(torch, fa, dev, stream, reps=10):
    """The 8-bit forward (fa_fwd_fp8, quantisation included) on the 4k and 16k
    configs and at d = 256, with plain block quantisation and with incoherent
    processing.  TFLOPS use the same 4 N^2 d count (halved when causal) as the
    bf16 lines."""
    sh = stream.cuda_stream
    out = []
    wls = [fa_inputs.WORKLOADS["fwd_4k"], fa_inputs.WORKLOADS["fwd_4k_causal"]]
    wls += [w for w in fa_inputs.sweep_workloads(False) + fa_inputs.sweep_workloads(True) if w.N_q == 16384]
    wls += [fa_inputs.WORKLOADS["hdim256_8k"], fa_inputs.WORKLOADS["hdim256_8k_causal"]]
    for w in wls:
        qb, kb, vb = fa_inputs.make_qkv(w)
        q, k, v = (torch.from_numpy(x.view(np.int16)).to(dev).view(torch.bfloat16) for x in (qb, kb, vb))
        o = torch.empty_like(q)
        lse = torch.empty((w.B, w.H, w.N_q), dtype=torch.float32, device=dev)
        ws_bytes = fa.fa_fwd_fp8_workspace_bytes(w.B, w.H, w.N_q, w.N_kv, w.d)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
        for signs in (None, FP8_SIGNS[:w.d // 32]):
            def call():
                st = fa.fa_fwd_fp8(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                   w.B, w.H, w.N_q, w.N_kv, w.d, int(w.causal), w.scale, signs,
                                   ws.data_ptr(), ws_bytes, sh)
                if st != fa.FA_OK:
                    raise fa.FAError(st, "fa_fwd_fp8")
            ms = statistics.median(event_times(torch, stream, call, reps))
            out.append({"workload": "fp8_" + w.name + ("_hadamard" if signs else ""), "B": w.B, "N": w.N_q,
                        "d": w.d, "causal": w.causal, "dtype": "e4m3", "ms": ms,
                        "tflops": w.fwd_flops() / (ms * 1e-3) / 1e12})
        del q, k, v, o, lse, ws
    return out


def run_profile_case(args):
    """fwd + bwd on one named workload, W + K times, for ncu captures (prints ms only)."""
    import torch
    import exact_attention_74_gb300 as fa
    w = fa_inputs.WORKLOADS[args.profile]
    qb, kb, vb = fa_inputs.make_qkv(w)
    dob = fa_inputs.make_dout(w)
    q, k, v, do = (torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16) for x in (qb, kb, vb, dob))
    ws = torch.empty(fa.fa_bwd_workspace_bytes(w.B, w.H, w.N_q, w.N_kv, w.d), dtype=torch.uint8, device="cuda")
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for i in range(args.warmup + args.steps):
        if i == args.warmup:
            e0.record()
        if args.fp8:
            fa.forward_fp8(q, k, v, causal=w.causal, scale=w.scale, signs=FP8_SIGNS[:w.d // 32])
            continue
        o, lse = fa.forward(q, k, v, causal=w.causal, scale=w.scale,
                            emu_per_32=None if args.emu is None else args.emu)
        if not args.fwd_only:
            fa.backward(q, k, v, o, do, lse, causal=w.causal, scale=w.scale, workspace=ws,
                        deterministic=args.deterministic, pair=args.pair)
    e1.record()
    torch.cuda.synchronize()
    st = fa.fa_get_last_device_status(torch.cuda.current_stream().cuda_stream)
    if st != fa.FA_OK:
        raise fa.FAError(st, "device status")
    print(json.dumps({"profile_case": w.name, "ms_per_step": e0.elapsed_time(e1) / max(1, args.steps)}))
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-configs", action="store_true", help="skip the per-workload timings")
    ap.add_argument("--extras", action="store_true", help="also time the 8-bit forward on more workloads")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle work")
    ap.add_argument("--ref-budget", type=float, default=4.0, help="oracle seconds per reference step")
    ap.add_argument("--profile", choices=sorted(fa_inputs.WORKLOADS), default=None,
                    help="only run fwd+bwd on this workload (for profiler captures)")
    ap.add_argument("--fwd-only", action="store_true", help="with --profile: forward only")
    ap.add_argument("--fp8", action="store_true", help="with --profile: the 8-bit forward only")
    ap.add_argument("--deterministic", action="store_true", help="with --profile: the fixed-order backward")
    ap.add_argument("--pair", action="store_true", help="with --profile: the backward on CTA pairs (d = 64)")
    ap.add_argument("--emu", type=int, choices=(0, 8, 16), default=None,
                    help="with --profile: exponentials per 32 on the FMA-pipe emulation (default: the library's)")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)      # at least 3 untimed warm-up steps, always
    if args.impl == "reference":
        return run_reference(args)
    if args.profile:
        return run_profile_case(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
