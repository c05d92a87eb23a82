"""Benchmark of the exact-attention hot path on one GB300 (or N, one process each).

A step is one pass of the whole path over one batch of synthetic input:
fa_fwd, then fa_bwd on the forward's O and LSE (the backward's three kernels:
D = rowsum(dO*O), the main pass, the dQ conversion).  The workload is
B=4, H=16, N=4096, d=128, bf16, non-causal, with inputs larger than L2
(Q, K, V, O, dO: 5 x 67 MB).

Printed (rank 0, one JSON line): whole-job TFLOPS (forward 4*B*H*N^2*d plus
backward 2.5x that, per step time), per-kernel times, the roofline of the
dominant kernel against the measured peaks, an end-to-end figure through the
Python API with pinned host buffers, SM clocks sampled during the timed
region, and the fp64 CPU oracle timed on a bounded sample (cpu_baseline).

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
WORKLOAD = fa_inputs.WORKLOADS["fwd_4k"]          # B4 H16 N4096 d128, non-causal
KERNEL_SOURCES = ["fa_fwd_kernel.cuh", "fa_bwd_kernel.cuh", "ptx.cuh", "exp2.cuh"]


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


def ncu_traffic(kernel: str):
    """DRAM bytes per launch from the committed ncu summary, if still current."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        t = json.load(f).get(kernel)
    if not t:
        return None
    for src, h in t.get("source_hashes", {}).items():
        if kernel_source_hash(src) != h:
            return None
    return t.get("bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
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
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


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
        return fa.fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(),
                         lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                         B, H, N, N, d, causal, w.scale, ws.data_ptr(), ws_bytes, sh)

    fwd()
    has_bwd = bwd() == fa.FA_OK
    torch.cuda.synchronize(dev)
    launches_per_step = 1 + (3 if has_bwd else 0)

    # warm-up
    for _ in range(args.warmup):
        fwd()
        if has_bwd:
            bwd()
    torch.cuda.synchronize(dev)

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    with ClockSampler(local) as clocks:
        if pg:
            pg.barrier()
        torch.cuda.synchronize(dev)
        t_wall = time.perf_counter()
        for i in range(args.steps):
            ev[i][0].record(stream)
            fwd()
            ev[i][1].record(stream)
            if has_bwd:
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
    t_bwd = [e[1].elapsed_time(e[2]) for e in ev] if has_bwd else [0.0] * args.steps
    ms_step = max_over_ranks(statistics.mean(a + b for a, b in zip(t_fwd, t_bwd)), pg, dev)

    flops_step = w.fwd_flops() + (w.bwd_flops() if has_bwd else 0.0)
    value = flops_step * world / (ms_step * 1e-3) / 1e12

    # ---- end to end through the Python API with pinned host buffers
    host_in = [torch.from_numpy(x.view(np.int16)).pin_memory() for x in (qb, kb, vb, dob)]
    host_out = [torch.empty(x.shape, dtype=torch.int16).pin_memory() for x in (qb, qb, kb, vb)]
    host_lse = torch.empty((B, H, N), dtype=torch.float32).pin_memory()
    h2d = sum(x.numel() * 2 for x in host_in)
    d2h = sum(x.numel() * 2 for x in host_out[: (4 if has_bwd else 1)]) + host_lse.numel() * 4

    def e2e_step():
        qq, kk, vv, dd = (h.to(dev, non_blocking=True).view(torch.bfloat16) for h in host_in)
        oo, ll = fa.forward(qq, kk, vv, causal=w.causal, scale=w.scale)
        outs = [oo]
        if has_bwd:
            outs += list(fa.backward(qq, kk, vv, oo, dd, ll, causal=w.causal, scale=w.scale,
                                     workspace=ws))
        for hbuf, t in zip(host_out, outs):
            hbuf.copy_(t.view(torch.int16), non_blocking=True)
        host_lse.copy_(ll, non_blocking=True)

    # (a) serial: every step uploads, computes and downloads on one stream
    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ms_e2e_serial = max_over_ranks(e0.elapsed_time(e1) / args.steps, pg, dev)

    # (b) pipelined, as a serving loop runs: uploads, compute and downloads on
    # three streams with two device buffer sets, so that step k+1's inputs
    # upload and step k-1's outputs download while step k computes.  Every
    # step's own copies are inside the timed region (first upload to last
    # download).
    s_up, s_down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    s_cmp = torch.cuda.current_stream(dev)
    n_out = 4 if has_bwd else 1
    dev_in = [[torch.empty(h.shape, dtype=torch.int16, device=dev) for h in host_in] for _ in range(2)]
    dev_out = [[torch.empty(h.shape, dtype=torch.int16, device=dev) for h in host_out[:n_out]] +
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
        oo, dq_, dk_, dv_ = (x.view(torch.bfloat16) for x in (dev_out[b][:4] if has_bwd else dev_out[b][:1] * 4))
        ll = dev_out[b][-1]
        fa.forward(qq, kk, vv, causal=w.causal, scale=w.scale, out=oo, lse=ll, stream=s_cmp)
        if has_bwd:
            st_ = fa.fa_bwd(qq.data_ptr(), kk.data_ptr(), vv.data_ptr(), oo.data_ptr(), dd.data_ptr(),
                            ll.data_ptr(), dq_.data_ptr(), dk_.data_ptr(), dv_.data_ptr(), B, H, N, N, d,
                            int(w.causal), w.scale, ws.data_ptr(), ws_bytes, s_cmp.cuda_stream)
            if st_ != fa.FA_OK:
                raise fa.FAError(st_, "fa_bwd")
        ev_cmp[b].record(s_cmp)
        with torch.cuda.stream(s_down):
            s_down.wait_event(ev_cmp[b])
            for h_, d_ in zip(host_out[:n_out], dev_out[b][:n_out]):
                h_.copy_(d_, non_blocking=True)
            host_lse.copy_(dev_out[b][-1], non_blocking=True)
            ev_out[b].record(s_down)

    for i in range(2):
        e2e_step_pipelined(i)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_up)
    for i in range(args.steps):
        e2e_step_pipelined(i)
    e1.record(s_down)
    torch.cuda.synchronize(dev)
    ms_e2e = max_over_ranks(e0.elapsed_time(e1) / args.steps, pg, dev)

    # ---- roofline of the dominant kernel
    peaks = measured_peaks()
    mean_fwd = statistics.mean(t_fwd)
    mean_bwd = statistics.mean(t_bwd) if has_bwd else 0.0
    if mean_bwd > mean_fwd:
        dom, dom_ms, dom_flops = "fa_bwd", mean_bwd, w.bwd_flops()
    else:
        dom, dom_ms, dom_flops = "fa_fwd", mean_fwd, w.fwd_flops()
    achieved = dom_flops / (dom_ms * 1e-3) / 1e12
    roofline = {"bound": "tensor", "kernel": dom, "achieved": achieved, "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "frac": achieved / peaks["bf16_tflops"],
                "peak_source": f"{peaks['source']} (burst bf16 GEMM)",
                "traffic": ncu_traffic(dom)}

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"B{B} H{H} N{N} d{d} non-causal, fwd+bwd" if has_bwd
                   else f"B{B} H{H} N{N} d{d} non-causal, fwd only (backward not built)",
                   "l2": "inputs larger than L2 (5 x 67 MB), no flush",
                   "parallelism": f"{world} independent replica(s), no collective"},
        "pct_of_peak": value / world / peaks["bf16_tflops"] * 100.0,
        "kernels_ms": {"fa_fwd": mean_fwd, "fa_bwd": mean_bwd if has_bwd else None},
        "fwd_tflops": w.fwd_flops() / (mean_fwd * 1e-3) / 1e12,
        "bwd_tflops": (w.bwd_flops() / (mean_bwd * 1e-3) / 1e12) if has_bwd else None,
        "roofline": roofline,
        "e2e": {"value": flops_step * world / (ms_e2e * 1e-3) / 1e12, "unit": "TFLOPS",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ms_e2e,
                "mode": "pipelined: copies of neighbouring steps overlap the compute (3 streams)",
                "serial": {"value": flops_step * world / (ms_e2e_serial * 1e-3) / 1e12,
                           "ms_per_step": ms_e2e_serial}},
        "gpu_launches": launches_per_step * args.steps,
        "wall_s_timed_region": wall,
        "clocks": clocks.summary(),
    }
    if has_bwd:
        line["bwd_deterministic_tflops"] = deterministic_bwd_tflops(torch, fa, w, q, k, v, o, do, lse,
                                                                    dq, dk, dv, ws, ws_bytes, stream)
    if w.d in (128, 256):
        line["fwd_fp8_tflops"] = fp8_fwd_tflops(torch, fa, w, q, k, v, stream)
    if args.sweep:
        line["sweep"] = sweep(torch, fa, dev, sh)
    if rank == 0 and not args.no_cpu_baseline:
        flops, secs, heads, threads = oracle_sample(WORKLOAD, args.cpu_budget, with_bwd=has_bwd)
        line["cpu_baseline"] = {"value": flops / secs / 1e12, "unit": "TFLOPS", "cores": threads,
                                "kind": "oracle",
                                "sample": f"{heads} whole heads (B=1,H=1,N={N},d={d}) fwd"
                                          f"{'+bwd' if has_bwd else ''}, fp64 numpy, {secs:.1f} s"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if pg:
        pg.destroy_process_group()
    return 0


def deterministic_bwd_tflops(torch, fa, w, q, k, v, o, do, lse, dq, dk, dv, ws, ws_bytes, stream, reps=20):
    """Backward TFLOPS of fa_bwd_ex in its fixed-order (bit-reproducible) mode."""
    sh = stream.cuda_stream

    def call():
        st = fa.fa_bwd_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(),
                          lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), w.B, w.H, w.N_q,
                          w.N_kv, w.d, int(w.causal), w.scale, 1, ws.data_ptr(), ws_bytes, sh)
        if st != fa.FA_OK:
            raise fa.FAError(st, "fa_bwd_ex")

    for _ in range(3):
        call()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        call()
    e1.record(stream)
    torch.cuda.synchronize()
    return w.bwd_flops() / (e0.elapsed_time(e1) / reps * 1e-3) / 1e12


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
        for _ in range(3):
            call()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            call()
        e1.record(stream)
        torch.cuda.synchronize()
        out[name] = w.fwd_flops() / (e0.elapsed_time(e1) / reps * 1e-3) / 1e12
    return out


def sweep(torch, fa, dev, sh, reps=10):
    """Forward TFLOPS over the 16k-token sequence sweep and the 4k / 8k configs."""
    out = []
    wls = fa_inputs.sweep_workloads(False) + fa_inputs.sweep_workloads(True)
    wls += [fa_inputs.WORKLOADS["stress_8k"]]
    wls += [fa_inputs.WORKLOADS["hdim64_8k"],
            fa_inputs.Workload("hdim64_8k_causal", 2, 16, 8192, 8192, 64, True, 0.125, 20266),
            fa_inputs.WORKLOADS["hdim256_8k"], fa_inputs.WORKLOADS["hdim256_8k_causal"]]
    for w in wls:
        qb, kb, vb = fa_inputs.make_qkv(w)
        q, k, v = (torch.from_numpy(x.view(np.int16)).to(dev).view(torch.bfloat16) for x in (qb, kb, vb))
        o = torch.empty_like(q)
        lse = torch.empty((w.B, w.H, w.N_q), dtype=torch.float32, device=dev)

        def call():
            st = fa.fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                           w.B, w.H, w.N_q, w.N_kv, w.d, int(w.causal), w.scale, sh)
            assert st == fa.FA_OK

        for _ in range(3):
            call()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            call()
        e1.record()
        torch.cuda.synchronize(dev)
        ms = e0.elapsed_time(e1) / reps
        out.append({"workload": w.name, "B": w.B, "N": w.N_q, "d": w.d, "causal": w.causal, "ms": ms,
                    "tflops": w.fwd_flops() / (ms * 1e-3) / 1e12})
        del q, k, v, o, lse
    out += sweep_fp8(torch, fa, dev, sh, reps)
    # the backward workload: B2 H16 N8192 d128 causal, both reduction orders
    w = fa_inputs.WORKLOADS["bwd_8k"]
    qb, kb, vb = fa_inputs.make_qkv(w)
    dob = fa_inputs.make_dout(w)
    q, k, v, do = (torch.from_numpy(x.view(np.int16)).to(dev).view(torch.bfloat16) for x in (qb, kb, vb, dob))
    o, lse = fa.forward(q, k, v, causal=True, scale=w.scale)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws_bytes = fa.fa_bwd_workspace_bytes(w.B, w.H, w.N_q, w.N_kv, w.d)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    for det in (0, 1):
        def call():
            st = fa.fa_bwd_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(),
                              lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), w.B, w.H, w.N_q,
                              w.N_kv, w.d, 1, w.scale, det, ws.data_ptr(), ws_bytes, sh)
            assert st == fa.FA_OK
        for _ in range(3):
            call()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            call()
        e1.record()
        torch.cuda.synchronize(dev)
        ms = e0.elapsed_time(e1) / reps
        out.append({"workload": "bwd_8k" + ("_deterministic" if det else ""), "B": w.B, "N": w.N_q, "d": w.d,
                    "causal": True, "ms": ms, "tflops": w.bwd_flops() / (ms * 1e-3) / 1e12})
    return out


FP8_SIGNS = (0x9E3779B9, 0x7F4A7C15, 0x2545F491, 0x4F6CDD1D, 0x85EBCA6B, 0xC2B2AE35, 0x27D4EB2F, 0x165667B1)


def sweep_fp8(torch, fa, dev, sh, reps=10):
    """The 8-bit forward (fa_fwd_fp8, quantisation included) on the 4k and 16k
    configs, with plain block quantisation and with incoherent processing.
    TFLOPS use the same 4 N^2 d count (halved when causal) as the bf16 lines."""
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
                assert st == fa.FA_OK
            for _ in range(3):
                call()
            torch.cuda.synchronize(dev)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(reps):
                call()
            e1.record()
            torch.cuda.synchronize(dev)
            ms = e0.elapsed_time(e1) / reps
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
        o, lse = fa.forward(q, k, v, causal=w.causal, scale=w.scale)
        if not args.fwd_only:
            fa.backward(q, k, v, o, do, lse, causal=w.causal, scale=w.scale, workspace=ws)
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
    ap.add_argument("--sweep", action="store_true", help="also time the forward sequence sweep")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle work")
    ap.add_argument("--ref-budget", type=float, default=4.0, help="oracle seconds per reference step")
    ap.add_argument("--profile", choices=sorted(fa_inputs.WORKLOADS), default=None,
                    help="only run fwd+bwd on this workload (for profiler captures)")
    ap.add_argument("--fwd-only", action="store_true", help="with --profile: forward only")
    ap.add_argument("--fp8", action="store_true", help="with --profile: the 8-bit forward only")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)      # at least 3 untimed warm-up steps, always
    if args.impl == "reference":
        return run_reference(args)
    if args.profile:
        return run_profile_case(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
