"""Benchmark of the KDA forward (and single-token decode) on one GB300.

One step = one ``kda_fwd`` call (plan, fused prologue + intra-chunk kernel,
inter-chunk scan) over the dense workload B=2, T=16384, H_qk=H_v=32,
K=V=128 with an fp32 initial state and final-state output.  The timed region
holds exactly ``--steps`` calls bracketed by a barrier and device
synchronisation; inputs (1.4 GB per step) are larger than L2, so no flush is
needed between steps.  Prints one JSON line (rank 0).

``--impl reference`` times the fp64 CPU oracle instead, on a bounded sample of
the same workload per step (the pages publish no runnable implementation).
"""
from __future__ import annotations

import argparse
import csv
import io
import json
import math
import os
import statistics
import subprocess
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import kda_inputs as KI  # noqa: E402

METRIC = "KDA fwd tokens*heads/s & % bf16 TC peak (T=16K); decode state GB/s % HBM"
UNIT = "token*heads/s"
WORKLOAD = "KDA fwd dense B=2 T=16384 H_qk=H_v=32 K=V=128, fp32 initial/final state"
# Algorithmic work of the forward (per token and value head, K = V = 128, chunk 64):
#   bytes: q, k, v, graw (4 x 256 B) + b (2 B) + out (256 B); plus 2 x 64 KiB of state per (sequence, head)
#   flops: 2 [3 K V + (C/2)(2K + (K+V) + V)] = 139,264 (causal chunked form)
BYTES_PER_TOKEN_HEAD = 1282
STATE_BYTES_PER_SEQ_HEAD = 2 * 128 * 128 * 4
FLOPS_PER_TOKEN_HEAD = 139264
# Decode step: state read + write (2 x 64 KiB per (b, h)) plus q/k/v/graw/b/out (~1.3 KB)
# Backward (token recurrence run twice forwards and once backwards on CUDA cores): per token and
# value head 2 x 3 K V (recomputed updates) + 11 K V (the backward step's products) multiply-adds,
# 2 flops each.
BWD_FLOPS_PER_TOKEN_HEAD = 2 * (2 * 3 + 11) * 128 * 128
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def recorded_traffic(kernel: str):
    """DRAM bytes per launch of `kernel` from the committed ncu record, or None
    when the record is for another kernel or the kernel source changed since."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "roofline_traffic.json")
    try:
        rec = json.load(open(path))
        src = open(os.path.join(ROOT, rec["source"]), "rb").read()
    except Exception:
        return None
    if rec.get("kernel") != kernel or hashlib.sha256(src).hexdigest() != rec.get("source_sha256"):
        return None
    return rec["dram_read_bytes"] + rec["dram_write_bytes"]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            d = json.load(open(path))
            return d, "measured"
        except Exception:
            pass
    return FALLBACK_PEAKS, "fallback"


def peak_value(peaks, *keys):
    for k in keys:
        v = peaks.get(k)
        if isinstance(v, (int, float)):
            return float(v)
        if isinstance(v, dict):
            for kk in ("value", "median", "gbs", "tflops"):
                if isinstance(v.get(kk), (int, float)):
                    return float(v[kk])
    return None


# ---------------------------------------------------------------- distributed plumbing
def dist_init():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def whole_job_value(units_per_rank: int, ms_max: float, world: int) -> float:
    """Throughput of the whole job: every rank processes its own replica of the
    workload (no data-path exchange), so the units add up and the slowest rank
    sets the time."""
    return world * units_per_rank / (ms_max * 1e-3)


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- clocks
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.idx = gpu_index

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = [r for r in csv.reader(io.StringIO(out)) if len(r) >= 9]
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
            except ValueError:
                continue
            for n, val in zip(names, r[5:9]):
                if val.strip().lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- CPU baseline (oracle)
def oracle_sample(inp: KI.KdaInputs, tokens: int) -> KI.KdaInputs:
    """The first ``tokens`` tokens of every sequence of a fixed-length
    workload (same heads, same initial state)."""
    sl = lambda x: x[:, :tokens].contiguous()
    return KI.KdaInputs(q=sl(inp.q), k=sl(inp.k), v=sl(inp.v), graw=sl(inp.graw), b=sl(inp.b), A_log=inp.A_log,
                        scale=inp.scale, initial_state=inp.initial_state, cu_seqlens=None)


def cpu_baseline(inp: KI.KdaInputs, target_s: float = 12.0):
    import oracle
    nthreads = os.cpu_count() or 1
    cal = oracle_sample(inp, 256)
    t0 = time.perf_counter()
    oracle.fwd_inputs(cal, nthreads=nthreads)
    rate = cal.token_heads() / max(time.perf_counter() - t0, 1e-6)
    tokens = int(min(inp.T, max(256, 64 * round(rate * target_s / (inp.B * inp.H_v) / 64))))
    smp = oracle_sample(inp, tokens)
    t0 = time.perf_counter()
    oracle.fwd_inputs(smp, nthreads=nthreads)
    dt = time.perf_counter() - t0
    return {"value": smp.token_heads() / dt, "unit": UNIT, "cores": min(nthreads, inp.B * inp.H_v),
            "kind": "oracle", "seconds": round(dt, 3),
            "sample": f"first {tokens} of {inp.T} tokens of all {inp.B}x{inp.H_v} (sequence, head) chains "
                      f"of the timed workload ({smp.token_heads()} token*heads), fp64 C oracle"}


def run_reference(args, rank, world):
    """--impl reference: the fp64 oracle on the host cores, each step a bounded
    sample of the dense workload."""
    if rank != 0:
        return
    import oracle
    inp = KI.workload("dense")
    nthreads = os.cpu_count() or 1
    cal = oracle_sample(inp, 128)
    t0 = time.perf_counter()
    oracle.fwd_inputs(cal, nthreads=nthreads)
    rate = cal.token_heads() / max(time.perf_counter() - t0, 1e-6)
    budget = 150.0 / max(1, args.steps + args.warmup)
    tokens = int(min(inp.T, max(64, 64 * int(rate * budget / (inp.B * inp.H_v) / 64))))
    smp = oracle_sample(inp, tokens)
    for _ in range(args.warmup):
        oracle.fwd_inputs(smp, nthreads=nthreads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.fwd_inputs(smp, nthreads=nthreads)
    dt = (time.perf_counter() - t0) / max(1, args.steps)
    value = smp.token_heads() / dt
    sample = (f"first {tokens} of {inp.T} tokens of all {inp.B}x{inp.H_v} (sequence, head) chains per step "
              f"({smp.token_heads()} token*heads), fp64 C oracle")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "B": 2, "T": 16384, "H_qk": 32, "H_v": 32, "sample_tokens": tokens},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": nthreads, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- GPU arm
def time_events(fn, steps, stream):
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(steps):
        fn()
    end.record(stream)
    end.synchronize()
    return start.elapsed_time(end) / steps


def run_gpu(args, rank, world, local):
    from gated_delta_rule_40_gb300 import kda
    kda.load()
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    peaks, peak_src = load_peaks()
    hbm_peak = peak_value(peaks, "hbm_gbs", "hbm_GBps", "hbm") or FALLBACK_PEAKS["hbm_gbs"]
    tc_peak = peak_value(peaks, "bf16_tflops_sustained", "bf16_tflops") or FALLBACK_PEAKS["bf16_tflops_sustained"]

    inp = KI.workload("dense", seed=rank)
    d = {n: getattr(inp, n).to(dev) for n in ("q", "k", "v", "graw", "b", "A_log", "initial_state")}
    out = torch.empty((inp.B, inp.T, inp.H_v, 128), dtype=torch.bfloat16, device=dev)
    fin = torch.empty_like(d["initial_state"])

    def step():
        kda.kda_fwd(d["q"], d["k"], d["v"], d["graw"], d["b"], d["A_log"], inp.scale,
                    initial_state=d["initial_state"], out=out, final_state=fin, stream=stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    launches_per_step = kda.kda_last_launch_count()
    clocks = ClockSampler(local)
    clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    ms = time_events(step, args.steps, stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    ms = max_over_ranks(ms, world)
    status = kda.kda_get_status()
    if status != 0:
        raise RuntimeError(f"device status after the timed region: {kda.status_string(status)}")

    units = inp.token_heads()
    value = whole_job_value(units, ms, world)
    alg_bytes = units * BYTES_PER_TOKEN_HEAD + inp.N * inp.H_v * STATE_BYTES_PER_SEQ_HEAD
    alg_flops = units * FLOPS_PER_TOKEN_HEAD
    gbs = alg_bytes / (ms * 1e-3) / 1e9
    tflops = alg_flops / (ms * 1e-3) / 1e12

    # ---- per-kernel durations: a second pass of the same steps with CUDA events
    # recorded by the library between its launches (on the launching stream)
    kda.kda_set_kernel_timing(True)
    per = {}
    for _ in range(args.steps):
        step()
        for name, t in kda.kda_kernel_times():
            per.setdefault(name, []).append(t)
    kda.kda_set_kernel_timing(False)
    kernels = {n: sum(v) / len(v) for n, v in per.items()}
    ksum = sum(kernels.values()) or 1.0
    dom = max(kernels, key=kernels.get) if kernels else None
    dom_ms = kernels.get(dom, ms)

    # ---- end to end through the public call with host buffers
    pin = {n: t.pin_memory() for n, t in
           (("q", inp.q), ("k", inp.k), ("v", inp.v), ("graw", inp.graw), ("b", inp.b),
            ("A_log", inp.A_log), ("initial_state", inp.initial_state))}
    host_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    host_fin = torch.empty(fin.shape, dtype=fin.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in pin.values())
    d2h = host_out.numel() * 2 + host_fin.numel() * 4

    def e2e_step():
        # one C-ABI call on host buffers: H2D of the inputs, the forward and D2H of out and the
        # final state, overlapped piece by piece inside the library
        kda.kda_fwd_host(pin["q"], pin["k"], pin["v"], pin["graw"], pin["b"], pin["A_log"], inp.scale,
                         initial_state=pin["initial_state"], out=host_out, final_state=host_fin, stream=stream,
                         synchronize=False)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    e2e_steps = max(3, min(args.steps, 10))
    barrier(world)
    e2e_ms = max_over_ranks(time_events(e2e_step, e2e_steps, stream), world)

    # ---- scalar gate (one gate value per token and value head): the grouped-value-head
    # workload (28672 + 4096 tokens, H_qk=16, H_v=64) through kda_fwd_scalar_gate, and the
    # general kernel on the same inputs with the gate broadcast along K
    sg = KI.workload("gva")
    sd = {n: getattr(sg, n).to(dev) for n in ("q", "k", "v", "graw", "b", "A_log", "initial_state", "cu_seqlens")}
    sg_g = sg.graw[..., 0].contiguous().to(dev)
    sg_out = torch.empty_like(sd["v"])
    sg_fin = torch.empty_like(sd["initial_state"])

    def sg_step():
        kda.kda_fwd_scalar_gate(sd["q"], sd["k"], sd["v"], sg_g, sd["b"], sd["A_log"], sg.scale,
                                initial_state=sd["initial_state"], cu_seqlens=sd["cu_seqlens"], out=sg_out,
                                final_state=sg_fin, stream=stream)

    def sg_general_step():
        kda.kda_fwd(sd["q"], sd["k"], sd["v"], sd["graw"], sd["b"], sd["A_log"], sg.scale,
                    initial_state=sd["initial_state"], cu_seqlens=sd["cu_seqlens"], out=sg_out, final_state=sg_fin,
                    stream=stream)

    for _ in range(3):
        sg_step()
        sg_general_step()
    torch.cuda.synchronize()
    sg_ms = time_events(sg_step, 10, stream)
    sg_gen_ms = time_events(sg_general_step, 10, stream)
    sg_units = sg.token_heads()
    ntok = sg.q.shape[0] * sg.q.shape[1]
    sg_bytes = (ntok * sg.H_qk * 2 * 256 + ntok * sg.H_v * (256 + 2 + 2 + 256)
                + sg.N * sg.H_v * STATE_BYTES_PER_SEQ_HEAD)
    del sd, sg_g, sg_out, sg_fin

    # ---- decode (B=256, H=64): state GB/s against HBM
    dec = KI.decode_inputs(B=256, H=64, seed=rank)
    dd = {n: getattr(dec, n).to(dev) for n in ("q", "k", "v", "graw", "b", "A_log", "state")}
    dout = torch.empty((256, 64, 128), dtype=torch.bfloat16, device=dev)

    def dec_step():
        kda.kda_decode_step(dd["q"], dd["k"], dd["v"], dd["graw"], dd["b"], dd["A_log"], dec.scale, dd["state"],
                            out=dout, stream=stream)

    for _ in range(5):
        dec_step()
    torch.cuda.synchronize()
    dec_ms = time_events(dec_step, 50, stream)
    dec_bytes = 256 * 64 * (2 * 128 * 128 * 4 + 5 * 256 + 2)
    dec_gbs = dec_bytes / (dec_ms * 1e-3) / 1e9

    # ---- multi-token decode (kda_decode_tokens): Tq = 1 and 4 tokens per pass, fp32 and bf16 state
    multi = {}
    for tq in (1, 4):
        mt = KI.make_inputs(256, tq, 64, 64, seed=rank + 7, with_state=True)
        md = {n: getattr(mt, n).to(dev) for n in ("q", "k", "v", "graw", "b", "A_log")}
        mout = torch.empty((256, tq, 64, 128), dtype=torch.bfloat16, device=dev)
        for sdt, sname, sbytes in ((torch.float32, "fp32", 4), (torch.bfloat16, "bf16", 2)):
            mst = mt.initial_state.to(sdt).to(dev)

            def mstep():
                kda.kda_decode_tokens(md["q"], md["k"], md["v"], md["graw"], md["b"], md["A_log"], mt.scale, mst,
                                      out=mout, stream=stream)

            for _ in range(3):
                mstep()
            torch.cuda.synchronize()
            mms = time_events(mstep, 30, stream)
            mbytes = 256 * 64 * (2 * 128 * 128 * sbytes + tq * (5 * 256 + 2))
            multi[f"T{tq}_{sname}_state"] = {"ms": mms, "tokens_per_s": 256 * tq / (mms * 1e-3),
                                             "GB/s": mbytes / (mms * 1e-3) / 1e9}
        del md, mst, mout

    # ---- lightning attention (fixed per-head decay): forward on the dense and varlen workloads
    # (kda_la_fwd) and the single-token step at B=256, H=64 (kda_la_decode)
    lightning = {}
    for wname in ("la_dense", "la_varlen"):
        la = KI.la_workload(wname, seed=rank)
        ld = {n: getattr(la, n).to(dev) for n in ("q", "k", "v", "slope", "initial_state")}
        lcu = None if la.cu_seqlens is None else la.cu_seqlens.to(dev)
        lout = torch.empty_like(ld["v"])
        lfin = torch.empty_like(ld["initial_state"])

        def la_step():
            kda.kda_la_fwd(ld["q"], ld["k"], ld["v"], ld["slope"], la.scale, initial_state=ld["initial_state"],
                           cu_seqlens=lcu, out=lout, final_state=lfin, stream=stream)

        for _ in range(3):
            la_step()
        torch.cuda.synchronize()
        la_ms = time_events(la_step, 10, stream)
        ntok = la.B * la.T
        la_bytes = ntok * (2 * la.H_qk + 2 * la.H_v) * 256 + la.N * la.H_v * STATE_BYTES_PER_SEQ_HEAD
        lightning[wname] = {"B": la.B, "T": la.T, "N": la.N, "H": la.H_v, "ms": la_ms,
                            "value": la.token_heads() / (la_ms * 1e-3), "unit": UNIT,
                            "algorithmic_bytes": la_bytes, "GB/s": la_bytes / (la_ms * 1e-3) / 1e9,
                            "hbm_peak": hbm_peak, "frac": la_bytes / (la_ms * 1e-3) / 1e9 / hbm_peak}
        del ld, lout, lfin
    lad = KI.la_decode_inputs(B=256, H=64, seed=rank)
    ldd = {n: getattr(lad, n).to(dev) for n in ("q", "k", "v", "slope", "state")}
    ldout = torch.empty((256, 64, 128), dtype=torch.bfloat16, device=dev)

    def la_dec_step():
        kda.kda_la_decode(ldd["q"], ldd["k"], ldd["v"], ldd["slope"], lad.scale, ldd["state"], out=ldout,
                          stream=stream)

    for _ in range(5):
        la_dec_step()
    torch.cuda.synchronize()
    la_dec_ms = time_events(la_dec_step, 50, stream)
    la_dec_bytes = 256 * 64 * (2 * 128 * 128 * 4 + 3 * 256)
    lightning["la_decode"] = {"B": 256, "H": 64, "ms": la_dec_ms, "GB/s": la_dec_bytes / (la_dec_ms * 1e-3) / 1e9,
                              "hbm_peak": hbm_peak, "frac": la_dec_bytes / (la_dec_ms * 1e-3) / 1e9 / hbm_peak}
    del ldd, ldout
    status = kda.kda_get_status()
    if status != 0:
        raise RuntimeError(f"device status after the side measurements: {kda.status_string(status)}")

    # ---- backward of the forward (kda_bwd) on the dense workload: all input gradients from dL/dout
    # and dL/dfinal_state; the token recurrence on CUDA cores, so its roofline is the fp32 FMA rate
    gd = torch.randn(out.shape, generator=torch.Generator().manual_seed(rank), dtype=torch.float32)
    gout = gd.to(torch.bfloat16).to(dev)
    ght = (torch.randn(fin.shape, generator=torch.Generator().manual_seed(rank + 1)) * 0.1).to(dev)
    del gd

    def bwd_step():
        kda.kda_bwd(d["q"], d["k"], d["v"], d["graw"], d["b"], d["A_log"], inp.scale, gout,
                    initial_state=d["initial_state"], dht=ght, stream=stream)

    bwd_step()
    torch.cuda.synchronize()
    bwd_ms = time_events(bwd_step, 3, stream)
    # per-kernel split of one more call (events recorded by the library between its launches)
    kda.kda_set_kernel_timing(True)
    bwd_step()
    bwd_kernels = {name: t for name, t in kda.kda_kernel_times()}
    kda.kda_set_kernel_timing(False)
    bwd_flops = units * BWD_FLOPS_PER_TOKEN_HEAD
    sm_count = torch.cuda.get_device_properties(dev).multi_processor_count
    alu_peak = sm_count * 128 * 2 * (clk.get("sm_max_mhz") or 2070.0) * 1e6 / 1e12
    backward = {"workload": WORKLOAD, "ms": bwd_ms, "value": units / (bwd_ms * 1e-3), "unit": UNIT,
                "roofline": {"bound": "alu", "achieved": bwd_flops / (bwd_ms * 1e-3) / 1e12,
                             "peak": alu_peak, "unit": "TFLOP/s",
                             "frac": bwd_flops / (bwd_ms * 1e-3) / 1e12 / alu_peak,
                             "peak_source": "SMs x 128 fp32 lanes x 2 flops x max SM clock",
                             "flops_per_token_head": BWD_FLOPS_PER_TOKEN_HEAD},
                "kernels_ms": bwd_kernels}
    del gout, ght
    status = kda.kda_get_status()
    if status != 0:
        raise RuntimeError(f"device status after the backward: {kda.status_string(status)}")

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(inp)

    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD, "B": inp.B, "T": inp.T, "H_qk": inp.H_qk, "H_v": inp.H_v, "K": 128,
                   "V": 128, "chunk": 64, "seed": 0,
                   "l2": "inputs larger than L2 (1.4 GB read per step), no flush",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": {"bound": "hbm", "kernel": dom,
                     "achieved": alg_bytes / (dom_ms * 1e-3) / 1e9, "peak": hbm_peak, "unit": "GB/s",
                     "frac": alg_bytes / (dom_ms * 1e-3) / 1e9 / hbm_peak, "traffic": recorded_traffic(dom),
                     "peak_source": peak_src, "kernel_ms": dom_ms,
                     "algorithmic_bytes_per_launch": alg_bytes,
                     "note": "the forward's algorithmic bytes (1282 B per token*head + 128 KiB state per "
                             "sequence*head) over the dominant kernel's event-timed duration"},
        "roofline_step": {"bound": "hbm", "achieved": gbs, "peak": hbm_peak, "unit": "GB/s",
                          "frac": gbs / hbm_peak, "kernel": "whole kda_fwd step"},
        "kernels": {n: {"ms": t, "share": t / ksum} for n, t in kernels.items()},
        "tensor": {"achieved_tflops": tflops, "peak_tflops": tc_peak, "frac": tflops / tc_peak,
                   "flops_per_step": alg_flops, "peak_source": peak_src},
        "e2e": {"value": world * units / (e2e_ms * 1e-3), "unit": UNIT, "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "scalar_gate": {"workload": "grouped value heads, 28672+4096 tokens, H_qk=16 H_v=64, scalar gate",
                        "value": sg_units / (sg_ms * 1e-3), "unit": UNIT, "ms": sg_ms,
                        "general_path_ms": sg_gen_ms, "algorithmic_bytes": sg_bytes,
                        "GB/s": sg_bytes / (sg_ms * 1e-3) / 1e9, "hbm_peak": hbm_peak,
                        "frac": sg_bytes / (sg_ms * 1e-3) / 1e9 / hbm_peak},
        "decode_tokens": {"workload": "B=256 H=64 K=V=128, Tq tokens per pass, state in place", **multi},
        "decode": {"workload": "B=256 H=64 K=V=128 fp32 state in place", "ms": dec_ms, "GB/s": dec_gbs,
                   "hbm_peak": hbm_peak, "frac": dec_gbs / hbm_peak},
        "backward": backward,
        "lightning": {"method": "linear attention with a fixed per-head decay (lightning attention)",
                      "slopes": "2^(-8 (h+1) / H)", **lightning},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    rank, world, local = dist_init()
    try:
        if args.impl == "reference":
            run_reference(args, rank, world)
        else:
            run_gpu(args, rank, world, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
