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
# Backward in the chunk form (tf32 tensor-core products), multiply-adds per (64-token chunk, value
# head): prep 10 sub-block pairs x 16x16x128 for A and for P, W and U (64x128x64 each), N (64x128x64);
# forward chain 2 V blocks x (64x64x128 + 64x128x64); backward chain 2 x (64x64x128 + 2 x 64x128x64);
# value side Delta 64x128x128, dDelta 64x128x(64 + 128), dKd / dQg / dW 64x128x128 each, dP and dT
# 64x64x128 each, dBV 64x128x64; key side dT 64x64x128, X and dA 64x64x64 each, dBW 64x128x64, pair
# products 10 x 4 x 16x128x16.  2 flops each, per token and value head (64 tokens per chunk).
BWD_MACS_PER_CHUNK_HEAD = (10 * 2 * 16 * 16 * 128 + 3 * 64 * 128 * 64
                           + 2 * (64 * 64 * 128 + 64 * 128 * 64) + 2 * (64 * 64 * 128 + 2 * 64 * 128 * 64)
                           + 64 * 128 * 128 + 64 * 128 * 192 + 3 * 64 * 128 * 128 + 2 * 64 * 64 * 128
                           + 64 * 128 * 64
                           + 64 * 64 * 128 + 2 * 64 * 64 * 64 + 64 * 128 * 64 + 10 * 4 * 16 * 128 * 16)
BWD_FLOPS_PER_TOKEN_HEAD = 2 * BWD_MACS_PER_CHUNK_HEAD // 64
# nominal dense tf32 : bf16 tensor rates (1.1 : 2.25 PFLOP/s per GPU)
TF32_PER_BF16 = 1.1 / 2.25
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


def bench_config(world: int) -> dict:
    """The timed workload; both arms print the same object."""
    return {"workload": WORKLOAD, "B": 2, "T": 16384, "H_qk": 32, "H_v": 32, "K": 128, "V": 128, "chunk": 64,
            "seed": 0, "l2": "inputs larger than L2 (1.4 GB read per step), no flush",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}


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
            "config": bench_config(world),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": nthreads, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- GPU arm
def time_events(fn, steps, stream):
    """Mean device time of ``steps`` back-to-back calls (one event pair around all)."""
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(steps):
        fn()
    end.record(stream)
    end.synchronize()
    return start.elapsed_time(end) / steps


class L2Flush:
    """Writes a buffer of twice the L2 size on the stream: whatever a previous call
    left in L2 is evicted before the next timed call."""

    def __init__(self, dev):
        l2 = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or (128 << 20)
        self.bytes = max(2 * int(l2), 256 << 20)
        self.buf = torch.empty(self.bytes // 4, dtype=torch.float32, device=dev)

    def __call__(self):
        self.buf.fill_(1.0)


def time_flushed(fn, reps, stream, flush):
    """Median / p10 / p90 device time of ``reps`` calls, each timed by its own event pair
    on the launching stream after an L2 flush outside the timed pair."""
    evs = []
    for _ in range(reps):
        flush()
        s = torch.cuda.Event(enable_timing=True)
        e = torch.cuda.Event(enable_timing=True)
        s.record(stream)
        fn()
        e.record(stream)
        evs.append((s, e))
    stream.synchronize()
    t = sorted(s.elapsed_time(e) for s, e in evs)
    pick = lambda f: t[min(len(t) - 1, int(round(f * (len(t) - 1))))]
    return {"ms": statistics.median(t), "p10_ms": pick(0.1), "p90_ms": pick(0.9), "reps": reps}


def fwd_alg(inp_B, inp_T, H_qk, H_v, nseq, ntok=None):
    """Algorithmic bytes and flops of one forward call (K = V = 128, chunk 64); q and k are
    counted once per q/k head (shared by the value heads of a group)."""
    ntok = inp_B * inp_T if ntok is None else ntok
    units = ntok * H_v
    nbytes = (ntok * H_qk * 2 * 256 + ntok * H_v * (2 * 256 + 2 + 256) + nseq * H_v * STATE_BYTES_PER_SEQ_HEAD)
    return units, nbytes, units * FLOPS_PER_TOKEN_HEAD


def rate_fields(t, units, nbytes, flops, hbm_peak, tc_peak):
    ms = t["ms"]
    gbs = nbytes / (ms * 1e-3) / 1e9
    d = dict(t)
    d.update({"token_heads_per_s": units / (ms * 1e-3), "TFLOP/s": flops / (ms * 1e-3) / 1e12,
              "tensor_frac": flops / (ms * 1e-3) / 1e12 / tc_peak, "algorithmic_bytes": nbytes, "GB/s": gbs,
              "hbm_frac": gbs / hbm_peak})
    if gbs > hbm_peak:
        d["note"] = "above the measured copy bandwidth: some inputs were still cache-resident"
    return d


def bench_configs(kda, d, inp, stream, flush, hbm_peak, tc_peak):
    """Every forward workload of the method's benchmark pages, timed one call at a time
    (median of flushed repetitions): the tiny case, the dense sweep over T and B (the cuLA
    page's KDA fixed-length table), the skewed varlen batch (its varlen table) and the
    grouped-value-head batch through both forward entry points (the FlashQLA table)."""
    res = {}

    def run(name, dd, scale, B, T, H_qk, H_v, nseq, cu=None, fn=None, reps=15, ntok=None):
        out = torch.empty((dd["v"].shape[0], dd["v"].shape[1], H_v, 128), dtype=torch.bfloat16, device=dd["v"].device)
        fin = None if dd.get("initial_state") is None else torch.empty_like(dd["initial_state"])
        call = fn or kda.kda_fwd

        def step():
            call(dd["q"], dd["k"], dd["v"], dd["graw"], dd["b"], dd["A_log"], scale,
                 initial_state=dd.get("initial_state"), cu_seqlens=cu, out=out, final_state=fin, stream=stream)

        for _ in range(3):
            step()
        t = time_flushed(step, reps, stream, flush)
        units, nbytes, flops = fwd_alg(B, T, H_qk, H_v, nseq, ntok)
        res[name] = {"B": B, "T": T, "N": nseq, "H_qk": H_qk, "H_v": H_v,
                     **rate_fields(t, units, nbytes, flops, hbm_peak, tc_peak)}

    tiny = KI.workload("tiny")
    td = {n: getattr(tiny, n).to(d["q"].device) for n in ("q", "k", "v", "graw", "b", "A_log")}
    td["initial_state"] = None
    run("tiny_B1_T256_H2", td, tiny.scale, 1, 256, 2, 2, 1, reps=30)
    for B in (1, 2):
        for T in (512, 1024, 4096, 8192, 16384):
            sub = {n: d[n][:B, :T].contiguous() for n in ("q", "k", "v", "graw", "b")}
            sub["A_log"] = d["A_log"]
            sub["initial_state"] = d["initial_state"][:B].contiguous()
            run(f"dense_B{B}_T{T}", sub, inp.scale, B, T, inp.H_qk, inp.H_v, B)
            del sub
    vl = KI.workload("varlen")
    vd = {n: getattr(vl, n).to(d["q"].device) for n in ("q", "k", "v", "graw", "b", "A_log", "initial_state")}
    run("varlen_20seqs_T16384", vd, vl.scale, 1, vl.T, vl.H_qk, vl.H_v, vl.N, cu=vl.cu_seqlens.to(d["q"].device))
    res["varlen_20seqs_T16384"]["seqlens"] = vl.seqlens()
    del vd
    g = KI.workload("gva")
    gd = {n: getattr(g, n).to(d["q"].device) for n in ("q", "k", "v", "graw", "b", "A_log", "initial_state")}
    gcu = g.cu_seqlens.to(d["q"].device)
    run("gva_28672+4096_general", gd, g.scale, 1, g.T, g.H_qk, g.H_v, g.N, cu=gcu)
    gd["graw"] = g.graw[..., 0].contiguous().to(d["q"].device)
    run("gva_28672+4096_scalar_gate", gd, g.scale, 1, g.T, g.H_qk, g.H_v, g.N, cu=gcu, fn=kda.kda_fwd_scalar_gate)
    # the scalar-gate call reads one gate value per (token, value head): 254 B less per token*head
    sg = res["gva_28672+4096_scalar_gate"]
    ntok = g.T
    sg_bytes = sg["algorithmic_bytes"] - ntok * g.H_v * 254
    sg.update({"algorithmic_bytes": sg_bytes, "GB/s": sg_bytes / (sg["ms"] * 1e-3) / 1e9,
               "hbm_frac": sg_bytes / (sg["ms"] * 1e-3) / 1e9 / hbm_peak})
    del gd
    return res


def bench_decode(kda, dev, stream, flush, hbm_peak, rank):
    """Single-token decode at B in {1, 4, 16, 64, 256}, H = 64 (the cuLA page's decode batch
    column), the state read and written once in place; before each repetition, outside the
    timed pair, the state is restored from a pristine copy and L2 is flushed."""
    res = {}
    for B in (1, 4, 16, 64, 256):
        dec = KI.decode_inputs(B=B, H=64, seed=rank)
        dd = {n: getattr(dec, n).to(dev) for n in ("q", "k", "v", "graw", "b", "A_log", "state")}
        pristine = dd["state"].clone()
        dout = torch.empty((B, 64, 128), dtype=torch.bfloat16, device=dev)

        def dec_step():
            kda.kda_decode_step(dd["q"], dd["k"], dd["v"], dd["graw"], dd["b"], dd["A_log"], dec.scale, dd["state"],
                                out=dout, stream=stream)

        def restore_and_flush():
            dd["state"].copy_(pristine)
            flush()

        for _ in range(5):
            dec_step()
        t = time_flushed(dec_step, 30, stream, restore_and_flush)
        nbytes = B * 64 * (2 * 128 * 128 * 4 + 5 * 256 + 2)
        gbs = nbytes / (t["ms"] * 1e-3) / 1e9
        r = {"B": B, "H": 64, **t, "algorithmic_bytes": nbytes, "GB/s": gbs, "hbm_peak": hbm_peak,
             "frac": gbs / hbm_peak}
        if B <= 16:
            r["note"] = "state of a few MB: launch-latency bound"
        if gbs > hbm_peak:
            r["note"] = "above the measured copy bandwidth"
        res[f"B{B}"] = r
        del dd, dout, pristine
    return res


def bench_link(dev, stream, host_in, host_out):
    """Host-link rates of this machine, measured on the end-to-end call's own pinned buffers (their
    placement in host memory is what that call sees): every input host to device, every output
    device to host, and both at once on two streams."""
    dev_in = [torch.empty(t.shape, dtype=t.dtype, device=dev) for t in host_in]
    dev_out = [torch.empty(t.shape, dtype=t.dtype, device=dev) for t in host_out]
    nbytes_in = sum(t.numel() * t.element_size() for t in host_in)
    nbytes_out = sum(t.numel() * t.element_size() for t in host_out)
    other = torch.cuda.Stream(dev)

    def h2d():
        for d, h in zip(dev_in, host_in):
            d.copy_(h, non_blocking=True)

    def d2h():
        for h, d in zip(host_out, dev_out):
            h.copy_(d, non_blocking=True)

    def one(fn, s):
        fn()
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(s)
        fn()
        b.record(s)
        b.synchronize()
        return a.elapsed_time(b)

    with torch.cuda.stream(stream):
        h2d_ms = one(h2d, stream)
        d2h_ms = one(d2h, stream)

    def both():
        # device time from an event on the launching stream to one after both copy streams
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        other.wait_stream(stream)
        with torch.cuda.stream(stream):
            h2d()
        with torch.cuda.stream(other):
            d2h()
        stream.wait_stream(other)
        b.record(stream)
        b.synchronize()
        return a.elapsed_time(b)

    both()
    both_ms = both()
    return {"h2d_GBps": nbytes_in / (h2d_ms * 1e-3) / 1e9, "d2h_GBps": nbytes_out / (d2h_ms * 1e-3) / 1e9,
            "h2d_ms": h2d_ms, "d2h_ms": d2h_ms, "concurrent_ms": both_ms,
            "note": "measured on the e2e call's own pinned buffers; the e2e step cannot be shorter than "
                    "the input copy alone (h2d_ms)"}


def run_gpu(args, rank, world, local):
    from gated_delta_rule_40_gb300 import kda
    kda.load()
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    peaks, peak_src = load_peaks()
    hbm_peak = peak_value(peaks, "hbm_gbs", "hbm_GBps", "hbm") or FALLBACK_PEAKS["hbm_gbs"]
    # every forward call here lasts milliseconds: the burst tensor peak is its ceiling
    tc_peak = peak_value(peaks, "bf16_tflops", "bf16_tflops_sustained") or FALLBACK_PEAKS["bf16_tflops"]

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
    link = bench_link(dev, stream, list(pin.values()), [host_out, host_fin])
    del pin, host_out, host_fin

    # ---- every workload of the benchmark pages, one call at a time after an L2 flush
    flush = L2Flush(dev)
    configs = bench_configs(kda, d, inp, stream, flush, hbm_peak, tc_peak)
    decode = bench_decode(kda, dev, stream, flush, hbm_peak, rank)

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
            t = time_flushed(mstep, 20, stream, flush)
            mbytes = 256 * 64 * (2 * 128 * 128 * sbytes + tq * (5 * 256 + 2))
            multi[f"T{tq}_{sname}_state"] = {**t, "tokens_per_s": 256 * tq / (t["ms"] * 1e-3),
                                             "GB/s": mbytes / (t["ms"] * 1e-3) / 1e9,
                                             "frac": mbytes / (t["ms"] * 1e-3) / 1e9 / hbm_peak}
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
        t = time_flushed(la_step, 10, stream, flush)
        ntok = la.B * la.T
        la_bytes = ntok * (2 * la.H_qk + 2 * la.H_v) * 256 + la.N * la.H_v * STATE_BYTES_PER_SEQ_HEAD
        lightning[wname] = {"B": la.B, "T": la.T, "N": la.N, "H": la.H_v, **t,
                            "value": la.token_heads() / (t["ms"] * 1e-3), "unit": UNIT,
                            "algorithmic_bytes": la_bytes, "GB/s": la_bytes / (t["ms"] * 1e-3) / 1e9,
                            "hbm_peak": hbm_peak, "frac": la_bytes / (t["ms"] * 1e-3) / 1e9 / hbm_peak}
        del ld, lout, lfin
    lad = KI.la_decode_inputs(B=256, H=64, seed=rank)
    ldd = {n: getattr(lad, n).to(dev) for n in ("q", "k", "v", "slope", "state")}
    ldout = torch.empty((256, 64, 128), dtype=torch.bfloat16, device=dev)

    def la_dec_step():
        kda.kda_la_decode(ldd["q"], ldd["k"], ldd["v"], ldd["slope"], lad.scale, ldd["state"], out=ldout,
                          stream=stream)

    for _ in range(5):
        la_dec_step()
    t = time_flushed(la_dec_step, 30, stream, flush)
    la_dec_bytes = 256 * 64 * (2 * 128 * 128 * 4 + 3 * 256)
    lightning["la_decode"] = {"B": 256, "H": 64, **t, "GB/s": la_dec_bytes / (t["ms"] * 1e-3) / 1e9,
                              "hbm_peak": hbm_peak, "frac": la_dec_bytes / (t["ms"] * 1e-3) / 1e9 / hbm_peak}
    del ldd, ldout
    status = kda.kda_get_status()
    if status != 0:
        raise RuntimeError(f"device status after the side measurements: {kda.status_string(status)}")

    # ---- backward of the forward (kda_bwd) on the dense workload: all input gradients from dL/dout
    # and dL/dfinal_state
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
    tf32_peak = tc_peak * TF32_PER_BF16
    backward = {"workload": WORKLOAD, "ms": bwd_ms, "value": units / (bwd_ms * 1e-3), "unit": UNIT,
                "roofline": {"bound": "tensor", "achieved": bwd_flops / (bwd_ms * 1e-3) / 1e12,
                             "peak": tf32_peak, "unit": "TFLOP/s",
                             "frac": bwd_flops / (bwd_ms * 1e-3) / 1e12 / tf32_peak,
                             "peak_source": f"{peak_src} bf16 burst x nominal tf32/bf16 ratio {TF32_PER_BF16:.3f}",
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
        "config": bench_config(world),
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
                   "flops_per_step": alg_flops, "peak_source": peak_src + " (burst)"},
        "e2e": {"value": world * units / (e2e_ms * 1e-3), "unit": UNIT, "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "link": link},
        "configs": configs,
        "decode": {"workload": "H=64 K=V=128 fp32 state in place, L2 flushed before each repetition",
                   "ms": decode["B256"]["ms"], "GB/s": decode["B256"]["GB/s"], "hbm_peak": hbm_peak,
                   "frac": decode["B256"]["frac"], "batch": decode},
        "decode_tokens": {"workload": "B=256 H=64 K=V=128, Tq tokens per pass, state in place", **multi},
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
