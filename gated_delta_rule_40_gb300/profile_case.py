"""Run the KDA (or lightning-attention) forward a few times on one seeded workload, for profilers.

    python -m gated_delta_rule_40_gb300.profile_case --B 1 --T 8192 --H 32 --iters 4
    python -m gated_delta_rule_40_gb300.profile_case --method la --B 1 --T 8192 --H 64 --iters 4
    python -m gated_delta_rule_40_gb300.profile_case --method bwd --B 1 --T 2048 --H 8 --iters 3
    python -m gated_delta_rule_40_gb300.profile_case --method bwd --B 2 --T 16384 --H 32 --iters 2 --kernel-times
    python -m gated_delta_rule_40_gb300.profile_case --method la_decode --B 256 --H 64 --iters 4
    python -m gated_delta_rule_40_gb300.profile_case --method decode --B 256 --H 64 --iters 4
    python -m gated_delta_rule_40_gb300.profile_case --method gdn --B 1 --T 8192 --H 32 --iters 4
    python -m gated_delta_rule_40_gb300.profile_case --method decode_tokens --B 256 --T 4 --H 64 --iters 4

Inputs come from ``kda_inputs`` (same recipe as the tests and the benchmark);
the workspace is allocated once, so every iteration is exactly the three
kernel launches of ``kda_fwd`` (three for ``kda_fwd_scalar_gate``: plan, intra_gdn_kernel
and scan_kernel; two for ``kda_la_fwd``: plan and la_fwd_kernel; eight for ``kda_bwd``:
plan, bwdc_prep_kernel, bwdc_chain_kernel forward and backward, bwdc_gradv_kernel,
bwdc_gradk_kernel, bwdc_jacobian_kernel and bwdc_dalog_kernel; one for ``kda_decode_tokens``, whose
``--T`` is the token count Tq of the step and whose state is fp32 unless
``--bf16-state``; one for ``kda_decode_step``).  A profiler then selects launches by kernel name and index (e.g.
``ncu -k regex:intra_kernel -s 2 -c 1``).  ``--kernel-times`` (kda and bwd) times the
last iteration's kernels with the library's CUDA events instead and prints them.
"""
import argparse
import os
import sys

import torch

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import kda_inputs  # noqa: E402
from gated_delta_rule_40_gb300 import kda  # noqa: E402


def main() -> None:
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--B", type=int, default=1)
    ap.add_argument("--T", type=int, default=8192)
    ap.add_argument("--H", type=int, default=32, help="value heads (= q/k heads)")
    ap.add_argument("--iters", type=int, default=4)
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--method", choices=["kda", "gdn", "la", "bwd", "la_decode", "decode_tokens", "decode"],
                    default="kda")
    ap.add_argument("--bf16-state", action="store_true", help="decode_tokens: bf16 state")
    ap.add_argument("--kernel-times", action="store_true",
                    help="time the last iteration's kernels with the library's events and print them")
    a = ap.parse_args()
    def timed(i):
        if a.kernel_times:
            kda.kda_set_kernel_timing(i == a.iters - 1)

    def report():
        if a.kernel_times:
            for name, ms in kda.kda_kernel_times():
                print(f"  {name}: {ms:.4f} ms")
            kda.kda_set_kernel_timing(False)
    if a.method == "decode_tokens":
        x = kda_inputs.make_inputs(a.B, a.T, a.H, a.H, seed=a.seed, with_state=True)
        q, k, v, gr, b, A = (t.cuda() for t in (x.q, x.k, x.v, x.graw, x.b, x.A_log))
        st = x.initial_state.to(torch.bfloat16 if a.bf16_state else torch.float32).cuda()
        for _ in range(a.iters):
            o = kda.kda_decode_tokens(q, k, v, gr, b, A, x.scale, st)
        torch.cuda.synchronize()
        print(f"kda_decode_tokens B={a.B} Tq={a.T} H={a.H} state {st.dtype} x{a.iters}: "
              f"|o| {float(o.float().abs().mean()):.6f}")
        return
    if a.method == "decode":
        d = kda_inputs.decode_inputs(B=a.B, H=a.H, seed=a.seed)
        q, k, v, gr, b, A, st = (t.cuda() for t in (d.q, d.k, d.v, d.graw, d.b, d.A_log, d.state))
        for _ in range(a.iters):
            o = kda.kda_decode_step(q, k, v, gr, b, A, d.scale, st)
        torch.cuda.synchronize()
        print(f"kda_decode_step B={a.B} H={a.H} x{a.iters}: |o| {float(o.float().abs().mean()):.6f}")
        return
    if a.method == "la_decode":
        d = kda_inputs.la_decode_inputs(B=a.B, H=a.H, seed=a.seed)
        q, k, v, sl, st = (t.cuda() for t in (d.q, d.k, d.v, d.slope, d.state))
        for _ in range(a.iters):
            o = kda.kda_la_decode(q, k, v, sl, d.scale, st)
        torch.cuda.synchronize()
        print(f"kda_la_decode B={a.B} H={a.H} x{a.iters}: |o| {float(o.float().abs().mean()):.6f}")
        return
    if a.method == "la":
        x = kda_inputs.make_la_inputs(a.B, a.T, a.H, a.H, seed=a.seed)
        q, k, v, sl, s0 = (t.cuda() for t in (x.q, x.k, x.v, x.slope, x.initial_state))
        for _ in range(a.iters):
            out, fin = kda.kda_la_fwd(q, k, v, sl, x.scale, initial_state=s0)
        torch.cuda.synchronize()
        print(f"kda_la_fwd B={a.B} T={a.T} H={a.H} x{a.iters}: |out| {float(out.float().abs().mean()):.6f} "
              f"|S| {float(fin.abs().mean()):.6f}")
        return
    x = kda_inputs.make_inputs(B=a.B, T=a.T, H_qk=a.H, H_v=a.H, seed=a.seed, with_state=True,
                               scalar_gate=a.method == "gdn")
    if a.method == "gdn":
        q, k, v, b, A, s0 = (t.cuda() for t in (x.q, x.k, x.v, x.b, x.A_log, x.initial_state))
        gr = x.graw[..., 0].contiguous().cuda()
        for _ in range(a.iters):
            out, fin = kda.kda_fwd_scalar_gate(q, k, v, gr, b, A, x.scale, initial_state=s0)
        torch.cuda.synchronize()
        print(f"kda_fwd_scalar_gate B={a.B} T={a.T} H={a.H} x{a.iters}: |out| {float(out.float().abs().mean()):.6f} "
              f"|S| {float(fin.abs().mean()):.6f}")
        return
    if a.method == "bwd":
        g = torch.Generator().manual_seed(a.seed + 1)
        dout = torch.randn(x.v.shape, generator=g).to(torch.bfloat16).cuda()
        q, k, v, gr, b, A, s0 = (t.cuda() for t in (x.q, x.k, x.v, x.graw, x.b, x.A_log, x.initial_state))
        for i in range(a.iters):
            timed(i)
            grads = kda.kda_bwd(q, k, v, gr, b, A, x.scale, dout, initial_state=s0)
        torch.cuda.synchronize()
        print(f"kda_bwd B={a.B} T={a.T} H={a.H} x{a.iters}: |dq| {float(grads['dq'].abs().mean()):.6f} "
              f"|dh0| {float(grads['dh0'].abs().mean()):.6f}")
        report()
        return
    dev = lambda t: t.cuda() if t is not None else None  # noqa: E731
    q, k, v, g, b, A, s0 = map(dev, (x.q, x.k, x.v, x.graw, x.b, x.A_log, x.initial_state))
    ws = torch.empty(kda.kda_fwd_workspace_size(a.B, a.B, a.T, a.H, a.H), dtype=torch.uint8, device="cuda")
    for i in range(a.iters):
        timed(i)
        out, fin = kda.kda_fwd(q, k, v, g, b, A, x.scale, initial_state=s0, workspace=ws)
    torch.cuda.synchronize()
    print(f"kda_fwd B={a.B} T={a.T} H={a.H} x{a.iters}: |out| {float(out.float().abs().mean()):.6f} "
          f"|S| {float(fin.abs().mean()):.6f}")
    report()


if __name__ == "__main__":
    main()
