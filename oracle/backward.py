"""fp64 gradients of the KDA forward (the backward pass), for the tests.

TEST INFRASTRUCTURE ONLY (see the package docstring).  The CUDA library never
imports this module and it imports nothing from the library.

What it computes.  The pages report timings of a gated-delta-rule backward (the
FlashQLA table "benchmark_results_H200.txt", BACKWARD BENCHMARKS) but print no
formula; the backward of a function is fixed by the function, so this module
differentiates the forward recurrence the oracle runs (per sequence and value
head h, S in R^{V x K}):

    qt = scale q / sqrt(|q|^2 + eps),   kh = k / sqrt(|k|^2 + eps),   beta = sigmoid(b)
    g  = -exp(A_log[h]) softplus(graw),   S <- S Diag(exp g),   d = S kh
    S  <- S + beta (v - d) kh^T,          o = S qt

with respect to q, k, v, graw, b, A_log and the initial state, given the
gradients of the loss with respect to the outputs o (do) and the final states
(dht).  It is written as the plain recurrence in torch fp64 and differentiated
by torch.autograd; the pins in the tests compare it with central finite
differences of the independent NumPy explicit-matrix forward
(``oracle.brute_force``).  Value head h reads query/key head h / (H_v / H_qk),
so dq and dk sum over the value heads of a group.
"""
from __future__ import annotations

from typing import Dict, Optional

import torch

EPS = 1e-6


def _recurrence(q, k, v, graw, b, A_log, scale, s0, cu_seqlens, H_qk, mutation=0):
    """The forward in differentiable fp64 torch ops.  q, k [B,T,H_qk,K];
    v, graw [B,T,H_v,*]; b [B,T,H_v]; A_log [H_v]; s0 [N,H_v,V,K]."""
    B, T = q.shape[0], q.shape[1]
    H_v = v.shape[2]
    G = H_v // H_qk
    if cu_seqlens is None:
        segs = [(bi, 0, T) for bi in range(B)]
    else:
        c = [int(x) for x in cu_seqlens.tolist()]
        segs = [(0, c[i], c[i + 1]) for i in range(len(c) - 1)]
    qn = q / torch.sqrt((q * q).sum(-1, keepdim=True) + EPS) * scale
    kn = k / torch.sqrt((k * k).sum(-1, keepdim=True) + EPS)
    beta = torch.sigmoid(b)
    g = -torch.exp(A_log)[None, None, :, None] * torch.nn.functional.softplus(graw)
    rows = {}
    finals = []
    for n, (bi, t0, t1) in enumerate(segs):
        fin_h = []
        for h in range(H_v):
            S = s0[n, h]
            for t in range(t0, t1):
                kk = kn[bi, t, h // G]
                e = torch.exp(g[bi, t, h])
                S = S * (e.detach() if mutation == 1 else e)[None, :]
                d = S @ kk
                if mutation == 2:
                    d = d.detach()
                S = S + beta[bi, t, h] * torch.outer(v[bi, t, h] - d, kk)
                rows[(bi, t, h)] = S @ qn[bi, t, h // G]
            fin_h.append(S)
        finals.append(torch.stack(fin_h))
    out = torch.zeros(v.shape, dtype=torch.float64)
    if rows:
        idx = list(rows.keys())
        out = out.index_put(tuple(torch.tensor([i[j] for i in idx]) for j in range(3)),
                            torch.stack([rows[i] for i in idx]))
    return out, (torch.stack(finals) if finals else s0)


def bwd(q, k, v, graw, b, A_log, scale, initial_state=None, cu_seqlens=None, do=None, dht=None,
        mutation: int = 0) -> Dict[str, torch.Tensor]:
    """Gradients of sum(o * do) + sum(S_final * dht).  Inputs as the forward
    oracle takes them (host tensors, any float dtype; they are promoted to
    fp64 exactly); ``do`` [B,T,H_v,V], ``dht`` [N,H_v,V,K] (None: zero).
    Returns fp64 tensors dq, dk, dv, dgraw, db, dA_log, dh0 (dh0 is the
    gradient with respect to the initial state; zero-initial-state calls get
    it too).  ``mutation`` plants one deliberate mistake for the pin tests:
    1 drops the decay from the gradient path (detaches exp(g)), 2 drops the
    erase term's gradient (detaches d)."""
    f = lambda t: t.detach().to(torch.float64).clone().requires_grad_(True)  # noqa: E731
    B, T, H_qk, K = q.shape
    H_v, V = v.shape[2], v.shape[3]
    N = B if cu_seqlens is None else cu_seqlens.numel() - 1
    qq, kk, vv, gg, bb, aa = f(q), f(k), f(v), f(graw), f(b), f(A_log)
    s0 = f(initial_state) if initial_state is not None else torch.zeros((N, H_v, V, K), dtype=torch.float64,
                                                                        requires_grad=True)
    sc = float(torch.tensor(scale, dtype=torch.float32))
    out, fin = _recurrence(qq, kk, vv, gg, bb, aa, sc, s0, cu_seqlens, H_qk, mutation)
    loss = torch.zeros((), dtype=torch.float64)
    if do is not None:
        loss = loss + (out * do.to(torch.float64)).sum()
    if dht is not None:
        loss = loss + (fin * dht.to(torch.float64)).sum()
    grads = torch.autograd.grad(loss, [qq, kk, vv, gg, bb, aa, s0], allow_unused=True)
    names = ["dq", "dk", "dv", "dgraw", "db", "dA_log", "dh0"]
    refs = [qq, kk, vv, gg, bb, aa, s0]
    return {n: (g_ if g_ is not None else torch.zeros_like(r)).detach() for n, g_, r in zip(names, grads, refs)}


def bwd_inputs(inp, do, dht=None, **kw):
    """``bwd`` on a ``kda_inputs.KdaInputs``."""
    return bwd(inp.q, inp.k, inp.v, inp.graw, inp.b, inp.A_log, inp.scale, inp.initial_state, inp.cu_seqlens,
               do=do, dht=dht, **kw)
