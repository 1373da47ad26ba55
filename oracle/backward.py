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


def bwd_recurrent(q, k, v, graw, b, A_log, scale, initial_state=None, cu_seqlens=None, do=None, dht=None,
                  checkpoint: int = 64) -> Dict[str, "object"]:
    """The same gradients as ``bwd``, by an explicit reverse pass in NumPy fp64
    with the state stored every ``checkpoint`` tokens (memory O(T/checkpoint)
    states per chain instead of autograd's tape), for long sequences.  Per
    token, walking backwards with dS = dL/dS_t:
    dS += do qt^T, dqt = S_t^T do, ddel = dS kh, dkh = dS^T delta + S'^T dd
    (dd = -beta ddel), dv = beta ddel, dbeta = ddel . (v - d), dS' = dS + dd kh^T,
    de = colsum(S_{t-1} * dS'), dS_{t-1} = dS' Diag(e); then the Jacobians of
    the norms, the gate and the sigmoid.  Pinned to ``bwd`` (autograd) by the
    tests."""
    import numpy as np
    f64 = lambda t: t.detach().to(torch.float64).numpy()  # noqa: E731
    qq, kk, vv, gg, bb, aa = (f64(t) for t in (q, k, v, graw, b, A_log))
    B, T, H_qk, K = qq.shape
    H_v, V = vv.shape[2], vv.shape[3]
    G = H_v // H_qk
    segs = ([(bi, 0, T) for bi in range(B)] if cu_seqlens is None else
            [(0, int(cu_seqlens[i]), int(cu_seqlens[i + 1])) for i in range(cu_seqlens.numel() - 1)])
    sc = float(np.float32(scale))
    nq = np.sqrt((qq * qq).sum(-1, keepdims=True) + EPS)
    nk = np.sqrt((kk * kk).sum(-1, keepdims=True) + EPS)
    qt, kh = sc * qq / nq, kk / nk
    beta = 1.0 / (1.0 + np.exp(-bb))
    a = np.exp(aa)
    sp = np.maximum(gg, 0.0) + np.log1p(np.exp(-np.abs(gg)))
    g = -a[None, None, :, None] * sp
    e = np.exp(g)
    dO = np.zeros(vv.shape) if do is None else f64(do)
    dqt, dkh = np.zeros((B, T, H_v, K)), np.zeros((B, T, H_v, K))
    de, dbeta, dv = np.zeros((B, T, H_v, K)), np.zeros((B, T, H_v)), np.zeros(vv.shape)
    dh0 = np.zeros((len(segs), H_v, V, K))
    for n, (bi, t0, t1) in enumerate(segs):
        for h in range(H_v):
            hq = h // G
            S = np.zeros((V, K)) if initial_state is None else f64(initial_state[n, h]).copy()
            ck = {}
            for t in range(t0, t1):
                if (t - t0) % checkpoint == 0:
                    ck[t] = S.copy()
                S = S * e[bi, t, h][None, :]
                S = S + beta[bi, t, h] * np.outer(vv[bi, t, h] - S @ kh[bi, t, hq], kh[bi, t, hq])
            dS = np.zeros((V, K)) if dht is None else f64(dht[n, h]).copy()
            starts = sorted(ck.keys(), reverse=True)
            for c0 in starts:
                c1 = min(c0 + checkpoint, t1)
                states = [ck[c0].copy()]
                for t in range(c0, c1 - 1):
                    Sx = states[-1] * e[bi, t, h][None, :]
                    states.append(Sx + beta[bi, t, h] * np.outer(vv[bi, t, h] - Sx @ kh[bi, t, hq], kh[bi, t, hq]))
                for t in range(c1 - 1, c0 - 1, -1):
                    Sp = states[t - c0]
                    k_, q_, b_ = kh[bi, t, hq], qt[bi, t, hq], beta[bi, t, h]
                    S1 = Sp * e[bi, t, h][None, :]
                    d = S1 @ k_
                    delta = b_ * (vv[bi, t, h] - d)
                    St = S1 + np.outer(delta, k_)
                    dS = dS + np.outer(dO[bi, t, h], q_)
                    dqt[bi, t, h] = St.T @ dO[bi, t, h]
                    ddel = dS @ k_
                    dv[bi, t, h] = b_ * ddel
                    dbeta[bi, t, h] = ddel @ (vv[bi, t, h] - d)
                    dd = -b_ * ddel
                    dkh[bi, t, h] = dS.T @ delta + S1.T @ dd
                    dS = dS + np.outer(dd, k_)
                    de[bi, t, h] = (Sp * dS).sum(0)
                    dS = dS * e[bi, t, h][None, :]
            dh0[n, h] = dS
    # Jacobians: norms (dq, dk summed over each group's value heads), gate, sigmoid
    dqs = dqt.reshape(B, T, H_qk, G, K).sum(3)
    dks = dkh.reshape(B, T, H_qk, G, K).sum(3)
    rq, rk = 1.0 / nq, 1.0 / nk
    dq = sc * rq * (dqs - rq * rq * qq * (qq * dqs).sum(-1, keepdims=True))
    dk = rk * (dks - rk * rk * kk * (kk * dks).sum(-1, keepdims=True))
    dg = de * e
    sig = 1.0 / (1.0 + np.exp(-gg))
    dgraw = dg * (-a[None, None, :, None]) * sig
    dA_log = (dg * g).sum(axis=(0, 1, 3))
    db = dbeta * beta * (1.0 - beta)
    out = dict(dq=dq, dk=dk, dv=dv, dgraw=dgraw, db=db, dA_log=dA_log, dh0=dh0)
    return {n_: torch.from_numpy(np.ascontiguousarray(x)) for n_, x in out.items()}


def bwd_recurrent_inputs(inp, do, dht=None, **kw):
    """``bwd_recurrent`` on a ``kda_inputs.KdaInputs``."""
    return bwd_recurrent(inp.q, inp.k, inp.v, inp.graw, inp.b, inp.A_log, inp.scale, inp.initial_state,
                         inp.cu_seqlens, do=do, dht=dht, **kw)
