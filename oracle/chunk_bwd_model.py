"""Chunked (UT / WY) backward of the KDA forward in NumPy fp64.

TEST INFRASTRUCTURE ONLY (see the package docstring).  The algebra a chunked,
tensor-core backward is built on, written out plainly so the tests can pin it
against the autograd oracle; the GPU code shares nothing with it.

Forward per chunk (C rows; S_0 the state entering it; Gam the inclusive in-chunk
prefix of the log decay g, per channel; Gam_C its last row; natural units):

  Kg = Kh e^{Gam},  Kn = Kh e^{-Gam},  Qg = Qt e^{Gam},  Kd = Kh e^{Gam_C - Gam}
  A  = strict_lower(diag(beta) Kg Kn^T),   P = lower(Qg Kn^T),   T = (I + A)^{-1}
  U  = T diag(beta) V,   W = T diag(beta) Kg,   Delta = U - W S_0^T
  O  = Qg S_0^T + P Delta,   S_C = S_0 Diag(e^{Gam_C}) + Delta^T Kd

Backward of one chunk, given dO and dS_C (products read right to left):

  dDelta = P^T dO + Kd dS_C^T          dKd = Delta dS_C         dQg = dO S_0
  dS_0   = dO^T Qg + dS_C Diag(e^{Gam_C}) - dDelta^T W
  dP     = lower(dO Delta^T)           dU = dDelta              dW = -dDelta S_0
  dT     = dU (diag(beta) V)^T + dW (diag(beta) Kg)^T
  dA     = strict_lower(-T^T dT T^T)
  then the products A, P, U, W and the decayed copies pass their gradients to
  Kh, Qt, V, beta and Gam, and dg_s = sum_{r >= s} dGam_r (plus the Gam_C terms).

Chunks are visited in reverse with dS carried from each chunk's S_0 to the
previous chunk's S_C; the forward states S_0 come from a forward pass.  The
prologue's Jacobians (norms, gate, sigmoid) are those of ``backward.bwd``.

``form="pairwise"`` writes the products that pair a key with an earlier key or
query (A, P and their gradients) with the pairwise decays e^{Gam_r - Gam_j}
(j <= r, at most 1) instead of the e^{+Gam} / e^{-Gam} split, so no factor
overflows however strong the gate (the split's e^{-Gam} exceeds the fp64 range
once a chunk's decay passes 709 nats).  With M = diag(beta) dA and N = dP:

  dKh_r += sum_j M_rj Kh_j e^{Gam_r - Gam_j} + sum_i M_ir Kh_i e^{Gam_i - Gam_r}
           + sum_i N_ir Qt_i e^{Gam_i - Gam_r}
  dQt_r += sum_j N_rj Kh_j e^{Gam_r - Gam_j}
  dGam_r  gets each term above times Kh_r or Qt_r, with the sign of Gam_r in its
          exponent (plus for the row side, minus for the column side); P's diagonal
          (decay e^0) enters dQt and dKh but not dGam

and the other terms as in the split form, except that Kd_r = Kh_r e^{Gam_C - Gam_r},
which depends on g_s for s > r only, reaches dg through an exclusive prefix sum
(the split form adds it to every token through Gam_C and takes it back from the
tokens s <= r, two equal amounts that cancel when the gate is strong).

``form="blocked"`` computes those key products as a kernel does: per pair of
16-row sub-blocks, one product of the gradient block (diag(beta) dA or dP) with a
decayed operand (Kh or Qt times a factor <= 1 against the block's reference point,
as the forward builds A and P; diagonal blocks use the midpoint with exponents
clamped at ``clamp``, exact while a channel decays by less than 2 clamp nats
across a block), scaled afterwards by the other factor.  Its Gam terms multiply
the products by the same (rounded) decayed operands that entered them, so that a
pair (r, j) reaches row r and row j as one and the same product and the two
cancel in dg's suffix sums as they do in exact arithmetic.

``rounding`` maps operand names to a number format the operand is rounded to
where it enters a product (``"bf16"`` nearest-even, ``"tf32"`` nearest-even to
10 fraction bits, ``"tf32_trunc"`` the low 13 bits dropped, ``"f32"``), so the
tests can choose a tensor-core backward's operand formats: the state side S0,
dS, W, Qg (in dOᵀQg), P, Kd, Delta, dDelta, dW, BV = diag(beta) V, T, dT, dA and
dP, and in the blocked form the decayed keys and queries (Kdec, Qdec), whose
products then accumulate in fp32.  The split and pairwise forms do not round the
key products: in the split form they cancel (bf16 there costs rel-L2 0.3 to 11
on dk and dgraw), and the pairwise form is the definition the blocked form
factors.
"""
from __future__ import annotations

from typing import Dict, Optional

import numpy as np
import torch

from .backward import EPS

ROUNDABLE = ("S0", "dS", "W", "Qg", "P", "Kd", "Delta", "dDelta", "dW", "BV", "T", "dT", "dA", "dP",
             "Kdec", "Qdec")
SUB = 16   # sub-block rows of the blocked form (the forward's decay blocks)


def _round(x: np.ndarray, fmt: str) -> np.ndarray:
    """``x`` rounded to ``fmt`` (through fp32) and returned in fp64."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    if fmt == "bf16":
        u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    elif fmt == "tf32":
        u = (u + 0xFFF + ((u >> 13) & 1)) & 0xFFFFE000
    elif fmt == "tf32_trunc":
        u = u & 0xFFFFE000
    elif fmt == "f32":
        pass
    else:
        raise ValueError(fmt)
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


def _block_factors(Gam: np.ndarray, clamp: float):
    """Per (row block i, column block b <= i) of SUB rows: (rowf, colf) with
    e^{Gam_r - Gam_j} = rowf[r] * colf[j] (per channel) for r in block i, j in block b,
    j < r.  Below the diagonal the reference is Gam at the end of block i - 1 (both
    factors <= 1); on it, the block's per-channel midpoint with both exponents
    clamped at ``clamp`` (exact unless a channel decays by more than 2 clamp nats
    across the block), as the forward builds A and P."""
    L = Gam.shape[0]
    nb = (L + SUB - 1) // SUB
    out = {}
    for i in range(nb):
        r0, r1 = i * SUB, min(L, (i + 1) * SUB)
        if i > 0:
            m = Gam[r0 - 1]
            rowf = np.exp(Gam[r0:r1] - m)
            for bb in range(i):
                out[(i, bb)] = (rowf, np.exp(m - Gam[bb * SUB:(bb + 1) * SUB]))
        mid = 0.5 * (Gam[r0] + Gam[r1 - 1])
        out[(i, i)] = (np.exp(np.minimum(Gam[r0:r1] - mid, clamp)), np.exp(np.minimum(mid - Gam[r0:r1], clamp)))
    return out, nb


def _key_products(M, Kh, Qt, Gam, clamp, rk, rq, acc=lambda x: x):
    """For a strictly lower L x L matrix M (diag(beta) dA, or dP without its
    diagonal) the four contractions of the key products, block pair by block pair
    as a kernel forms them: one product of M's block with a decayed operand
    (``rk`` / ``rq``: its rounding), scaled afterwards by the other factor.
      XK[r] = sum_j M_rj Kh_j e^{Gam_r - Gam_j}     YK[j] = sum_r M_rj Kh_r e^{Gam_r - Gam_j}
      YQ[j] = sum_r M_rj Qt_r e^{Gam_r - Gam_j}
    (XK with the keys is also the query-side sum of P's gradient), each product's
    accumulator passed through ``acc``; and the four Gam-side terms Kh_r XK_r,
    Kh_j YK_j, Qt_r XK_r, Kh_j YQ_j formed from the rounded operands."""
    L, K = Kh.shape
    fac, nb = _block_factors(Gam, clamp)
    XK, YK, YQ = np.zeros((L, K)), np.zeros((L, K)), np.zeros((L, K))
    gXK, gYK, gXQ, gYQ = (np.zeros((L, K)) for _ in range(4))
    strict16 = np.tril(np.ones((SUB, SUB)), -1)
    for (i, bb), (rowf, colf) in fac.items():
        r0, r1 = i * SUB, min(L, (i + 1) * SUB)
        j0, j1 = bb * SUB, min(L, (bb + 1) * SUB)
        Mb = M[r0:r1, j0:j1]
        if i == bb:
            Mb = Mb * strict16[:r1 - r0, :j1 - j0]
        Hk = rk(Kh[j0:j1] * colf)          # the decayed operands as they enter the products
        Fk = rk(Kh[r0:r1] * rowf)
        Fq = rq(Qt[r0:r1] * rowf)
        MH, MtF, MtQ = acc(Mb @ Hk), acc(Mb.T @ Fk), acc(Mb.T @ Fq)
        XK[r0:r1] += rowf * MH
        YK[j0:j1] += colf * MtF
        YQ[j0:j1] += colf * MtQ
        # the Gam terms multiply by the same rounded operands, so that each pair (r, j)
        # enters row r and row j as the same product and the two cancel in dg's suffix sums
        gXK[r0:r1] += Fk * MH
        gYK[j0:j1] += Hk * MtF
        gXQ[r0:r1] += Fq * MH
        gYQ[j0:j1] += Hk * MtQ
    return XK, YK, YQ, (gXK, gYK, gXQ, gYQ)


def chunk_bwd(q, k, v, graw, b, A_log, scale, initial_state=None, cu_seqlens=None, do=None, dht=None,
              C: int = 64, rounding: Optional[Dict[str, str]] = None, form: str = "split",
              clamp: float = 85.0, return_intermediates: bool = False):
    """Gradients as ``backward.bwd`` returns them (fp64 tensors), computed with
    the chunked formulas above (operands rounded as ``rounding`` names; key
    products in the ``form`` "split", "pairwise" or "blocked").

    With ``return_intermediates`` it returns ``(grads, inter)``, ``inter`` holding
    per (sequence n, value head h, chunk start c0) the quantities a phased kernel
    passes between its phases: ``"S0"`` the state entering the chunk, ``"dS_end"``
    the gradient with respect to the state leaving it, ``"dDelta"`` the gradient
    with respect to the chunk's rows Delta (fp64 NumPy arrays)."""
    if form not in ("split", "pairwise", "blocked"):
        raise ValueError(form)
    pairwise = form in ("pairwise", "blocked")
    rnd = dict(rounding or {})
    bad = set(rnd) - set(ROUNDABLE if form == "blocked" else ROUNDABLE[:-2])
    if bad:
        raise ValueError(f"not roundable in the {form} form: {sorted(bad)}")
    r = lambda name, x: _round(x, rnd[name]) if name in rnd else x  # noqa: E731
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
    qt_all, kh_all = sc * qq / nq, kk / nk
    beta_all = 1.0 / (1.0 + np.exp(-bb))
    a = np.exp(aa)
    sp = np.maximum(gg, 0.0) + np.log1p(np.exp(-np.abs(gg)))
    g_all = -a[None, None, :, None] * sp
    dO_all = np.zeros(vv.shape) if do is None else f64(do)
    dqt, dkh = np.zeros((B, T, H_v, K)), np.zeros((B, T, H_v, K))
    dg, dbeta, dv = np.zeros((B, T, H_v, K)), np.zeros((B, T, H_v)), np.zeros(vv.shape)
    dh0 = np.zeros((len(segs), H_v, V, K))
    inter = {"S0": {}, "dS_end": {}, "dDelta": {}}
    for n, (bi, t0, t1) in enumerate(segs):
        for h in range(H_v):
            hq = h // G
            S = np.zeros((V, K)) if initial_state is None else f64(initial_state[n, h]).copy()
            starts = list(range(t0, t1, C))
            S0s = []
            for c0 in starts:                                  # forward: states at chunk starts
                S0s.append(S.copy())
                for t in range(c0, min(c0 + C, t1)):
                    S = S * np.exp(g_all[bi, t, h])[None, :]
                    kh = kh_all[bi, t, hq]
                    S = S + beta_all[bi, t, h] * np.outer(vv[bi, t, h] - S @ kh, kh)
            dS = np.zeros((V, K)) if dht is None else f64(dht[n, h]).copy()
            for c0, S0 in reversed(list(zip(starts, S0s))):
                c1 = min(c0 + C, t1)
                Qt, Kh = qt_all[bi, c0:c1, hq], kh_all[bi, c0:c1, hq]
                Vc, be, gc = vv[bi, c0:c1, h], beta_all[bi, c0:c1, h], g_all[bi, c0:c1, h]
                dO = dO_all[bi, c0:c1, h]
                L = c1 - c0
                inter["S0"][(n, h, c0)] = S0.copy()
                inter["dS_end"][(n, h, c0)] = dS.copy()
                Gam = np.cumsum(gc, axis=0)
                GC = Gam[-1]
                eG = np.exp(Gam)
                Kg, Qg, Kd = Kh * eG, Qt * eG, Kh * np.exp(GC[None, :] - Gam)
                strict = np.tril(np.ones((L, L)), -1)
                incl = np.tril(np.ones((L, L)))
                if pairwise:
                    # E[r, j, c] = e^{Gam_rc - Gam_jc} for j <= r, 0 above the diagonal
                    E = np.exp(np.where(incl[:, :, None] > 0, Gam[:, None, :] - Gam[None, :, :], -np.inf))
                    KK = np.einsum("rc,jc,rjc->rj", Kh, Kh, E)
                    P = incl * np.einsum("rc,jc,rjc->rj", Qt, Kh, E)
                else:
                    enG = np.exp(-Gam)
                    Kn = Kh * enG
                    KK = Kg @ Kn.T
                    P = incl * (Qg @ Kn.T)
                A = strict * (be[:, None] * KK)
                Tm = np.linalg.inv(np.eye(L) + A)
                BV, BW = be[:, None] * Vc, be[:, None] * Kg
                U, W = Tm @ BV, Tm @ BW
                Delta = U - W @ S0.T
                # ---- backward of the chunk (r(): an operand as it enters a product)
                S0r, dSr, Wr = r("S0", S0), r("dS", dS), r("W", W)
                if rnd:
                    Delta = U - Wr @ S0r.T
                dDelta = r("P", P).T @ dO + r("Kd", Kd) @ dSr.T
                dKd = r("Delta", Delta) @ dSr
                dQg = dO @ S0r
                dDr = r("dDelta", dDelta)
                dS0 = dO.T @ r("Qg", Qg) + dS * np.exp(GC)[None, :] - dDr.T @ Wr
                dGC = (S0 * dS).sum(0) * np.exp(GC)
                dP = incl * (dO @ r("Delta", Delta).T)
                dU, dW = dDelta, -dDr @ S0r
                dWr, Tr = r("dW", dW), r("T", Tm)
                dT = dDr @ r("BV", BV).T + dWr @ BW.T
                dBV, dBW = Tr.T @ dDr, Tr.T @ dWr
                dA = strict * (-(Tr.T @ r("dT", dT) @ Tr.T))
                dbe = (dBV * Vc).sum(1) + (dBW * Kg).sum(1) + (dA * KK).sum(1)
                dVc = be[:, None] * dBV
                dAr, dPr = r("dA", dA), r("dP", dP)
                if pairwise:
                    M = be[:, None] * dAr
                    # P's diagonal (decay e^0 = 1) has no Gam gradient: its terms enter dQt and dKh
                    # only, so the Gam terms never add and subtract O(1) amounts that cancel exactly
                    dPs, dPd = strict * dPr, np.diag(dPr)[:, None]
                    if form == "blocked":
                        rk = lambda x: r("Kdec", x)  # noqa: E731
                        rq = lambda x: r("Qdec", x)  # noqa: E731
                        acc = (lambda x: _round(x, "f32")) if rnd else (lambda x: x)  # noqa: E731
                        XA, YA, _, gA = _key_products(M, Kh, Qt, Gam, clamp, rk, rq, acc)
                        XP, _, YP, gP = _key_products(dPs, Kh, Qt, Gam, clamp, rk, rq, acc)
                        gamKey = gA[0] - gA[1] + gP[2] - gP[3]
                    else:
                        XA = np.einsum("rj,jc,rjc->rc", M, Kh, E)      # row side of A
                        YA = np.einsum("rj,rc,rjc->jc", M, Kh, E)      # column side of A
                        XP = np.einsum("rj,jc,rjc->rc", dPs, Kh, E)    # row side of P (the query)
                        YP = np.einsum("rj,rc,rjc->jc", dPs, Qt, E)    # column side of P (the key)
                    dKgW = be[:, None] * dBW
                    dKh_c = dKgW * eG + XA + YA + YP + dPd * Qt + dKd * np.exp(GC[None, :] - Gam)
                    dQt_c = dQg * eG + XP + dPd * Kh
                    if form == "blocked":
                        dGam = dKgW * Kg + gamKey + dQg * Qg
                    else:
                        dGam = dKgW * Kg + Kh * (XA - YA - YP) + dQg * Qg + Qt * XP
                else:
                    dKg = be[:, None] * dBW + be[:, None] * (dAr @ Kn)
                    dKn = dAr.T @ (be[:, None] * Kg) + dPr.T @ Qg
                    dQg = dQg + dPr @ Kn
                    dKh_c = dKg * eG + dKn * enG + dKd * np.exp(GC[None, :] - Gam)
                    dGam = dKg * Kg - dKn * Kn + dQg * Qg - dKd * Kd
                    dQt_c = dQg * eG
                if not pairwise:
                    dGC = dGC + (dKd * Kd).sum(0)
                # Gam_r = sum_{s <= r} g_s and Gam_C = Gam_{L-1}: dg_s = sum_{r >= s} dGam_r + dGam_C
                if pairwise:
                    # Kd_r = Kh_r e^{Gam_C - Gam_r} depends on g_s for s > r only: an exclusive
                    # prefix sum, instead of a whole-chunk term minus the rows r >= s
                    kdk = dKd * Kd
                    dgc = np.cumsum(dGam[::-1], axis=0)[::-1] + dGC[None, :] + np.cumsum(kdk, axis=0) - kdk
                else:
                    dgc = np.cumsum(dGam[::-1], axis=0)[::-1] + dGC[None, :]
                inter["dDelta"][(n, h, c0)] = dDelta.copy()
                dqt[bi, c0:c1, h] = dQt_c
                dkh[bi, c0:c1, h] = dKh_c
                dv[bi, c0:c1, h] = dVc
                dbeta[bi, c0:c1, h] = dbe
                dg[bi, c0:c1, h] = dgc
                dS = dS0
            dh0[n, h] = dS
    dqs = dqt.reshape(B, T, H_qk, G, K).sum(3)
    dks = dkh.reshape(B, T, H_qk, G, K).sum(3)
    rq, rk = 1.0 / nq, 1.0 / nk
    dq = sc * rq * (dqs - rq * rq * qq * (qq * dqs).sum(-1, keepdims=True))
    dk = rk * (dks - rk * rk * kk * (kk * dks).sum(-1, keepdims=True))
    sig = 1.0 / (1.0 + np.exp(-gg))
    dgraw = dg * (-a[None, None, :, None]) * sig
    dA_log = (dg * g_all).sum(axis=(0, 1, 3))
    db = dbeta * beta_all * (1.0 - beta_all)
    out = dict(dq=dq, dk=dk, dv=dv, dgraw=dgraw, db=db, dA_log=dA_log, dh0=dh0)
    grads = {n_: torch.from_numpy(np.ascontiguousarray(x)) for n_, x in out.items()}
    return (grads, inter) if return_intermediates else grads


def chunk_bwd_inputs(inp, do, dht=None, **kw):
    """``chunk_bwd`` on a ``kda_inputs.KdaInputs``."""
    return chunk_bwd(inp.q, inp.k, inp.v, inp.graw, inp.b, inp.A_log, inp.scale, inp.initial_state,
                     inp.cu_seqlens, do=do, dht=dht, **kw)
