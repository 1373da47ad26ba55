"""Chunked (UT / WY) formulation of the KDA forward in NumPy fp64.

TEST INFRASTRUCTURE ONLY (see the package docstring).  This is the algebra the
chunked GPU path is designed around, written out plainly so the tests can pin
it against the token-by-token oracle; the GPU code shares nothing with it.

Per sequence, value head and chunk of C rows (positions r = 0..C-1), with the
state S_0 (V x K) entering the chunk, per-channel log decay g and its inclusive
in-chunk prefix sum Gam_r = sum_{s<=r} g_s:

  A[r,j] = beta_r sum_c kh[r,c] kh[j,c] exp(Gam[r,c] - Gam[j,c])   (j < r)
  P[r,j] = sum_c qt[r,c] kh[j,c] exp(Gam[r,c] - Gam[j,c])          (j <= r)
  T      = (I + A)^{-1}                                            (unit lower triangular)
  W      = T diag(beta) (Kh * exp(Gam))        U = T diag(beta) V
  Delta  = U - W S_0^T                          (rows are the per-token delta-rule writes)
  O      = (Qt * exp(Gam)) S_0^T + P Delta
  S_C    = S_0 Diag(exp(Gam_C)) + Delta^T (Kh * exp(Gam_C - Gam))

Derivation: writing the recurrence as S_r = S_{r-1} D_r + delta_r kh_r^T with
delta_r = beta_r (v_r - S_{r-1} D_r kh_r) and unrolling S_{r-1} D_r inside the
chunk gives (I + A) Delta = diag(beta) V - diag(beta) (Kh * exp(Gam)) S_0^T;
the output o_r = S_r qt_r and the carried state follow by substitution.

``exp(Gam_r - Gam_j)`` is never formed from ``exp(Gam_r) * exp(-Gam_j)`` over a
whole chunk (that overflows for strong gates).  The decay matrix is built from
16-row sub-blocks the same way the GPU path builds it: below-diagonal blocks of
block-row i use the reference m_i = Gam[16 i - 1] (both factors <= 1), diagonal
blocks use, per channel, the midpoint of the block's first and last Gam as
reference with both exponents clamped at ``clamp`` (exact unless a channel
decays by more than ``2 * clamp`` nats across the sixteen rows), and the j = r
term uses its exact factor 1.  ``rounding`` optionally rounds named operands to bf16 or tf32
to model a kernel's operand precision.
"""
from __future__ import annotations

from typing import Callable, Dict, Optional

import numpy as np

from . import prologue, _f64, _segments

SUB = 16


def _round_bf16(x: np.ndarray) -> np.ndarray:
    x32 = np.asarray(x, dtype=np.float32)
    u = x32.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    u = ((u + 0x7FFF + lsb) >> 16) << 16
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


def _round_tf32(x: np.ndarray) -> np.ndarray:
    x32 = np.asarray(x, dtype=np.float32)
    u = x32.view(np.uint32).astype(np.uint64)
    lsb = (u >> 13) & 1
    u = ((u + 0xFFF + lsb) >> 13) << 13
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


def _round_f32(x: np.ndarray) -> np.ndarray:
    return np.asarray(x, dtype=np.float32).astype(np.float64)


ROUNDERS: Dict[str, Callable[[np.ndarray], np.ndarray]] = {
    "f64": lambda x: x,
    "f32": _round_f32,
    "tf32": _round_tf32,
    "bf16": _round_bf16,
}


def decay_pairs(Gam: np.ndarray, clamp: float = 85.0):
    """Return E with E[r, j, c] = exp(Gam[r,c] - Gam[j,c]) for j <= r (zero
    above the diagonal), assembled from 16-row sub-blocks with per-block
    reference points as described in the module docstring."""
    C, K = Gam.shape
    E = np.zeros((C, C, K))
    nb = (C + SUB - 1) // SUB
    for i in range(nb):
        r0, r1 = i * SUB, min(C, (i + 1) * SUB)
        if i > 0:
            m = Gam[r0 - 1]
            rowf = np.exp(Gam[r0:r1] - m)            # <= 1
            colf = np.exp(m - Gam[:r0])              # <= 1
            E[r0:r1, :r0] = rowf[:, None, :] * colf[None, :, :]
        mid = 0.5 * (Gam[r0] + Gam[r1 - 1])
        rowf = np.exp(np.minimum(Gam[r0:r1] - mid, clamp))
        colf = np.exp(np.minimum(mid - Gam[r0:r1], clamp))
        blk = rowf[:, None, :] * colf[None, :, :]
        n = r1 - r0
        E[r0:r1, r0:r1] = blk * np.tril(np.ones((n, n)), -1)[:, :, None]
        E[np.arange(r0, r1), np.arange(r0, r1)] = 1.0   # the j = r factor is exactly 1
    return E


def chunk_fwd(q, k, v, graw, b, A_log, scale, initial_state=None, cu_seqlens=None,
              C: int = 64, clamp: float = 85.0, rounding: Optional[Dict[str, str]] = None):
    """Chunked forward.  ``rounding`` maps operand names to a rounding mode
    ("bf16", "tf32", "f32", "f64"): keys are ``ab`` (gated operands of A),
    ``abP`` (gated operands of P), ``T`` / ``TU`` (the inverse as an operand of
    W / of U), ``wkg`` (K*exp(Gam) in W), ``W``, ``U``, ``Qg``, ``Kd``, ``P``,
    ``S`` / ``SO`` (the state as an operand of W S^T / of Qg S^T), ``Delta`` /
    ``DeltaO`` (Delta as an operand of the state update / of P Delta) and ``M``
    (the A matrix entries)."""
    rnd = {key: ROUNDERS[mode] for key, mode in (rounding or {}).items()}
    R = lambda name, x: rnd[name](x) if name in rnd else x
    B, T_, _, K = q.shape
    H_v, V = v.shape[2], v.shape[3]
    qt, kh, beta, g = prologue(q, k, graw, b, A_log, scale, H_v)
    vv = _f64(v)
    segs = _segments(B, T_, cu_seqlens)
    out = np.zeros((B, T_, H_v, V))
    final = np.zeros((len(segs), H_v, V, K))
    for n, (bi, s0, s1) in enumerate(segs):
        for h in range(H_v):
            S = np.zeros((V, K)) if initial_state is None else _f64(initial_state[n, h]).copy()
            for c0 in range(s0, s1, C):
                L = min(C, s1 - c0)
                # padded rows: q = k = v = 0, beta = 0, g = 0
                Qt = np.zeros((C, K)); Kh = np.zeros((C, K)); Vc = np.zeros((C, V))
                be = np.zeros(C); gg = np.zeros((C, K))
                Qt[:L] = qt[bi, c0:c0 + L, h]; Kh[:L] = kh[bi, c0:c0 + L, h]
                Vc[:L] = vv[bi, c0:c0 + L, h]; be[:L] = beta[bi, c0:c0 + L, h]
                gg[:L] = g[bi, c0:c0 + L, h]
                Gam = np.cumsum(gg, axis=0)
                E = decay_pairs(Gam, clamp)
                Ka, Qa, Kp = R("ab", Kh), R("abP", Qt), R("abP", Kh)
                Akk = np.einsum("rc,jc,rjc->rj", Ka, Ka, E)
                Akk = np.tril(Akk, -1) * be[:, None]
                Akk = R("M", Akk)
                Pm = np.tril(np.einsum("rc,jc,rjc->rj", Qa, Kp, E))
                Tinv = np.linalg.inv(np.eye(C) + Akk)
                eG = np.exp(Gam)
                Tb = R("T", Tinv * be[None, :])
                W = R("W", Tb @ R("wkg", Kh * eG))
                U = R("U", R("TU", Tinv * be[None, :]) @ Vc)
                Qg = R("Qg", Qt * eG)
                Kd = R("Kd", Kh * np.exp(Gam[-1][None, :] - Gam))
                Sop = R("S", S)
                Delta = U - W @ Sop.T
                Dop = R("Delta", Delta)
                O = Qg @ R("SO", S).T + R("P", Pm) @ R("DeltaO", Delta)
                S = S * np.exp(Gam[-1])[None, :] + Dop.T @ Kd
                out[bi, c0:c0 + L, h] = O[:L]
            final[n, h] = S
    return out, final


def chunk_fwd_inputs(inp, **kw):
    return chunk_fwd(inp.q, inp.k, inp.v, inp.graw, inp.b, inp.A_log, inp.scale,
                     inp.initial_state, inp.cu_seqlens, **kw)
