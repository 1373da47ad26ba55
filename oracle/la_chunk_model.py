"""Chunked formulation of the lightning-attention forward in NumPy fp64.

TEST INFRASTRUCTURE ONLY (see the package docstring).  This is the algebra the
chunked GPU kernel is designed around, written out plainly so the tests can pin
it against the token recurrence, and with optional rounding of the operands the
kernel keeps in bf16, so the tests can check its precision choices.  The GPU
code shares nothing with it.

Per sequence and value head (lambda = exp(-slope)), for a chunk of len <= C rows
entering with state S_0 (V x K), with Gam_r = -(r + 1) slope:

  O[r] = scale [ exp(Gam_r) S_0 q_r + sum_{j <= r} exp(Gam_r - Gam_j) (q_r . k_j) v_j ]
  S_C  = exp(Gam_len) S_0 + sum_r v_r (k_r exp(Gam_len - Gam_r))^T

obtained by unrolling S_t = lambda S_{t-1} + v_t k_t^T inside the chunk.

``rounding`` names operands to round to bf16 the way the kernel stores them:
``"S"`` (the state copy the output product reads), ``"P"`` (the masked, decayed
and scaled q.k matrix), ``"Kd"`` (k exp(Gam_len - Gam_r) as one bf16 term) or
``"Kd_split"`` (the same as a bf16 value plus its bf16 remainder, the kernel's
choice).
"""
from __future__ import annotations

from typing import Iterable, Optional

import numpy as np

from . import _f64, _segments


def _bf16(x: np.ndarray) -> np.ndarray:
    """Round to bf16 (nearest even) and back to fp64."""
    f = np.asarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


def la_chunk_fwd(q, k, v, slope, scale, initial_state=None, cu_seqlens=None, C: int = 64,
                 rounding: Optional[Iterable[str]] = None):
    """Chunked lightning-attention forward; returns ``(out, final)`` like
    ``oracle.la_fwd``."""
    rnd = set(rounding or ())
    B, T, H_qk, K = q.shape
    H_v, V = v.shape[2], v.shape[3]
    G = H_v // H_qk
    qq, kk, vv = _f64(q), _f64(k), _f64(v)
    sl = _f64(slope)
    sc = np.float64(np.float32(scale))
    segs = _segments(B, T, cu_seqlens)
    out = np.zeros((B, T, H_v, V))
    final = np.zeros((len(segs), H_v, V, K))
    for n, (bi, s0, s1) in enumerate(segs):
        for h in range(H_v):
            S = np.zeros((V, K)) if initial_state is None else _f64(initial_state[n, h]).copy()
            for c0 in range(s0, s1, C):
                ln = min(C, s1 - c0)
                Q, Kc, Vc = qq[bi, c0:c0 + ln, h // G], kk[bi, c0:c0 + ln, h // G], vv[bi, c0:c0 + ln, h]
                r = np.arange(ln, dtype=np.float64)
                gam = -(r + 1) * sl[h]
                lag = r[:, None] - r[None, :]
                D = np.where(lag >= 0, np.exp(-sl[h] * np.maximum(lag, 0.0)), 0.0)
                P = sc * (Q @ Kc.T) * D
                if "P" in rnd:
                    P = _bf16(P)
                Sm = _bf16(S) if "S" in rnd else S
                out[bi, c0:c0 + ln, h] = sc * np.exp(gam)[:, None] * (Q @ Sm.T) + P @ Vc
                Kd = Kc * np.exp(gam[-1] - gam)[:, None]
                if "Kd" in rnd:
                    Kd = _bf16(Kd)
                elif "Kd_split" in rnd:
                    hi = _bf16(Kd)
                    Kd = hi + _bf16(Kd - hi)
                S = np.exp(gam[-1]) * S + Vc.T @ Kd
            final[n, h] = S
    return out, final


def la_chunk_fwd_inputs(inp, **kw):
    return la_chunk_fwd(inp.q, inp.k, inp.v, inp.slope, inp.scale, inp.initial_state, inp.cu_seqlens, **kw)
