"""fp64 CPU oracle for the KDA forward pass and the single-token decode step.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may use this package; the CUDA library and its
Python binding never import it, and it imports nothing from them.  Only the
seeded input generators in ``kda_inputs`` are shared.

Contents
--------
* ``fwd`` / ``decode``: the token-by-token fp64 recurrence in plain C
  (``kda_oracle.c``), threaded over (sequence, value head).
* ``brute_force``: a NumPy fp64 twin for short sequences that forms each
  step's K x K transition matrix explicitly (a different formulation of the
  same recurrence).
* ``prologue``: the per-token pre-processing in NumPy fp64 (L2 norm, scale,
  sigmoid, gate), used by the two NumPy formulations.
* ``la_fwd`` / ``la_decode``: lightning attention (linear attention with a
  fixed per-head decay), the token recurrence in plain C (``la_oracle.c``).
* ``la_quadratic``: the same method in its parallel (attention-matrix) form in
  NumPy fp64, a second formulation that pins the recurrence.
* ``la_chunk_model``: the chunked lightning-attention algebra in NumPy fp64
  with the kernel's operand roundings on request (its precision study).
* ``chunk_bwd_model``: the same gradients from the chunked (UT/WY) formulas, the
  algebra a tensor-core backward builds on, pinned to ``backward.bwd``.
* ``backward.bwd``: gradients of the KDA forward with respect to all inputs
  (fp64 autograd through the token recurrence), pinned by finite differences
  of ``brute_force``.

The recurrence (KDA, the method the page "FlashKDA: High-performance KDA CUDA
kernels for SM90+ GPUs" implements; gate, sigmoid and L2-norm fusion under its
"Technical Features") per sequence and value head h, state S in R^{V x K}:
``S_t = S_{t-1} Diag(exp g_t)(I - beta_t k_t k_t^T) + beta_t v_t k_t^T``,
``o_t = S_t q_t`` with unit-norm k, q scaled by ``scale`` after its L2 norm,
``beta = sigmoid(b)`` and ``g = -exp(A_log[h]) * softplus(graw)``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Tuple

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "libkda_oracle.so")
_SRC = os.path.join(_HERE, "kda_oracle.c")
_SRCS = [_SRC, os.path.join(_HERE, "la_oracle.c")]
EPS = 1e-6

_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (no fast-math, no FMA contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_SO) or any(os.path.getmtime(_SO) < os.path.getmtime(f) for f in _SRCS):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
                               "-pthread", *_SRCS, "-o", tmp, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_SO)
        P = ctypes.c_void_p
        i = ctypes.c_int
        lib.kda_oracle_fwd.argtypes = [P, P, P, P, P, P, ctypes.c_float, P, P, P,
                                       i, i, i, i, i, i, i, P, i, i]
        lib.kda_oracle_fwd.restype = i
        lib.la_oracle_fwd.argtypes = [P, P, P, P, ctypes.c_float, P, P, P, i, i, i, i, i, i, i, P, i, i]
        lib.la_oracle_fwd.restype = i
        _lib = lib
    return _lib


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def default_threads() -> int:
    return os.cpu_count() or 1


def fwd(q, k, v, graw, b, A_log, scale, initial_state=None, cu_seqlens=None,
        nthreads: Optional[int] = None, mutation: int = 0) -> Tuple[np.ndarray, np.ndarray]:
    """Token-by-token fp64 forward.  Takes the host tensors of a
    ``kda_inputs.KdaInputs`` (bf16 q/k/v/graw/b, fp32 A_log / initial_state,
    int32 cu_seqlens) and returns ``(out [B,T,H_v,V], final [N,H_v,V,K])`` as
    float64 NumPy arrays."""
    lib = _load()
    for t in (q, k, v, graw, b):
        assert t.dtype == torch.bfloat16 and t.device.type == "cpu"
    q, k, v, graw, b = (t.contiguous() for t in (q, k, v, graw, b))
    B, T, H_qk, K = q.shape
    H_v, V = v.shape[2], v.shape[3]
    A_log = A_log.to(torch.float32).contiguous()
    if initial_state is not None:
        initial_state = initial_state.to(torch.float32).contiguous()
    if cu_seqlens is not None:
        cu_seqlens = cu_seqlens.to(torch.int32).cpu().contiguous()
        N = cu_seqlens.numel() - 1
    else:
        N = B
    out = torch.zeros((B, T, H_v, V), dtype=torch.float64)
    final = torch.zeros((N, H_v, V, K), dtype=torch.float64)
    rc = lib.kda_oracle_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(graw), _ptr(b), _ptr(A_log),
                            ctypes.c_float(scale), _ptr(initial_state), _ptr(final),
                            _ptr(cu_seqlens), N, B, T, H_qk, H_v, K, V, _ptr(out),
                            nthreads or default_threads(), mutation)
    if rc != 0:
        raise ValueError(f"kda_oracle_fwd rejected its arguments ({rc})")
    return out.numpy(), final.numpy()


def fwd_inputs(inp, **kw):
    """``fwd`` on a ``kda_inputs.KdaInputs``."""
    return fwd(inp.q, inp.k, inp.v, inp.graw, inp.b, inp.A_log, inp.scale,
               inp.initial_state, inp.cu_seqlens, **kw)


def decode(d, nthreads: Optional[int] = None, mutation: int = 0) -> Tuple[np.ndarray, np.ndarray]:
    """One recurrence step for every (b, h) of a ``kda_inputs.DecodeInputs``:
    the decode step is the forward recurrence over a length-1 sequence whose
    initial state is the given state.  Returns ``(out [B,H_v,V], new_state
    [B,H_v,V,K])`` in float64; the input state is not modified."""
    out, fin = fwd(d.q[:, None], d.k[:, None], d.v[:, None], d.graw[:, None], d.b[:, None],
                   d.A_log, d.scale, d.state, None, nthreads=nthreads, mutation=mutation)
    return out[:, 0], fin


# ---------------------------------------------------------------------------
# NumPy formulations (fp64)
# ---------------------------------------------------------------------------

def _f64(t: torch.Tensor) -> np.ndarray:
    return t.to(torch.float64).numpy()


def prologue(q, k, graw, b, A_log, scale, H_v):
    """Per-token pre-processing in fp64: returns (qt, kh, beta, g) with
    qt, kh ``[B,T,H_v,K]`` (query/key heads repeated to value heads), beta
    ``[B,T,H_v]`` and g ``[B,T,H_v,K]``."""
    q, k, graw, b = _f64(q), _f64(k), _f64(graw), _f64(b)
    G = H_v // q.shape[2]
    q = np.repeat(q, G, axis=2)
    k = np.repeat(k, G, axis=2)
    qh = q / np.sqrt((q * q).sum(-1, keepdims=True) + EPS)
    kh = k / np.sqrt((k * k).sum(-1, keepdims=True) + EPS)
    qt = np.float64(np.float32(scale)) * qh
    with np.errstate(over="ignore"):
        beta = 1.0 / (1.0 + np.exp(-b))
    sp = np.maximum(graw, 0.0) + np.log1p(np.exp(-np.abs(graw)))
    a = np.exp(_f64(A_log))
    g = -a[None, None, :, None] * sp
    return qt, kh, beta, g


def _segments(inp_B, inp_T, cu):
    if cu is None:
        return [(bi, 0, inp_T) for bi in range(inp_B)]
    c = cu.tolist()
    return [(0, c[i], c[i + 1]) for i in range(len(c) - 1)]


def brute_force(q, k, v, graw, b, A_log, scale, initial_state=None, cu_seqlens=None):
    """Explicit-matrix form: ``M_t = Diag(exp g_t)(I - beta_t kh_t kh_t^T)``
    and ``S_t = S_{t-1} M_t + beta_t v_t kh_t^T``, ``o_t = S_t qt_t``.
    Meant for short sequences (it builds a K x K matrix per token)."""
    B, T, _, K = q.shape
    H_v, V = v.shape[2], v.shape[3]
    qt, kh, beta, g = prologue(q, k, graw, b, A_log, scale, H_v)
    vv = _f64(v)
    segs = _segments(B, T, cu_seqlens)
    out = np.zeros((B, T, H_v, V))
    final = np.zeros((len(segs), H_v, V, K))
    I = np.eye(K)
    for n, (bi, s0, s1) in enumerate(segs):
        for h in range(H_v):
            S = np.zeros((V, K)) if initial_state is None else _f64(initial_state[n, h]).copy()
            for t in range(s0, s1):
                kk = kh[bi, t, h]
                M = np.diag(np.exp(g[bi, t, h])) @ (I - beta[bi, t, h] * np.outer(kk, kk))
                S = S @ M + beta[bi, t, h] * np.outer(vv[bi, t, h], kk)
                out[bi, t, h] = S @ qt[bi, t, h]
            final[n, h] = S
    return out, final


def brute_force_inputs(inp):
    return brute_force(inp.q, inp.k, inp.v, inp.graw, inp.b, inp.A_log, inp.scale,
                       inp.initial_state, inp.cu_seqlens)


# ---------------------------------------------------------------------------
# Lightning attention (fixed per-head decay, no delta rule)
# ---------------------------------------------------------------------------
# The cuLA page ("cuLA benchmark results on GB200") times a lightning-attention
# forward and `la_decode` but prints no formula; the reading here is the
# standard recurrence S_t = lambda_h S_{t-1} + v_t k_t^T, o_t = scale S_t q_t,
# lambda_h = exp(-slope[h]), with raw (unnormalised) q and k.

def la_fwd(q, k, v, slope, scale, initial_state=None, cu_seqlens=None,
           nthreads: Optional[int] = None, mutation: int = 0) -> Tuple[np.ndarray, np.ndarray]:
    """Token-by-token fp64 lightning-attention forward on host tensors (bf16
    q/k/v, fp32 slope / initial_state, int32 cu_seqlens).  Returns
    ``(out [B,T,H_v,V], final [N,H_v,V,K])`` as float64 NumPy arrays."""
    lib = _load()
    for t in (q, k, v):
        assert t.dtype == torch.bfloat16 and t.device.type == "cpu"
    q, k, v = (t.contiguous() for t in (q, k, v))
    B, T, H_qk, K = q.shape
    H_v, V = v.shape[2], v.shape[3]
    slope = slope.to(torch.float32).contiguous()
    if initial_state is not None:
        initial_state = initial_state.to(torch.float32).contiguous()
    if cu_seqlens is not None:
        cu_seqlens = cu_seqlens.to(torch.int32).cpu().contiguous()
        N = cu_seqlens.numel() - 1
    else:
        N = B
    out = torch.zeros((B, T, H_v, V), dtype=torch.float64)
    final = torch.zeros((N, H_v, V, K), dtype=torch.float64)
    rc = lib.la_oracle_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(slope), ctypes.c_float(scale),
                           _ptr(initial_state), _ptr(final), _ptr(cu_seqlens), N, B, T, H_qk, H_v, K, V,
                           _ptr(out), nthreads or default_threads(), mutation)
    if rc != 0:
        raise ValueError(f"la_oracle_fwd rejected its arguments ({rc})")
    return out.numpy(), final.numpy()


def la_fwd_inputs(inp, **kw):
    """``la_fwd`` on a ``kda_inputs.LaInputs``."""
    return la_fwd(inp.q, inp.k, inp.v, inp.slope, inp.scale, inp.initial_state, inp.cu_seqlens, **kw)


def la_decode(d, nthreads: Optional[int] = None, mutation: int = 0) -> Tuple[np.ndarray, np.ndarray]:
    """One lightning-attention step for every (b, h) of a
    ``kda_inputs.LaDecodeInputs``: the forward over a length-1 sequence from
    the given state.  Returns ``(out [B,H_v,V], new_state [B,H_v,V,K])``."""
    out, fin = la_fwd(d.q[:, None], d.k[:, None], d.v[:, None], d.slope, d.scale, d.state, None,
                      nthreads=nthreads, mutation=mutation)
    return out[:, 0], fin


def la_quadratic(q, k, v, slope, scale, initial_state=None, cu_seqlens=None):
    """Parallel form of the same method, per sequence and value head, with t, j
    counted from the sequence start and L its length:
    ``O = scale [ (Q K^T * D) V + diag(lambda^(t+1)) Q S_0^T ]`` with
    ``D[t][j] = lambda^(t-j)`` for j <= t (else 0), and
    ``S_L = lambda^L S_0 + sum_j lambda^(L-1-j) v_j k_j^T``."""
    B, T, H_qk, K = q.shape
    H_v, V = v.shape[2], v.shape[3]
    G = H_v // H_qk
    qq, kk, vv = _f64(q), _f64(k), _f64(v)
    lam = np.exp(-_f64(slope))
    sc = np.float64(np.float32(scale))
    segs = _segments(B, T, cu_seqlens)
    out = np.zeros((B, T, H_v, V))
    final = np.zeros((len(segs), H_v, V, K))
    for n, (bi, s0, s1) in enumerate(segs):
        L = s1 - s0
        t = np.arange(L, dtype=np.float64)
        for h in range(H_v):
            Q, Kt, Vt = qq[bi, s0:s1, h // G], kk[bi, s0:s1, h // G], vv[bi, s0:s1, h]
            S0 = np.zeros((V, K)) if initial_state is None else _f64(initial_state[n, h])
            lag = t[:, None] - t[None, :]
            D = np.where(lag >= 0, lam[h] ** np.maximum(lag, 0.0), 0.0)
            out[bi, s0:s1, h] = sc * (((Q @ Kt.T) * D) @ Vt + (lam[h] ** (t + 1))[:, None] * (Q @ S0.T))
            final[n, h] = lam[h] ** L * S0 + (Vt * (lam[h] ** (L - 1 - t))[:, None]).T @ Kt
    return out, final


def la_quadratic_inputs(inp):
    return la_quadratic(inp.q, inp.k, inp.v, inp.slope, inp.scale, inp.initial_state, inp.cu_seqlens)
