"""Pins that tie the fp64 oracle to facts fixed by the mathematics of the KDA
recurrence rather than to the oracle itself.

Each pin takes a forward callable with the signature of ``oracle.fwd`` and
returns the largest violation it found (0 means exact agreement); ``PINS``
lists them with their tolerances.  The tests run every pin on the oracle and,
with one deliberate mistake planted in the C oracle at a time, check that some
pin fails (so a dropped term, a wrong sign, a transposed state or a wrong
index cannot pass unnoticed).
"""
from __future__ import annotations

import math

import numpy as np
import torch

import kda_inputs as KI
import oracle

NEG_INF = float("-inf")
POS_INF = float("inf")


def _bf(x) -> torch.Tensor:
    return torch.as_tensor(x, dtype=torch.float32).to(torch.bfloat16)


def _f64(t):
    return t.to(torch.float64).numpy()


def _unit(x: np.ndarray) -> np.ndarray:
    return x / np.sqrt((x * x).sum(-1, keepdims=True) + oracle.EPS)


def _run(fwd, inp: KI.KdaInputs, **over):
    d = dict(q=inp.q, k=inp.k, v=inp.v, graw=inp.graw, b=inp.b, A_log=inp.A_log,
             scale=inp.scale, initial_state=inp.initial_state, cu_seqlens=inp.cu_seqlens)
    d.update(over)
    return fwd(d["q"], d["k"], d["v"], d["graw"], d["b"], d["A_log"], d["scale"],
               d["initial_state"], d["cu_seqlens"])


def pin_t1_zero_state(fwd) -> float:
    """T=1 from a zero state: S_1 = beta v kh^T, so o = beta (kh . qt) v."""
    inp = KI.make_inputs(3, 1, 2, 4, seed=11, with_state=False)
    out, fin = _run(fwd, inp)
    G = 2
    qt = np.float32(inp.scale) * _unit(np.repeat(_f64(inp.q), G, 2))
    kh = _unit(np.repeat(_f64(inp.k), G, 2))
    beta = 1.0 / (1.0 + np.exp(-_f64(inp.b)))
    v = _f64(inp.v)
    ref_o = beta[..., None] * (kh * qt).sum(-1, keepdims=True) * v
    ref_S = beta[:, 0, :, None, None] * v[:, 0, :, :, None] * kh[:, 0, :, None, :]
    return max(np.abs(out - ref_o).max() / np.abs(ref_o).max(), np.abs(fin - ref_S).max() / np.abs(ref_S).max())


def pin_passthrough(fwd) -> float:
    """beta = 0 (b = -inf) and g = 0 (graw = -inf): the state never changes,
    o_t = S_0 qt_t and the final state equals the initial state."""
    inp = KI.make_inputs(2, 40, 2, 2, seed=12, with_state=True)
    graw = torch.full_like(inp.graw, NEG_INF)
    b = torch.full_like(inp.b, NEG_INF)
    out, fin = _run(fwd, inp, graw=graw, b=b)
    qt = np.float32(inp.scale) * _unit(_f64(inp.q))
    S0 = _f64(inp.initial_state)
    ref_o = np.einsum("bhvk,bthk->bthv", S0, qt)
    return max(np.abs(out - ref_o).max() / np.abs(ref_o).max(), np.abs(fin - S0).max())


def pin_linear_attention(fwd) -> float:
    """beta = 1, g = 0 and mutually orthogonal keys (Hadamard rows): the erase
    term vanishes and the layer is causal linear attention,
    o_t = sum_{j<=t} v_j (kh_j . qt_t)."""
    T = 48
    Hm = KI.hadamard(128)
    inp = KI.make_inputs(1, T, 1, 1, seed=13, with_state=False)
    k = _bf(Hm[torch.randperm(128, generator=torch.Generator().manual_seed(3))[:T]].reshape(1, T, 1, 128).float())
    graw = torch.full_like(inp.graw, NEG_INF)
    b = torch.full_like(inp.b, POS_INF)
    out, fin = _run(fwd, inp, k=k, graw=graw, b=b)
    qt = np.float32(inp.scale) * _unit(_f64(inp.q))[0, :, 0]
    kh = _unit(_f64(k))[0, :, 0]
    v = _f64(inp.v)[0, :, 0]
    sc = np.tril(qt @ kh.T)
    ref = sc @ v
    return np.abs(out[0, :, 0] - ref).max() / np.abs(ref).max()


def pin_full_forget(fwd) -> float:
    """graw = 1e4 makes exp(g) underflow to 0 and b = +inf gives beta = 1, so
    each token overwrites the state: o_t = (kh_t . qt_t) v_t and the final
    state is v_T kh_T^T."""
    inp = KI.make_inputs(1, 24, 2, 2, seed=14, with_state=True)
    graw = torch.full_like(inp.graw, 1e4)
    b = torch.full_like(inp.b, POS_INF)
    out, fin = _run(fwd, inp, graw=graw, b=b)
    qt = np.float32(inp.scale) * _unit(_f64(inp.q))
    kh = _unit(_f64(inp.k))
    v = _f64(inp.v)
    ref_o = (kh * qt).sum(-1, keepdims=True) * v
    ref_S = v[0, -1, :, :, None] * kh[0, -1, :, None, :]
    return max(np.abs(out - ref_o).max() / np.abs(ref_o).max(), np.abs(fin[0] - ref_S).max())


def pin_gate_special_values(fwd) -> float:
    """beta = 0, one token: the final state is S_0 Diag(exp g).  With A_log = 0
    a channel with graw = 0 has g = -softplus(0) = -ln 2 (decay exactly 1/2), a
    channel with graw = -inf has g = 0 (decay 1) and graw = 30 gives
    g = -(30 + log1p(e^-30)).  The channel pattern is asymmetric so a reversed
    channel index shows."""
    inp = KI.make_inputs(1, 1, 1, 1, seed=15, with_state=True)
    pat = torch.full((128,), NEG_INF)
    pat[0:40] = 0.0
    pat[100:103] = 30.0
    graw = _bf(pat).reshape(1, 1, 1, 128)
    b = torch.full_like(inp.b, NEG_INF)
    A_log = torch.zeros(1)
    _, fin = _run(fwd, inp, graw=graw, b=b, A_log=A_log)
    dec = np.ones(128)
    dec[0:40] = 0.5
    dec[100:103] = math.exp(-30.0) * math.exp(-math.log1p(math.exp(-30.0)))
    ref = _f64(inp.initial_state)[0, 0] * dec[None, :]
    return np.abs(fin[0, 0] - ref).max() / np.abs(ref).max()


def pin_repeated_key_overwrite(fwd) -> float:
    """beta = 1, g = 0 and the same key at every step, from a zero state: the
    delta rule replaces the value stored under that key, so after token t the
    state is v_t kh^T and o_t = (kh . qt_t) v_t (up to the norm's epsilon)."""
    T = 6
    inp = KI.make_inputs(1, T, 1, 1, seed=22, with_state=False)
    k = inp.k[:, :1].expand(1, T, 1, 128).contiguous()
    graw = torch.full_like(inp.graw, NEG_INF)
    b = torch.full_like(inp.b, POS_INF)
    out, fin = _run(fwd, inp, k=k, graw=graw, b=b)
    qt = np.float32(inp.scale) * _unit(_f64(inp.q))[0, :, 0]
    kh = _unit(_f64(k))[0, 0, 0]
    v = _f64(inp.v)[0, :, 0]
    ref = (qt @ kh)[:, None] * v
    return np.abs(out[0, :, 0] - ref).max() / np.abs(ref).max()


def pin_bruteforce(fwd) -> float:
    """Agreement with the explicit K x K transition-matrix form on short
    packed sequences with an initial state and grouped value heads."""
    inp = KI.make_inputs(1, 14, 2, 4, seed=16, with_state=True, seqlens=[5, 9])
    out, fin = _run(fwd, inp)
    ro, rf = oracle.brute_force_inputs(inp)
    return max(np.abs(out - ro).max() / np.abs(ro).max(), np.abs(fin - rf).max() / np.abs(rf).max())


def pin_split_invariance(fwd) -> float:
    """Running x[:t] then x[t:] from the first call's final state equals one
    call over x (t on and off a multiple of 64)."""
    inp = KI.make_inputs(2, 150, 1, 2, seed=17, with_state=True)
    out, fin = _run(fwd, inp)
    worst = 0.0
    for t in (64, 77):
        sl = lambda x, a, b_: x[:, a:b_].contiguous()
        o1, f1 = _run(fwd, inp, q=sl(inp.q, 0, t), k=sl(inp.k, 0, t), v=sl(inp.v, 0, t),
                      graw=sl(inp.graw, 0, t), b=sl(inp.b, 0, t))
        o2, f2 = _run(fwd, inp, q=sl(inp.q, t, 150), k=sl(inp.k, t, 150), v=sl(inp.v, t, 150),
                      graw=sl(inp.graw, t, 150), b=sl(inp.b, t, 150),
                      initial_state=torch.from_numpy(f1).float())
        # the handed-over state is rounded to fp32, as a caller's would be
        worst = max(worst, np.abs(np.concatenate([o1, o2], 1) - out).max() / np.abs(out).max(),
                    np.abs(f2 - fin).max() / np.abs(fin).max())
    return worst


def pin_varlen_invariance(fwd) -> float:
    """A packed call equals independent per-sequence calls."""
    lens = [7, 64, 1, 90]
    inp = KI.make_inputs(1, sum(lens), 2, 2, seed=18, with_state=True, seqlens=lens)
    out, fin = _run(fwd, inp)
    worst = 0.0
    c = inp.cu_seqlens.tolist()
    for n in range(len(lens)):
        s = lambda x: x[:, c[n]:c[n + 1]].contiguous()
        o, f = _run(fwd, inp, q=s(inp.q), k=s(inp.k), v=s(inp.v), graw=s(inp.graw), b=s(inp.b),
                    initial_state=inp.initial_state[n:n + 1].contiguous(), cu_seqlens=None)
        worst = max(worst, np.abs(o - out[:, c[n]:c[n + 1]]).max(), np.abs(f[0] - fin[n]).max())
    return worst


def pin_gva_repeat(fwd) -> float:
    """Grouped value heads equal the ungrouped call with each query/key head
    repeated for its group of value heads (head h uses q/k head h // G)."""
    inp = KI.make_inputs(1, 30, 2, 6, seed=19, with_state=True)
    out, fin = _run(fwd, inp)
    rep = lambda x: x.repeat_interleave(3, dim=2).contiguous()
    o2, f2 = _run(fwd, inp, q=rep(inp.q), k=rep(inp.k))
    return max(np.abs(out - o2).max(), np.abs(fin - f2).max())


def pin_scale_invariance(fwd) -> float:
    """Multiplying q or k by a power of two is exact in bf16 and cancels in the
    L2 norm (up to the norm's epsilon, far below the tolerance used)."""
    inp = KI.make_inputs(1, 40, 1, 1, seed=20, with_state=True)
    out, fin = _run(fwd, inp)
    o2, f2 = _run(fwd, inp, q=(inp.q.float() * 8).to(torch.bfloat16), k=(inp.k.float() * 0.25).to(torch.bfloat16))
    return max(np.abs(out - o2).max() / np.abs(out).max(), np.abs(fin - f2).max() / np.abs(fin).max())


def pin_stability_bound(fwd) -> float:
    """Diag(exp g) and (I - beta k k^T) are contractions for unit k and
    beta in [0, 1], so ||S_t||_2 <= ||S_{t-1}||_2 + beta_t ||v_t||; returns the
    largest relative excess over the bound (0 when it holds)."""
    inp = KI.make_inputs(1, 12, 1, 1, seed=21, with_state=True)
    inp.initial_state.mul_(50.0)
    S = inp.initial_state
    worst = 0.0
    for t in range(12):
        s = lambda x: x[:, t:t + 1].contiguous()
        _, f = _run(fwd, inp, q=s(inp.q), k=s(inp.k), v=s(inp.v), graw=s(inp.graw), b=s(inp.b),
                    initial_state=S)
        beta = 1.0 / (1.0 + math.exp(-float(inp.b[0, t, 0])))
        bound = np.linalg.norm(_f64(S)[0, 0], 2) + beta * np.linalg.norm(_f64(inp.v[0, t, 0]))
        worst = max(worst, (np.linalg.norm(f[0, 0], 2) - bound) / bound)
        S = torch.from_numpy(f).float()
    return max(worst, 0.0)


PINS = [
    (pin_t1_zero_state, 1e-12),
    (pin_passthrough, 1e-12),
    (pin_linear_attention, 1e-7),
    (pin_full_forget, 1e-12),
    (pin_gate_special_values, 1e-12),
    (pin_repeated_key_overwrite, 1e-6),
    (pin_bruteforce, 1e-11),
    (pin_split_invariance, 1e-6),
    (pin_varlen_invariance, 1e-13),
    (pin_gva_repeat, 1e-14),
    (pin_scale_invariance, 1e-6),
    (pin_stability_bound, 1e-9),
]
