"""Seeded synthetic inputs for the KDA forward and decode workloads.

This module is shared by the fp64 oracle (``oracle/``), the tests and the
benchmark.  It draws random numbers and arranges them into the shapes, dtypes
and sequence structure of the workloads; it contains none of the method's
arithmetic (no normalisation, gate, decay or state update).

Workloads (shapes follow the kernel-library benchmark pages: cuLA's KDA tables
on GB200 and FlashQLA's gated-delta-rule tables on H200):

* ``tiny``    B=1, T=256, H_qk=H_v=2, no initial state.
* ``dense``   B=2, T=16384, H_qk=H_v=32, initial state ~ N(0, 0.02).
* ``varlen``  20 packed sequences, total T=16384 (one of 8192, the other 19
  log-uniform in [16, 4096] rescaled to sum 8192), H=32.
* ``gva``     packed 28672+4096, H_qk=16, H_v=64, the gate pre-activation
  drawn once per (token, v-head) and repeated along the 128 channels (the
  scalar-decay gated delta rule as a special case of the per-channel gate).
* ``decode``  B=256, H=64, one token, state ~ N(0, 0.02) updated in place.

Lightning attention (linear attention with a fixed per-head decay; shapes from
cuLA's lightning-attention tables, whose head count was lost from the page, and
its ``la_decode`` run with 64 heads of dimension 128):

* ``la_dense``   B=2, T=16384, H=64, q/k/v ~ N(0, 1), initial state ~ N(0, 1).
* ``la_varlen``  20 packed sequences, total T=16380 (one of 8190, the other 19
  log-uniform in [16, 4096] rescaled), H=64.
* ``la_decode``  B=256, H=64, one token, state ~ N(0, 1) updated in place.

The per-head decay rates are the geometric sequence ``2^(-8 (h+1) / H)``
(largest 2^(-8/H), smallest 2^-8): a fixed input pattern, not drawn.  Draw
order: q, k, v, initial_state.

Draw order for one workload: q, k, v, graw, b, A_log, initial_state, all from
one ``torch.Generator`` seeded with ``seed``.  Normal draws are fp32 and then
rounded to bf16 (round-to-nearest-even), so the oracle and the GPU path see
bit-identical bf16 inputs.  Sequence lengths use a second generator seeded with
``seed + 1``.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional

import torch

K_DIM = 128
V_DIM = 128
STATE_STD = 0.02


@dataclass
class KdaInputs:
    """Host (CPU) tensors for one forward call.

    Layouts: q, k ``[B,T,H_qk,K]`` bf16; v ``[B,T,H_v,V]`` bf16; graw
    ``[B,T,H_v,K]`` bf16; b ``[B,T,H_v]`` bf16; A_log ``[H_v]`` fp32;
    initial_state ``[N,H_v,V,K]`` fp32 or None; cu_seqlens ``[N+1]`` int32 or
    None (then N == B sequences of length T).
    """

    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    graw: torch.Tensor
    b: torch.Tensor
    A_log: torch.Tensor
    scale: float
    initial_state: Optional[torch.Tensor]
    cu_seqlens: Optional[torch.Tensor]
    name: str = ""
    meta: dict = field(default_factory=dict)

    @property
    def B(self) -> int:
        return self.q.shape[0]

    @property
    def T(self) -> int:
        return self.q.shape[1]

    @property
    def H_qk(self) -> int:
        return self.q.shape[2]

    @property
    def H_v(self) -> int:
        return self.v.shape[2]

    @property
    def N(self) -> int:
        return self.B if self.cu_seqlens is None else self.cu_seqlens.numel() - 1

    def seqlens(self) -> List[int]:
        if self.cu_seqlens is None:
            return [self.T] * self.B
        c = self.cu_seqlens.tolist()
        return [c[i + 1] - c[i] for i in range(len(c) - 1)]

    def token_heads(self) -> int:
        return self.B * self.T * self.H_v


def _bf16_normal(g: torch.Generator, shape, mean: float = 0.0, std: float = 1.0) -> torch.Tensor:
    x = torch.randn(shape, generator=g, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    if mean != 0.0:
        x.add_(mean)
    return x.to(torch.bfloat16)


def skewed_seqlens(total: int, n: int, long_len: int, lo: int, hi: int, seed: int) -> List[int]:
    """One sequence of ``long_len`` plus ``n-1`` log-uniform lengths in
    [lo, hi] rescaled (floor, remainder to the largest, minimum 1) so that all
    lengths sum to ``total``; the order is shuffled with the same generator."""
    g = torch.Generator().manual_seed(seed)
    rest_total = total - long_len
    u = torch.rand(n - 1, generator=g, dtype=torch.float64)
    raw = torch.exp(math.log(lo) + u * (math.log(hi) - math.log(lo)))
    scaled = raw * (rest_total / raw.sum())
    lens = [max(1, int(math.floor(x))) for x in scaled.tolist()]
    diff = rest_total - sum(lens)
    imax = max(range(len(lens)), key=lambda i: lens[i])
    lens[imax] += diff
    assert all(x >= 1 for x in lens) and sum(lens) == rest_total
    lens = [long_len] + lens
    perm = torch.randperm(n, generator=g).tolist()
    return [lens[i] for i in perm]


def make_inputs(B: int, T: int, H_qk: int, H_v: int, *, seed: int = 0,
                with_state: bool = True, seqlens: Optional[List[int]] = None,
                scalar_gate: bool = False, graw_mean: float = 0.0,
                graw_std: float = 1.0, A_log_value: Optional[float] = None,
                name: str = "") -> KdaInputs:
    """Draw one forward problem.  With ``seqlens`` the call is packed: B must
    be 1 and T == sum(seqlens)."""
    if seqlens is not None:
        assert B == 1 and T == sum(seqlens)
        cu = torch.tensor([0] + list(torch.cumsum(torch.tensor(seqlens), 0).tolist()),
                          dtype=torch.int32)
        n_seq = len(seqlens)
    else:
        cu = None
        n_seq = B
    g = torch.Generator().manual_seed(seed)
    q = _bf16_normal(g, (B, T, H_qk, K_DIM))
    k = _bf16_normal(g, (B, T, H_qk, K_DIM))
    v = _bf16_normal(g, (B, T, H_v, V_DIM))
    if scalar_gate:
        graw = _bf16_normal(g, (B, T, H_v, 1), graw_mean, graw_std).expand(B, T, H_v, K_DIM).contiguous()
    else:
        graw = _bf16_normal(g, (B, T, H_v, K_DIM), graw_mean, graw_std)
    b = _bf16_normal(g, (B, T, H_v))
    A_log = torch.rand(H_v, generator=g, dtype=torch.float32) * 2.0 - 1.0
    if A_log_value is not None:
        A_log.fill_(A_log_value)
    init = None
    if with_state:
        init = torch.randn((n_seq, H_v, V_DIM, K_DIM), generator=g, dtype=torch.float32) * STATE_STD
    return KdaInputs(q=q, k=k, v=v, graw=graw, b=b, A_log=A_log,
                     scale=1.0 / math.sqrt(K_DIM), initial_state=init,
                     cu_seqlens=cu, name=name)


def workload(name: str, seed: int = 0, **over) -> KdaInputs:
    """The named forward workloads (see module docstring)."""
    if name == "tiny":
        return make_inputs(1, 256, 2, 2, seed=seed, with_state=False, name=name, **over)
    if name == "dense":
        B = over.pop("B", 2)
        T = over.pop("T", 16384)
        H = over.pop("H", 32)
        return make_inputs(B, T, H, H, seed=seed, with_state=True, name=name, **over)
    if name == "varlen":
        lens = skewed_seqlens(16384, 20, 8192, 16, 4096, seed + 1)
        inp = make_inputs(1, 16384, 32, 32, seed=seed, with_state=True, seqlens=lens, name=name, **over)
        return inp
    if name == "gva":
        return make_inputs(1, 32768, 16, 64, seed=seed, with_state=True,
                           seqlens=[28672, 4096], scalar_gate=True, name=name, **over)
    raise KeyError(name)


@dataclass
class DecodeInputs:
    """One single-token step: q, k ``[B,H_qk,K]``; v ``[B,H_v,V]``; graw
    ``[B,H_v,K]``; b ``[B,H_v]`` (bf16); A_log ``[H_v]`` fp32; state
    ``[B,H_v,V,K]`` fp32 (updated in place by the step)."""

    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    graw: torch.Tensor
    b: torch.Tensor
    A_log: torch.Tensor
    scale: float
    state: torch.Tensor

    @property
    def B(self) -> int:
        return self.q.shape[0]

    @property
    def H_qk(self) -> int:
        return self.q.shape[1]

    @property
    def H_v(self) -> int:
        return self.v.shape[1]


def decode_inputs(B: int = 256, H: int = 64, *, H_qk: Optional[int] = None, seed: int = 0) -> DecodeInputs:
    H_qk = H if H_qk is None else H_qk
    g = torch.Generator().manual_seed(seed)
    q = _bf16_normal(g, (B, H_qk, K_DIM))
    k = _bf16_normal(g, (B, H_qk, K_DIM))
    v = _bf16_normal(g, (B, H, V_DIM))
    graw = _bf16_normal(g, (B, H, K_DIM))
    b = _bf16_normal(g, (B, H))
    A_log = torch.rand(H, generator=g, dtype=torch.float32) * 2.0 - 1.0
    state = torch.randn((B, H, V_DIM, K_DIM), generator=g, dtype=torch.float32) * STATE_STD
    return DecodeInputs(q=q, k=k, v=v, graw=graw, b=b, A_log=A_log,
                        scale=1.0 / math.sqrt(K_DIM), state=state)


def hadamard(n: int) -> torch.Tensor:
    """Sylvester Hadamard matrix (entries +-1, rows mutually orthogonal);
    exactly representable in bf16, used to build orthogonal key sets."""
    h = torch.ones((1, 1), dtype=torch.float64)
    while h.shape[0] < n:
        h = torch.cat([torch.cat([h, h], 1), torch.cat([h, -h], 1)], 0)
    assert h.shape[0] == n
    return h


# ---------------------------------------------------------------------------
# Lightning attention inputs
# ---------------------------------------------------------------------------
LA_STATE_STD = 1.0


def geometric_slopes(H: int) -> torch.Tensor:
    """Per-head decay rates 2^(-8 (h+1) / H), h = 0..H-1 (fp32)."""
    return torch.tensor([2.0 ** (-8.0 * (h + 1) / H) for h in range(H)], dtype=torch.float32)


@dataclass
class LaInputs:
    """Host tensors for one lightning-attention forward: q, k ``[B,T,H_qk,K]``
    bf16; v ``[B,T,H_v,V]`` bf16; slope ``[H_v]`` fp32; initial_state
    ``[N,H_v,V,K]`` fp32 or None; cu_seqlens ``[N+1]`` int32 or None."""

    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    slope: torch.Tensor
    scale: float
    initial_state: Optional[torch.Tensor]
    cu_seqlens: Optional[torch.Tensor]
    name: str = ""

    @property
    def B(self) -> int:
        return self.q.shape[0]

    @property
    def T(self) -> int:
        return self.q.shape[1]

    @property
    def H_qk(self) -> int:
        return self.q.shape[2]

    @property
    def H_v(self) -> int:
        return self.v.shape[2]

    @property
    def N(self) -> int:
        return self.B if self.cu_seqlens is None else self.cu_seqlens.numel() - 1

    def seqlens(self) -> List[int]:
        if self.cu_seqlens is None:
            return [self.T] * self.B
        c = self.cu_seqlens.tolist()
        return [c[i + 1] - c[i] for i in range(len(c) - 1)]

    def token_heads(self) -> int:
        return self.B * self.T * self.H_v


def make_la_inputs(B: int, T: int, H_qk: int, H_v: int, *, seed: int = 0, with_state: bool = True,
                   seqlens: Optional[List[int]] = None, slope: Optional[torch.Tensor] = None,
                   name: str = "") -> LaInputs:
    """Draw one lightning-attention forward problem (packed when ``seqlens``
    is given: B must be 1 and T == sum(seqlens))."""
    if seqlens is not None:
        assert B == 1 and T == sum(seqlens)
        cu = torch.tensor([0] + list(torch.cumsum(torch.tensor(seqlens), 0).tolist()), dtype=torch.int32)
        n_seq = len(seqlens)
    else:
        cu = None
        n_seq = B
    g = torch.Generator().manual_seed(seed)
    q = _bf16_normal(g, (B, T, H_qk, K_DIM))
    k = _bf16_normal(g, (B, T, H_qk, K_DIM))
    v = _bf16_normal(g, (B, T, H_v, V_DIM))
    init = None
    if with_state:
        init = torch.randn((n_seq, H_v, V_DIM, K_DIM), generator=g, dtype=torch.float32) * LA_STATE_STD
    return LaInputs(q=q, k=k, v=v, slope=geometric_slopes(H_v) if slope is None else slope.to(torch.float32),
                    scale=1.0 / math.sqrt(K_DIM), initial_state=init, cu_seqlens=cu, name=name)


def la_workload(name: str, seed: int = 0) -> LaInputs:
    """The named lightning-attention forward workloads (module docstring)."""
    if name == "la_dense":
        return make_la_inputs(2, 16384, 64, 64, seed=seed, name=name)
    if name == "la_varlen":
        lens = skewed_seqlens(16380, 20, 8190, 16, 4096, seed + 1)
        return make_la_inputs(1, 16380, 64, 64, seed=seed, seqlens=lens, name=name)
    raise KeyError(name)


@dataclass
class LaDecodeInputs:
    """One lightning-attention step: q, k ``[B,H_qk,K]``, v ``[B,H_v,V]`` bf16;
    slope ``[H_v]`` fp32; state ``[B,H_v,V,K]`` fp32 (updated in place)."""

    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    slope: torch.Tensor
    scale: float
    state: torch.Tensor

    @property
    def B(self) -> int:
        return self.q.shape[0]

    @property
    def H_v(self) -> int:
        return self.v.shape[1]


def la_decode_inputs(B: int = 256, H: int = 64, *, H_qk: Optional[int] = None, seed: int = 0) -> LaDecodeInputs:
    H_qk = H if H_qk is None else H_qk
    g = torch.Generator().manual_seed(seed)
    q = _bf16_normal(g, (B, H_qk, K_DIM))
    k = _bf16_normal(g, (B, H_qk, K_DIM))
    v = _bf16_normal(g, (B, H, V_DIM))
    state = torch.randn((B, H, V_DIM, K_DIM), generator=g, dtype=torch.float32) * LA_STATE_STD
    return LaDecodeInputs(q=q, k=k, v=v, slope=geometric_slopes(H), scale=1.0 / math.sqrt(K_DIM), state=state)
