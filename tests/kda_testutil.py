"""Helpers for the GPU parity tests: move seeded inputs to the device, call
libkda through its binding, and compare against the fp64 oracle with the
tolerances of the method's accuracy target (out: relative L2 <= 5e-3 and
max-abs <= 3e-2 over the whole tensor; final state: relative L2 <= 1e-3)."""
from __future__ import annotations

from dataclasses import dataclass
from typing import List, Optional, Sequence

import numpy as np
import torch

import kda_inputs as KI

OUT_REL_L2 = 5e-3
OUT_MAX_ABS = 3e-2
STATE_REL_L2 = 1e-3


def to_dev(inp: KI.KdaInputs, dev="cuda") -> dict:
    d = dict(q=inp.q.to(dev), k=inp.k.to(dev), v=inp.v.to(dev), graw=inp.graw.to(dev), b=inp.b.to(dev),
             A_log=inp.A_log.to(dev), scale=inp.scale,
             initial_state=None if inp.initial_state is None else inp.initial_state.to(dev),
             cu_seqlens=None if inp.cu_seqlens is None else inp.cu_seqlens.to(dev))
    return d


def gpu_fwd(inp: KI.KdaInputs, **kw):
    from gated_delta_rule_40_gb300 import kda
    d = to_dev(inp)
    out, fin = kda.kda_fwd(d["q"], d["k"], d["v"], d["graw"], d["b"], d["A_log"], d["scale"],
                           initial_state=d["initial_state"], cu_seqlens=d["cu_seqlens"], **kw)
    torch.cuda.synchronize()
    return out, fin


def rel_l2(a: np.ndarray, ref: np.ndarray) -> float:
    n = np.linalg.norm(ref)
    return float(np.linalg.norm(a - ref) / n) if n > 0 else float(np.linalg.norm(a - ref))


@dataclass
class Parity:
    out_rel: float
    out_max: float
    state_rel: float

    def ok(self) -> bool:
        return self.out_rel <= OUT_REL_L2 and self.out_max <= OUT_MAX_ABS and self.state_rel <= STATE_REL_L2

    def __str__(self):
        return f"out rel-L2 {self.out_rel:.3e} max-abs {self.out_max:.3e} state rel-L2 {self.state_rel:.3e}"


def parity(out_gpu: torch.Tensor, fin_gpu: Optional[torch.Tensor], out_ref: np.ndarray,
           fin_ref: Optional[np.ndarray]) -> Parity:
    o = out_gpu.double().cpu().numpy()
    assert o.shape == out_ref.shape, (o.shape, out_ref.shape)
    assert np.isfinite(o).all(), "non-finite output"
    out_rel = rel_l2(o, out_ref) if o.size else 0.0
    out_max = float(np.abs(o - out_ref).max()) if o.size else 0.0
    st = 0.0
    if fin_gpu is not None and fin_ref is not None:
        f = fin_gpu.double().cpu().numpy()
        assert np.isfinite(f).all(), "non-finite state"
        st = rel_l2(f, fin_ref)
    return Parity(out_rel, out_max, st)


def head_subset(inp: KI.KdaInputs, qk_heads: Sequence[int]) -> KI.KdaInputs:
    """The sub-problem made of the given query/key heads and all value heads
    that read them (each (sequence, value head) chain is independent, so the
    sub-problem's outputs equal the corresponding slices of the full one)."""
    G = inp.H_v // inp.H_qk
    vh: List[int] = [hq * G + j for hq in qk_heads for j in range(G)]
    qi = torch.tensor(list(qk_heads))
    vi = torch.tensor(vh)
    return KI.KdaInputs(
        q=inp.q.index_select(2, qi).contiguous(), k=inp.k.index_select(2, qi).contiguous(),
        v=inp.v.index_select(2, vi).contiguous(), graw=inp.graw.index_select(2, vi).contiguous(),
        b=inp.b.index_select(2, vi).contiguous(), A_log=inp.A_log.index_select(0, vi).contiguous(),
        scale=inp.scale,
        initial_state=None if inp.initial_state is None else inp.initial_state.index_select(1, vi).contiguous(),
        cu_seqlens=inp.cu_seqlens, name=inp.name + "-sub", meta=dict(v_heads=vh))
