"""GPU parity tests of kda_fwd_bf16_state (initial / final state stored in bf16)
against the fp64 oracle started from the same bf16 state values.

The recurrence runs with an fp32 state as in kda_fwd, so the outputs keep the
forward's tolerances; the final state is rounded to bf16 once (at most 2^-8
relative per element), so its bound is rel-L2 <= 4e-3."""
import numpy as np
import pytest
import torch

import kda_inputs as KI
import oracle
from kda_testutil import OUT_MAX_ABS, OUT_REL_L2, gpu_fwd, head_subset, rel_l2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gated_delta_rule_40_gb300 import kda
    kda.load()
    yield
    assert kda.kda_get_status() == 0


def _run(inp):
    from gated_delta_rule_40_gb300 import kda
    dev = lambda t: None if t is None else t.cuda()  # noqa: E731
    s0 = None if inp.initial_state is None else inp.initial_state.to(torch.bfloat16).cuda()
    out, fin = kda.kda_fwd_bf16_state(dev(inp.q), dev(inp.k), dev(inp.v), dev(inp.graw), dev(inp.b), dev(inp.A_log),
                                      inp.scale, initial_state=s0, cu_seqlens=dev(inp.cu_seqlens))
    torch.cuda.synchronize()
    return out, fin


def _bf16_state(inp):
    if inp.initial_state is not None:   # the oracle starts from the stored bf16 values
        inp.initial_state = inp.initial_state.to(torch.bfloat16).float()
    return inp


def _compare(out, fin, ro, rf):
    o = out.double().cpu().numpy()
    assert rel_l2(o, ro) <= OUT_REL_L2 and np.abs(o - ro).max() <= OUT_MAX_ABS
    f = fin.double().cpu().numpy()
    assert np.isfinite(f).all() and rel_l2(f, rf) <= 4e-3, rel_l2(f, rf)


@pytest.mark.parametrize("B,T,Hq,Hv", [(2, 200, 2, 4), (1, 129, 1, 2), (3, 1, 1, 1)])
def test_bf16_state_ragged(B, T, Hq, Hv):
    inp = _bf16_state(KI.make_inputs(B, T, Hq, Hv, seed=800 + T, with_state=True))
    out, fin = _run(inp)
    _compare(out, fin, *oracle.fwd_inputs(inp))


def test_bf16_state_varlen_and_no_initial_state():
    inp = _bf16_state(KI.make_inputs(1, 300, 1, 2, seed=801, with_state=True, seqlens=[0, 130, 1, 105, 64]))
    out, fin = _run(inp)
    _compare(out, fin, *oracle.fwd_inputs(inp))
    inp = KI.make_inputs(1, 100, 1, 1, seed=802, with_state=False)
    out, fin = _run(inp)
    _compare(out, fin, *oracle.fwd_inputs(inp))


def test_bf16_state_matches_fp32_state_path():
    """From the same (bf16-valued) initial state the outputs equal kda_fwd's bit for bit and
    the final state equals kda_fwd's fp32 final state rounded to bf16."""
    inp = _bf16_state(KI.make_inputs(2, 150, 2, 2, seed=803, with_state=True))
    out, fin = _run(inp)
    o32, f32 = gpu_fwd(inp)
    assert torch.equal(out.cpu(), o32.cpu())
    assert torch.equal(fin.cpu(), f32.to(torch.bfloat16).cpu())


def test_bf16_state_full_size_dense_sampled():
    inp = _bf16_state(KI.workload("dense"))
    out, fin = _run(inp)
    sub = head_subset(inp, [0, 31])
    ro, rf = oracle.fwd_inputs(sub)
    hi = torch.tensor([0, 31], device=out.device)
    _compare(out.index_select(2, hi), fin.index_select(1, hi), ro, rf)
