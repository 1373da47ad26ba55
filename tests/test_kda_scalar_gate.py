"""GPU parity tests of kda_fwd_scalar_gate (one gate value per token and value
head) against the fp64 oracle, which takes the same gate broadcast along K."""
import pytest
import torch

import kda_inputs as KI
import oracle
from kda_testutil import head_subset, parity, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gated_delta_rule_40_gb300 import kda
    kda.load()
    yield
    assert kda.kda_get_status() == 0


def _scalar(inp, **kw):
    """The scalar-gate call on inputs whose graw is constant along K."""
    from gated_delta_rule_40_gb300 import kda
    g = inp.graw[..., 0]
    assert torch.equal(inp.graw, g[..., None].expand_as(inp.graw)), "graw must be constant along K"
    d = to_dev(inp)
    out, fin = kda.kda_fwd_scalar_gate(d["q"], d["k"], d["v"], g.contiguous().cuda(), d["b"], d["A_log"], d["scale"],
                                       initial_state=d["initial_state"], cu_seqlens=d["cu_seqlens"], **kw)
    torch.cuda.synchronize()
    return out, fin


def _check(inp, **kw):
    out, fin = _scalar(inp, **kw)
    ro, rf = oracle.fwd_inputs(inp)
    pr = parity(out, fin, ro, rf)
    assert pr.ok(), f"{inp.name}: {pr}"
    return out, fin


@pytest.mark.parametrize("B,T,Hq,Hv", [(1, 256, 2, 2), (2, 200, 2, 4), (1, 65, 1, 2), (3, 1, 2, 2), (1, 129, 4, 8)])
def test_scalar_gate_ragged(B, T, Hq, Hv):
    _check(KI.make_inputs(B, T, Hq, Hv, seed=401 + T, with_state=True, scalar_gate=True, name="sg"))


def test_scalar_gate_varlen_with_empty_sequences():
    _check(KI.make_inputs(1, 300, 2, 4, seed=402, with_state=True, seqlens=[0, 130, 1, 0, 105, 64],
                          scalar_gate=True, name="sg-varlen"))


def test_scalar_gate_harsh_and_slow():
    _check(KI.make_inputs(1, 320, 1, 2, seed=403, with_state=True, scalar_gate=True, graw_mean=3.0,
                          A_log_value=1.0, name="sg-harsh"))
    _check(KI.make_inputs(1, 640, 1, 2, seed=404, with_state=True, scalar_gate=True, graw_mean=-4.0,
                          A_log_value=-1.0, name="sg-slow"))


def test_scalar_gate_passthrough_and_forget():
    inp = KI.make_inputs(1, 300, 1, 2, seed=405, with_state=True, scalar_gate=True, name="sg-pass")
    inp.graw.fill_(float("-inf"))
    inp.b.fill_(float("-inf"))
    _, fin = _check(inp)
    assert torch.equal(fin.cpu(), inp.initial_state)
    inp = KI.make_inputs(1, 150, 1, 1, seed=406, with_state=True, scalar_gate=True, name="sg-forget")
    inp.graw.fill_(1e4)
    inp.b.fill_(float("inf"))
    _check(inp)


def test_scalar_gate_zero_tokens_and_no_final_state():
    inp = KI.make_inputs(2, 0, 1, 2, seed=407, with_state=True, scalar_gate=True)
    out, fin = _scalar(inp)
    assert out.shape == (2, 0, 2, 128)
    assert torch.equal(fin.cpu(), inp.initial_state)
    inp = KI.make_inputs(1, 200, 1, 1, seed=408, with_state=False, scalar_gate=True)
    out, fin = _scalar(inp, output_final_state=False)
    assert fin is None
    ro, _ = oracle.fwd_inputs(inp)
    assert parity(out, None, ro, None).ok()


def test_scalar_gate_full_size_gva_sampled():
    """The grouped-value-head workload (two sequences of 28672 and 4096 tokens, H_qk=16,
    H_v=64) at full size; the oracle recomputes every chain of two q/k head groups."""
    inp = KI.workload("gva")
    out, fin = _scalar(inp)
    sub = head_subset(inp, [0, 11])
    ro, rf = oracle.fwd_inputs(sub)
    vh = torch.tensor(sub.meta["v_heads"], device=out.device)
    pr = parity(out.index_select(2, vh), fin.index_select(1, vh), ro, rf)
    assert pr.ok(), str(pr)
