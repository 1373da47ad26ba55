"""GPU parity tests of lightning attention (kda_la_fwd, kda_la_decode) against
the fp64 oracle, through the C ABI.

Tolerances.  Without normalisation the outputs grow with the decay window
(|o| reaches ~40 on these inputs), so the output bounds are relative: rel-L2
<= 5e-3 over the tensor and max-abs <= 1e-2 of the largest reference
magnitude.  bf16 rounding of the output alone is 2^-9 relative; the bf16 copy
of the state and of Q exp(Gam) in the output product and the bf16 P matrix add
errors of the same order.  The final state is fp32 with the decayed values
split into two bf16 terms, so rel-L2 <= 1e-3 (measured errors are ~1e-5).
The decode step is fp32 throughout: state rel-L2 <= 1e-5."""
import numpy as np
import pytest
import torch

import kda_inputs as KI
import oracle
from kda_testutil import rel_l2

pytestmark = pytest.mark.gpu

OUT_REL = 5e-3
OUT_MAX_FRAC = 1e-2
STATE_REL = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gated_delta_rule_40_gb300 import kda
    kda.load()
    yield
    assert kda.kda_get_status() == 0


def _gpu(inp, **kw):
    from gated_delta_rule_40_gb300 import kda
    dev = lambda t: None if t is None else t.cuda()
    out, fin = kda.kda_la_fwd(dev(inp.q), dev(inp.k), dev(inp.v), dev(inp.slope), inp.scale,
                              initial_state=dev(inp.initial_state), cu_seqlens=dev(inp.cu_seqlens), **kw)
    torch.cuda.synchronize()
    return out, fin


def _compare(out, fin, ro, rf):
    o = out.double().cpu().numpy()
    assert np.isfinite(o).all()
    if o.size:
        assert rel_l2(o, ro) <= OUT_REL, rel_l2(o, ro)
        assert np.abs(o - ro).max() <= OUT_MAX_FRAC * max(np.abs(ro).max(), 1.0), np.abs(o - ro).max()
    if fin is not None and rf is not None:
        f = fin.double().cpu().numpy()
        assert np.isfinite(f).all()
        assert rel_l2(f, rf) <= STATE_REL, rel_l2(f, rf)


def _check(inp, **kw):
    out, fin = _gpu(inp, **kw)
    ro, rf = oracle.la_fwd_inputs(inp)
    _compare(out, fin, ro, rf)
    return out, fin


@pytest.mark.parametrize("B,T,Hq,Hv", [(1, 256, 2, 2), (2, 200, 2, 4), (1, 65, 1, 2), (3, 1, 2, 2),
                                       (1, 64, 1, 1), (2, 63, 1, 3), (1, 1000, 1, 2)])
def test_la_ragged(B, T, Hq, Hv):
    _check(KI.make_la_inputs(B, T, Hq, Hv, seed=600 + T))


def test_la_varlen_with_empty_sequences():
    _check(KI.make_la_inputs(1, 400, 2, 4, seed=601, seqlens=[0, 130, 1, 0, 205, 64]))


def test_la_no_initial_state_and_no_final_state():
    inp = KI.make_la_inputs(2, 150, 2, 2, seed=602, with_state=False)
    _check(inp)
    out, fin = _gpu(inp, output_final_state=False)
    assert fin is None
    ro, _ = oracle.la_fwd_inputs(inp)
    _compare(out, None, ro, None)


def test_la_decay_extremes():
    """No decay (slope 0: the state only accumulates) and a fast decay (slope 4:
    lambda^64 underflows to 0 within a chunk)."""
    _check(KI.make_la_inputs(1, 300, 1, 2, seed=603, slope=torch.zeros(2)))
    _check(KI.make_la_inputs(1, 300, 1, 2, seed=604, slope=torch.tensor([4.0, 0.5])))


def test_la_zero_tokens_copies_state():
    inp = KI.make_la_inputs(2, 0, 1, 2, seed=605)
    out, fin = _gpu(inp)
    assert out.shape == (2, 0, 2, 128)
    assert torch.equal(fin.cpu(), inp.initial_state)


def _head_slice(inp, heads):
    """Sub-problem of the given heads (H_qk == H_v): each chain is independent."""
    hi = torch.tensor(heads)
    return KI.LaInputs(q=inp.q.index_select(2, hi).contiguous(), k=inp.k.index_select(2, hi).contiguous(),
                       v=inp.v.index_select(2, hi).contiguous(), slope=inp.slope.index_select(0, hi).contiguous(),
                       scale=inp.scale,
                       initial_state=None if inp.initial_state is None else
                       inp.initial_state.index_select(1, hi).contiguous(),
                       cu_seqlens=inp.cu_seqlens, name=inp.name)


@pytest.mark.parametrize("name", ["la_dense", "la_varlen"])
def test_la_full_size_sampled_heads(name):
    """The benchmark workloads at full size (64 heads); the oracle recomputes the
    fastest- and slowest-decaying heads and one in between."""
    inp = KI.la_workload(name)
    out, fin = _gpu(inp)
    heads = [0, 31, 63]
    sub = _head_slice(inp, heads)
    ro, rf = oracle.la_fwd_inputs(sub)
    hi = torch.tensor(heads, device=out.device)
    _compare(out.index_select(2, hi), fin.index_select(1, hi), ro, rf)


def test_la_decode_small_and_gva():
    from gated_delta_rule_40_gb300 import kda
    for B, H, Hq in [(4, 8, 8), (3, 8, 2)]:
        d = KI.la_decode_inputs(B=B, H=H, H_qk=Hq, seed=610 + B)
        st = d.state.cuda()
        o = kda.kda_la_decode(d.q.cuda(), d.k.cuda(), d.v.cuda(), d.slope.cuda(), d.scale, st)
        torch.cuda.synchronize()
        ro, rs = oracle.la_decode(d)
        assert rel_l2(st.double().cpu().numpy(), rs) <= 1e-5
        assert rel_l2(o.double().cpu().numpy(), ro) <= OUT_REL


def test_la_decode_serving_shape():
    """B=256, H=64 (the la_decode table's largest batch)."""
    from gated_delta_rule_40_gb300 import kda
    d = KI.la_decode_inputs(B=256, H=64, seed=620)
    st = d.state.cuda()
    o = kda.kda_la_decode(d.q.cuda(), d.k.cuda(), d.v.cuda(), d.slope.cuda(), d.scale, st)
    torch.cuda.synchronize()
    ro, rs = oracle.la_decode(d)
    assert rel_l2(st.double().cpu().numpy(), rs) <= 1e-5
    o = o.double().cpu().numpy()
    assert rel_l2(o, ro) <= OUT_REL and np.abs(o - ro).max() <= OUT_MAX_FRAC * np.abs(ro).max()


def test_la_decode_equals_one_token_forward():
    from gated_delta_rule_40_gb300 import kda
    d = KI.la_decode_inputs(B=8, H=4, seed=630)
    st = d.state.cuda()
    o1 = kda.kda_la_decode(d.q.cuda(), d.k.cuda(), d.v.cuda(), d.slope.cuda(), d.scale, st)
    o2, f2 = kda.kda_la_fwd(d.q[:, None].cuda(), d.k[:, None].cuda(), d.v[:, None].cuda(), d.slope.cuda(), d.scale,
                            initial_state=d.state.cuda())
    torch.cuda.synchronize()
    assert rel_l2(f2.double().cpu().numpy(), st.double().cpu().numpy()) <= 1e-5
    assert (o2[:, 0].float() - o1.float()).abs().max().item() <= 1e-2 * o1.float().abs().max().item()


def test_la_rejects_bad_arguments():
    from gated_delta_rule_40_gb300 import kda
    q = torch.zeros((1, 4, 2, 128), dtype=torch.bfloat16, device="cuda")
    v = torch.zeros((1, 4, 3, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(kda.KdaError) as e:
        kda.kda_la_fwd(q, q, v, torch.zeros(3, device="cuda"), 0.1)
    assert e.value.code == kda.KDA_ERR_INVALID_ARG
