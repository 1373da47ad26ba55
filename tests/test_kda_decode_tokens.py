"""GPU parity tests of kda_decode_tokens (Tq tokens per (b, h) in one pass over an
fp32 or bf16 state) against the fp64 oracle run on the same Tq-token sequences.

Tolerances: out as the forward (bf16 output); an fp32 state is computed in fp32
throughout, so it must match to 1e-5 relative; a bf16 state is rounded once to 8
significant bits, a relative error of at most 2^-8 per element, so rel-L2 <= 4e-3."""
import numpy as np
import pytest
import torch

import kda_inputs as KI
import oracle
from kda_testutil import OUT_MAX_ABS, OUT_REL_L2, rel_l2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gated_delta_rule_40_gb300 import kda
    kda.load()
    yield
    assert kda.kda_get_status() == 0


def _run(inp, state_dtype):
    from gated_delta_rule_40_gb300 import kda
    st = inp.initial_state.to(state_dtype).cuda()
    out = kda.kda_decode_tokens(inp.q.cuda(), inp.k.cuda(), inp.v.cuda(), inp.graw.cuda(), inp.b.cuda(),
                                inp.A_log.cuda(), inp.scale, st)
    torch.cuda.synchronize()
    return out, st


def _check(B, Tq, Hq, Hv, state_dtype, seed):
    inp = KI.make_inputs(B, Tq, Hq, Hv, seed=seed, with_state=True)
    if state_dtype == torch.bfloat16:   # the oracle starts from the stored bf16 values
        inp.initial_state = inp.initial_state.to(torch.bfloat16).float()
    out, st = _run(inp, state_dtype)
    ro, rf = oracle.fwd_inputs(inp)
    o = out.double().cpu().numpy()
    assert rel_l2(o, ro) <= OUT_REL_L2 and np.abs(o - ro).max() <= OUT_MAX_ABS
    s = st.double().cpu().numpy()
    assert np.isfinite(s).all()
    bound = 1e-5 if state_dtype == torch.float32 else 4e-3
    assert rel_l2(s, rf) <= bound, rel_l2(s, rf)


@pytest.mark.parametrize("Tq", [1, 2, 4, 8])
@pytest.mark.parametrize("Hq,Hv", [(8, 8), (2, 8)])
def test_decode_tokens_fp32_state(Tq, Hq, Hv):
    _check(4, Tq, Hq, Hv, torch.float32, seed=500 + Tq)


@pytest.mark.parametrize("Tq", [1, 4, 8])
def test_decode_tokens_bf16_state(Tq):
    _check(4, Tq, 4, 8, torch.bfloat16, seed=510 + Tq)


def test_decode_tokens_serving_shape():
    """B=256, H=64 with four tokens per step, fp32 and bf16 state."""
    _check(256, 4, 64, 64, torch.float32, seed=520)
    _check(256, 4, 64, 64, torch.bfloat16, seed=521)


def test_decode_tokens_one_equals_decode_step():
    from gated_delta_rule_40_gb300 import kda
    d = KI.decode_inputs(B=16, H=8, seed=530)
    st1, st2 = d.state.cuda(), d.state.cuda()
    o1 = kda.kda_decode_step(d.q.cuda(), d.k.cuda(), d.v.cuda(), d.graw.cuda(), d.b.cuda(), d.A_log.cuda(),
                             d.scale, st1)
    o2 = kda.kda_decode_tokens(d.q[:, None].cuda(), d.k[:, None].cuda(), d.v[:, None].cuda(), d.graw[:, None].cuda(),
                               d.b[:, None].cuda(), d.A_log.cuda(), d.scale, st2)
    torch.cuda.synchronize()
    assert rel_l2(st2.double().cpu().numpy(), st1.double().cpu().numpy()) <= 1e-6
    assert (o2[:, 0].float() - o1.float()).abs().max().item() <= 1e-2


@pytest.mark.parametrize("Tq", [0, 9])
def test_decode_tokens_rejects_token_count(Tq):
    from gated_delta_rule_40_gb300 import kda
    B, H = 2, 2
    q = torch.zeros((B, Tq, H, 128), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros((B, H, 128, 128), device="cuda")
    b = torch.zeros((B, Tq, H), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(kda.KdaError) as e:
        kda.kda_decode_tokens(q, q, q, q, b, torch.zeros(H, device="cuda"), 0.1, st)
    assert e.value.code == kda.KDA_ERR_INVALID_ARG


def test_decode_steps_replay_from_a_cuda_graph():
    """A serving loop captures its decode step once and replays it: kda_decode_step and
    kda_decode_tokens captured into one CUDA graph (in place on their states) and replayed twice
    equal the same calls made directly, bit for bit."""
    from gated_delta_rule_40_gb300 import kda
    d = KI.decode_inputs(B=8, H=8, H_qk=4, seed=540)
    m = KI.make_inputs(8, 4, 4, 8, seed=541, with_state=True)
    dd = {n: getattr(d, n).cuda() for n in ("q", "k", "v", "graw", "b", "A_log")}
    md = {n: getattr(m, n).cuda() for n in ("q", "k", "v", "graw", "b", "A_log")}
    st1, st2 = d.state.cuda(), m.initial_state.to(torch.bfloat16).cuda()
    r1, r2 = st1.clone(), st2.clone()
    o1 = torch.empty((8, 8, 128), dtype=torch.bfloat16, device="cuda")
    o2 = torch.empty((8, 4, 8, 128), dtype=torch.bfloat16, device="cuda")

    def step(a, b, oa, ob):
        kda.kda_decode_step(dd["q"], dd["k"], dd["v"], dd["graw"], dd["b"], dd["A_log"], d.scale, a, out=oa)
        kda.kda_decode_tokens(md["q"], md["k"], md["v"], md["graw"], md["b"], md["A_log"], m.scale, b, out=ob)

    step(st1, st2, o1, o2)   # warm-up outside the capture
    r1.copy_(st1)
    r2.copy_(st2)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step(st1, st2, o1, o2)
    ro1, ro2 = torch.empty_like(o1), torch.empty_like(o2)
    for _ in range(2):
        g.replay()
        step(r1, r2, ro1, ro2)
        torch.cuda.synchronize()
        assert torch.equal(st1, r1) and torch.equal(st2, r2)
        assert torch.equal(o1, ro1) and torch.equal(o2, ro2)
