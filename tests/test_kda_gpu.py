"""GPU parity tests: libkda (through its C ABI) against the fp64 oracle."""
import math

import numpy as np
import pytest
import torch

import kda_inputs as KI
import oracle
from kda_testutil import gpu_fwd, head_subset, parity, to_dev, rel_l2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gated_delta_rule_40_gb300 import kda
    kda.load()
    yield
    assert kda.kda_get_status() == 0


def _check_full(inp, **kw):
    out, fin = gpu_fwd(inp, **kw)
    ro, rf = oracle.fwd_inputs(inp)
    pr = parity(out, fin, ro, rf)
    assert pr.ok(), f"{inp.name}: {pr}"
    return out, fin


# ---------------------------------------------------------------- small cases, full oracle
def test_tiny_workload():
    """B=1, T=256, H_qk=H_v=2, no initial state, seed 0."""
    _check_full(KI.workload("tiny"))


@pytest.mark.parametrize("B,T,Hq,Hv", [(2, 200, 2, 4), (1, 64, 1, 1), (1, 65, 1, 2), (3, 1, 2, 2),
                                       (1, 129, 4, 4), (2, 63, 1, 3)])
def test_ragged_lengths(B, T, Hq, Hv):
    _check_full(KI.make_inputs(B, T, Hq, Hv, seed=100 + T, with_state=True, name=f"ragged{B}x{T}"))


def test_varlen_with_empty_and_single_token_sequences():
    lens = [0, 1, 64, 65, 0, 130, 7, 200]
    inp = KI.make_inputs(1, sum(lens), 2, 4, seed=101, with_state=True, seqlens=lens, name="varlen-edge")
    _check_full(inp)


def test_varlen_without_initial_state():
    lens = [33, 1, 190]
    _check_full(KI.make_inputs(1, sum(lens), 1, 2, seed=102, with_state=False, seqlens=lens, name="varlen-nostate"))


def test_harsh_gates():
    _check_full(KI.make_inputs(1, 320, 1, 2, seed=103, with_state=True, graw_mean=3.0, A_log_value=1.0,
                               name="harsh"))


def test_slow_gates():
    _check_full(KI.make_inputs(1, 640, 1, 2, seed=104, with_state=True, graw_mean=-4.0, A_log_value=-1.0,
                               name="slow"))


def test_scalar_gate_gva():
    inp = KI.make_inputs(1, 300, 2, 8, seed=105, with_state=True, seqlens=[229, 71], scalar_gate=True,
                         name="gdn-gva-small")
    _check_full(inp)


def test_passthrough_keeps_state():
    """beta = 0, g = 0: the state passes through unchanged."""
    inp = KI.make_inputs(1, 300, 1, 2, seed=106, with_state=True, name="passthrough")
    inp.graw.fill_(float("-inf"))
    inp.b.fill_(float("-inf"))
    out, fin = _check_full(inp)
    assert torch.equal(fin.cpu(), inp.initial_state)


def test_full_forget():
    inp = KI.make_inputs(1, 150, 1, 1, seed=107, with_state=True, name="forget")
    inp.graw.fill_(1e4)
    inp.b.fill_(float("inf"))
    _check_full(inp)


def test_zero_tokens_copies_state():
    inp = KI.make_inputs(2, 0, 1, 2, seed=108, with_state=True)
    out, fin = gpu_fwd(inp)
    assert out.shape == (2, 0, 2, 128)
    assert torch.equal(fin.cpu(), inp.initial_state)


def test_no_final_state_and_workspace_path():
    from gated_delta_rule_40_gb300 import kda
    inp = KI.make_inputs(1, 260, 2, 2, seed=109, with_state=True, seqlens=[100, 160])
    out_a, fin_a = gpu_fwd(inp)
    d = to_dev(inp)
    nbytes = kda.kda_fwd_workspace_size(2, 1, 260, 2, 2)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    out_b, fin_b = kda.kda_fwd(d["q"], d["k"], d["v"], d["graw"], d["b"], d["A_log"], d["scale"],
                               initial_state=d["initial_state"], cu_seqlens=d["cu_seqlens"], workspace=ws)
    out_c, fin_c = kda.kda_fwd(d["q"], d["k"], d["v"], d["graw"], d["b"], d["A_log"], d["scale"],
                               initial_state=d["initial_state"], cu_seqlens=d["cu_seqlens"],
                               output_final_state=False)
    torch.cuda.synchronize()
    assert fin_c is None
    assert torch.equal(out_a, out_b) and torch.equal(fin_a, fin_b) and torch.equal(out_a, out_c)


def test_workspace_pool_keeps_and_releases_memory():
    """The allocating entry keeps its workspace mapped in the library's pool across a
    synchronisation (free device memory stays lower by at least the workspace), the
    release entry hands it back, and calls before and after the release agree bit for bit."""
    from gated_delta_rule_40_gb300 import kda
    inp = KI.make_inputs(1, 4096, 2, 8, seed=111, with_state=True)
    d = to_dev(inp)
    need = kda.kda_fwd_workspace_size(1, 1, 4096, 2, 8)
    assert need > 32 << 20

    def call():
        return kda.kda_fwd(d["q"], d["k"], d["v"], d["graw"], d["b"], d["A_log"], d["scale"],
                           initial_state=d["initial_state"])

    kda.kda_release_cached_memory()
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    out_a, fin_a = call()
    torch.cuda.synchronize()
    free1 = torch.cuda.mem_get_info()[0]
    # outputs (4 MiB + 4 MiB) come from torch's caching allocator, the workspace from the pool
    assert free0 - free1 >= need
    kda.kda_release_cached_memory()
    free2 = torch.cuda.mem_get_info()[0]
    assert free2 - free1 >= need
    out_b, fin_b = call()
    torch.cuda.synchronize()
    assert torch.equal(out_a, out_b) and torch.equal(fin_a, fin_b)
    assert kda.kda_get_status() == 0


def test_split_call_equals_single_call():
    inp = KI.make_inputs(1, 400, 1, 2, seed=110, with_state=True)
    out, fin = gpu_fwd(inp)
    t = 173
    sl = lambda x, a, b: x[:, a:b].contiguous()
    first = KI.KdaInputs(q=sl(inp.q, 0, t), k=sl(inp.k, 0, t), v=sl(inp.v, 0, t), graw=sl(inp.graw, 0, t),
                         b=sl(inp.b, 0, t), A_log=inp.A_log, scale=inp.scale,
                         initial_state=inp.initial_state, cu_seqlens=None)
    o1, f1 = gpu_fwd(first)
    second = KI.KdaInputs(q=sl(inp.q, t, 400), k=sl(inp.k, t, 400), v=sl(inp.v, t, 400),
                          graw=sl(inp.graw, t, 400), b=sl(inp.b, t, 400), A_log=inp.A_log, scale=inp.scale,
                          initial_state=f1.cpu(), cu_seqlens=None)
    o2, f2 = gpu_fwd(second)
    both = torch.cat([o1, o2], 1).double().cpu().numpy()
    assert rel_l2(both, out.double().cpu().numpy()) < 5e-3
    assert rel_l2(f2.double().cpu().numpy(), fin.double().cpu().numpy()) < 1e-3


def test_varlen_equals_separate_calls():
    lens = [70, 1, 129]
    inp = KI.make_inputs(1, sum(lens), 1, 2, seed=111, with_state=True, seqlens=lens)
    out, fin = gpu_fwd(inp)
    c = inp.cu_seqlens.tolist()
    for n in range(len(lens)):
        s = lambda x: x[:, c[n]:c[n + 1]].contiguous()
        one = KI.KdaInputs(q=s(inp.q), k=s(inp.k), v=s(inp.v), graw=s(inp.graw), b=s(inp.b), A_log=inp.A_log,
                           scale=inp.scale, initial_state=inp.initial_state[n:n + 1].contiguous(), cu_seqlens=None)
        o, f = gpu_fwd(one)
        assert torch.equal(o[0], out[0, c[n]:c[n + 1]])
        assert torch.equal(f[0], fin[n])


def test_bad_cu_seqlens_sets_status():
    from gated_delta_rule_40_gb300 import kda
    inp = KI.make_inputs(1, 100, 1, 1, seed=112, with_state=True, seqlens=[50, 50])
    inp.cu_seqlens = torch.tensor([0, 60, 50], dtype=torch.int32)   # decreasing, ends at T
    gpu_fwd(inp)
    assert kda.kda_get_status() == kda.KDA_ERR_BAD_SEQLENS
    assert kda.kda_get_status() == 0


def test_misaligned_output_rejected():
    from gated_delta_rule_40_gb300 import kda
    inp = KI.make_inputs(1, 10, 1, 1, seed=113, with_state=False)
    d = to_dev(inp)
    buf = torch.empty(10 * 128 + 1, dtype=torch.bfloat16, device="cuda")
    bad_out = buf[1:].view(1, 10, 1, 128)
    with pytest.raises(kda.KdaError) as e:
        kda.kda_fwd(d["q"], d["k"], d["v"], d["graw"], d["b"], d["A_log"], d["scale"], out=bad_out)
    assert e.value.code == kda.KDA_ERR_INVALID_ARG


# ---------------------------------------------------------------- full-size workloads, sampled heads
@pytest.mark.parametrize("name,qk_heads", [("dense", [0, 13, 31]), ("varlen", [2, 29]), ("gva", [0, 9])])
def test_full_size_workload_sampled(name, qk_heads):
    """Full-size call (the launch configuration the benchmark times); the
    oracle recomputes every (sequence, value head) chain of a few heads."""
    inp = KI.workload(name)
    out, fin = gpu_fwd(inp)
    sub = head_subset(inp, qk_heads)
    ro, rf = oracle.fwd_inputs(sub)
    vh = torch.tensor(sub.meta["v_heads"], device=out.device)
    pr = parity(out.index_select(2, vh), fin.index_select(1, vh), ro, rf)
    assert pr.ok(), f"{name}: {pr}"


# ---------------------------------------------------------------- decode
DECODE_STATE_REL_L2 = 1e-5


def _decode_gpu(d):
    from gated_delta_rule_40_gb300 import kda
    st = d.state.cuda()
    out = kda.kda_decode_step(d.q.cuda(), d.k.cuda(), d.v.cuda(), d.graw.cuda(), d.b.cuda(), d.A_log.cuda(),
                              d.scale, st)
    torch.cuda.synchronize()
    return out, st


@pytest.mark.parametrize("B,H,Hq", [(256, 64, 64), (1, 64, 64), (4, 64, 64), (16, 64, 64), (64, 64, 64),
                                    (3, 8, 2)])
def test_decode_matches_oracle(B, H, Hq):
    d = KI.decode_inputs(B=B, H=H, H_qk=Hq, seed=7 + B)
    out, st = _decode_gpu(d)
    ro, rs = oracle.decode(d)
    pr = parity(out, st, ro, rs)
    assert pr.ok(), f"decode B={B}: {pr}"
    # the step runs in fp32 end to end (one fp32 update per state element), so the state
    # agrees with the fp64 oracle to a few fp32 roundings, not just the forward's bound
    assert pr.state_rel <= DECODE_STATE_REL_L2, f"decode B={B}: {pr}"


def test_decode_equals_fwd_t1():
    d = KI.decode_inputs(B=5, H=4, H_qk=2, seed=5)
    out_d, st_d = _decode_gpu(d)
    inp = KI.KdaInputs(q=d.q[:, None].contiguous(), k=d.k[:, None].contiguous(), v=d.v[:, None].contiguous(),
                       graw=d.graw[:, None].contiguous(), b=d.b[:, None].contiguous(), A_log=d.A_log,
                       scale=d.scale, initial_state=d.state, cu_seqlens=None)
    out_f, fin_f = gpu_fwd(inp)
    assert rel_l2(out_d.double().cpu().numpy(), out_f[:, 0].double().cpu().numpy()) < 5e-3
    assert rel_l2(st_d.double().cpu().numpy(), fin_f.double().cpu().numpy()) < 1e-3


# ---------------------------------------------------------------- device-side failure path
def test_bounded_wait_reports_timeout_and_context_survives():
    """A bounded wait on a barrier that nothing completes gives up, records
    KDA_ERR_DEVICE_TIMEOUT in the status word and returns; reading the status clears it
    and the next forward on the same context is still exact against the oracle."""
    from gated_delta_rule_40_gb300 import kda
    assert kda.kda_get_status() == 0
    kda.kda_selftest_wait_timeout()
    assert kda.kda_get_status() == kda.KDA_ERR_DEVICE_TIMEOUT
    assert kda.kda_get_status() == 0
    _check_full(KI.make_inputs(1, 130, 1, 2, seed=77, with_state=True, name="after-timeout"))
