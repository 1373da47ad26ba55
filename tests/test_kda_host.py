"""GPU tests of kda_fwd_host (the forward on host buffers, through the C ABI).

The host entry point runs the same kernels as kda_fwd on consecutive token
pieces, cutting sequences at chunk boundaries and carrying their states on the
device, which is the same chunking and arithmetic as one call: its results must
equal kda_fwd's bit for bit.  The first cases also check it against the fp64
oracle at the method's tolerances."""
import pytest
import torch

import kda_inputs as KI
import oracle
from kda_testutil import gpu_fwd, parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gated_delta_rule_40_gb300 import kda
    kda.load()
    yield
    assert kda.kda_get_status() == 0


def _host_fwd(inp, pinned=True, **kw):
    from gated_delta_rule_40_gb300 import kda
    h = (lambda t: None if t is None else t.contiguous().pin_memory()) if pinned else (lambda t: t)
    return kda.kda_fwd_host(h(inp.q), h(inp.k), h(inp.v), h(inp.graw), h(inp.b), h(inp.A_log), inp.scale,
                            initial_state=h(inp.initial_state), cu_seqlens=inp.cu_seqlens, **kw)


def _same(a, b):
    if a is None or b is None:
        assert a is None and b is None
        return
    assert torch.equal(a.cpu(), b.cpu())


@pytest.mark.parametrize("B,T,Hq,Hv", [(2, 300, 2, 4), (1, 129, 4, 4), (3, 64, 1, 2), (1, 1, 4, 8)])
def test_host_equals_device_and_oracle(B, T, Hq, Hv):
    inp = KI.make_inputs(B, T, Hq, Hv, seed=301 + T, with_state=True)
    ho, hf = _host_fwd(inp)
    do, df = gpu_fwd(inp)
    _same(ho, do)
    _same(hf, df)
    ro, rf = oracle.fwd_inputs(inp)
    pr = parity(ho, hf, ro, rf)
    assert pr.ok(), str(pr)


def test_host_varlen_with_empty_sequences():
    inp = KI.make_inputs(1, 400, 4, 4, seed=311, with_state=True, seqlens=[0, 130, 1, 0, 205, 64])
    ho, hf = _host_fwd(inp)
    do, df = gpu_fwd(inp)
    _same(ho, do)
    _same(hf, df)


def test_host_pageable_buffers_and_no_final_state():
    inp = KI.make_inputs(2, 150, 2, 2, seed=312, with_state=False)
    ho, hf = _host_fwd(inp, pinned=False, output_final_state=False)
    do, _ = gpu_fwd(inp, output_final_state=False)
    assert hf is None
    _same(ho, do)


def test_host_zero_tokens_copies_state():
    inp = KI.make_inputs(2, 0, 2, 2, seed=313, with_state=True)
    ho, hf = _host_fwd(inp)
    assert ho.numel() == 0
    _same(hf, inp.initial_state)


def test_host_full_size_dense_equals_device():
    """The benchmark's dense workload (B=2, T=16384, H=32), copied and computed in four token pieces."""
    inp = KI.workload("dense")
    ho, hf = _host_fwd(inp)
    do, df = gpu_fwd(inp)
    _same(ho, do)
    _same(hf, df)


def test_host_varlen_workload_equals_device():
    """The skewed 20-sequence workload (T=16384): pieces cut sequences at chunk boundaries."""
    inp = KI.workload("varlen")
    ho, hf = _host_fwd(inp)
    do, df = gpu_fwd(inp)
    _same(ho, do)
    _same(hf, df)


def test_host_rejects_malformed_cu_seqlens():
    from gated_delta_rule_40_gb300 import kda
    inp = KI.make_inputs(1, 100, 1, 1, seed=314, with_state=False, seqlens=[60, 40])
    bad = torch.tensor([0, 70, 60], dtype=torch.int32)
    with pytest.raises(kda.KdaError) as ei:
        kda.kda_fwd_host(inp.q, inp.k, inp.v, inp.graw, inp.b, inp.A_log, inp.scale, cu_seqlens=bad)
    assert ei.value.code == kda.KDA_ERR_BAD_SEQLENS
