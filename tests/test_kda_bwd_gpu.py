"""GPU parity tests of kda_bwd (the backward of the KDA forward) against the
fp64 autograd oracle, through the C ABI.

The GPU computes the chunked (UT / WY) backward on tensor cores with tf32
operands rounded to nearest and fp32 accumulation, so the gradients differ from
the fp64 oracle by the operands' roundings (a few 1e-4 relative): each gradient
tensor must match to relative L2 <= 1e-3 and max-abs <= 1e-2 of its largest
reference magnitude.  dA_log is a sum over tokens and channels of dg * g whose
terms cancel (by 50 to 200 fold on these inputs), so its error is bounded
relative to the sum of the terms' magnitudes, sum |dg g| (per value head),
which the reference's dgraw gives: dg g = dgraw softplus(graw) / sigmoid(graw)."""
import numpy as np
import pytest
import torch

import kda_inputs as KI
from oracle import backward as OB
from kda_testutil import rel_l2

pytestmark = pytest.mark.gpu

REL = 1e-3
MAX_FRAC = 1e-2
DALOG_FRAC = 1e-4   # |dA_log - ref| per head, relative to sum |dg g| of that head


def _dalog_scale(inp, dgraw_ref):
    """sum over tokens and channels of |dg g| per value head, from the reference dgraw."""
    gr = inp.graw.double().numpy()
    sp = np.maximum(gr, 0.0) + np.log1p(np.exp(-np.abs(gr)))
    sig = 1.0 / (1.0 + np.exp(-gr))
    return np.abs(np.asarray(dgraw_ref) * sp / sig).sum(axis=(0, 1, 3))


def _check_dalog(inp, got, ref, tag=""):
    scale = _dalog_scale(inp, ref["dgraw"])
    err = np.abs(got - ref["dA_log"])
    assert (err <= DALOG_FRAC * scale + 1e-30).all(), f"{tag}dA_log: error {err} vs sum|dg g| {scale}"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gated_delta_rule_40_gb300 import kda
    kda.load()
    yield
    assert kda.kda_get_status() == 0


def _grads(inp, seed, with_dht=True):
    g = torch.Generator().manual_seed(seed)
    do = torch.randn(inp.v.shape, generator=g).to(torch.bfloat16)
    dht = torch.randn((inp.N, inp.H_v, 128, 128), generator=g) * 0.1 if with_dht else None
    return do, dht


def _run_raw(inp, do, dht):
    from gated_delta_rule_40_gb300 import kda
    dev = lambda t: None if t is None else t.cuda()  # noqa: E731
    got = kda.kda_bwd(dev(inp.q), dev(inp.k), dev(inp.v), dev(inp.graw), dev(inp.b), dev(inp.A_log), inp.scale,
                      dev(do), initial_state=dev(inp.initial_state), cu_seqlens=dev(inp.cu_seqlens), dht=dev(dht))
    torch.cuda.synchronize()
    return got


def _run(inp, do, dht):
    return {k_: v_.double().cpu().numpy() for k_, v_ in _run_raw(inp, do, dht).items()}


def _check(inp, seed, with_dht=True):
    do, dht = _grads(inp, seed, with_dht)
    got = _run(inp, do, dht)
    ref = {k_: v_.numpy() for k_, v_ in OB.bwd_inputs(inp, do, dht).items()}
    _check_dalog(inp, got["dA_log"], ref)
    for name in ("dq", "dk", "dv", "dgraw", "db", "dh0"):
        a, r = got[name], ref[name]
        assert a.shape == r.shape, (name, a.shape, r.shape)
        assert np.isfinite(a).all(), name
        if r.size == 0 or not np.abs(r).max() > 0:
            assert np.abs(a).max() <= 1e-6 if a.size else True, name
            continue
        e = rel_l2(a, r)
        m = np.abs(a - r).max() / np.abs(r).max()
        assert e <= REL and m <= MAX_FRAC, f"{name}: rel-L2 {e:.2e}, max {m:.2e}"


@pytest.mark.parametrize("B,T,Hq,Hv", [(1, 100, 1, 2), (2, 70, 2, 2), (1, 129, 2, 4), (3, 1, 1, 1)])
def test_bwd_ragged(B, T, Hq, Hv):
    _check(KI.make_inputs(B, T, Hq, Hv, seed=700 + T, with_state=True), seed=1)


def test_bwd_varlen_with_empty_sequences():
    _check(KI.make_inputs(1, 200, 1, 2, seed=701, with_state=True, seqlens=[0, 65, 1, 0, 70, 64]), seed=2)


def test_bwd_no_state_no_dht_and_harsh_gate():
    _check(KI.make_inputs(1, 150, 1, 1, seed=702, with_state=False), seed=3, with_dht=False)
    _check(KI.make_inputs(1, 130, 1, 1, seed=703, with_state=True, graw_mean=3.0, A_log_value=1.0), seed=4)


def test_bwd_zero_tokens_passes_dht():
    inp = KI.make_inputs(2, 0, 1, 2, seed=704, with_state=True)
    do, dht = _grads(inp, 5)
    got = _run(inp, do, dht)
    assert np.array_equal(got["dh0"], dht.double().numpy())
    assert np.abs(got["dA_log"]).max() == 0.0


def test_bwd_longer_sequence():
    """T = 1024 (16 chunks): both state chains over many chunks."""
    _check(KI.make_inputs(1, 1024, 1, 1, seed=705, with_state=True), seed=6)


@pytest.mark.parametrize("name,qk_heads", [("dense", [0, 31]), ("varlen", [5]), ("gva", [3])])
def test_bwd_full_size_sampled_heads(name, qk_heads):
    """The workloads at full size (dense B=2 T=16384 H=32, the skewed 20-sequence varlen
    packing, grouped value heads 16/64 over 28672+4096 tokens); the fp64 reverse-pass oracle
    (checkpointed, pinned to autograd) recomputes every gradient of a few q/k heads and the
    value heads that read them (each chain is independent)."""
    from gated_delta_rule_40_gb300 import kda
    from kda_testutil import head_subset
    inp = KI.workload(name)
    do, dht = _grads(inp, 7)
    dev = lambda t: None if t is None else t.cuda()  # noqa: E731
    got = kda.kda_bwd(dev(inp.q), dev(inp.k), dev(inp.v), dev(inp.graw), dev(inp.b), dev(inp.A_log), inp.scale,
                      dev(do), initial_state=dev(inp.initial_state), cu_seqlens=dev(inp.cu_seqlens), dht=dev(dht))
    torch.cuda.synchronize()
    G = inp.H_v // inp.H_qk
    sub = head_subset(inp, qk_heads)
    vh = torch.tensor(sub.meta["v_heads"])
    qh = torch.tensor(qk_heads)
    ref = OB.bwd_recurrent_inputs(sub, do.index_select(2, vh).contiguous(),
                                  None if dht is None else dht.index_select(1, vh).contiguous())
    sel = {"dq": got["dq"].index_select(2, qh.cuda()), "dk": got["dk"].index_select(2, qh.cuda()),
           "dv": got["dv"].index_select(2, vh.cuda()), "dgraw": got["dgraw"].index_select(2, vh.cuda()),
           "db": got["db"].index_select(2, vh.cuda()), "dA_log": got["dA_log"].index_select(0, vh.cuda()),
           "dh0": got["dh0"].index_select(1, vh.cuda())}
    refn = {k_: v_.numpy() for k_, v_ in ref.items()}
    _check_dalog(sub, sel["dA_log"].double().cpu().numpy(), refn, f"{name} ")
    for n_, a in sel.items():
        if n_ == "dA_log":
            continue
        a = a.double().cpu().numpy()
        r = refn[n_]
        e = rel_l2(a, r)
        m = np.abs(a - r).max() / max(np.abs(r).max(), 1e-30)
        assert e <= REL and m <= MAX_FRAC, f"{name} {n_} (group {G}): rel-L2 {e:.2e}, max {m:.2e}"


def test_bwd_large_value_head_group():
    """20 value heads share one q/k head (more than the 16 the Jacobian kernel keeps dA_log
    partials for in registers): dq and dk sum over all 20, dA_log per head."""
    _check(KI.make_inputs(1, 40, 1, 20, seed=706, with_state=True), seed=8)


def test_bwd_allocating_entry_equals_workspace_entry():
    """kda_bwd (workspace from cudaMallocAsync) and kda_bwd_ws (the binding's default, a
    torch buffer) run the same kernels: bit-identical gradients."""
    import ctypes
    from gated_delta_rule_40_gb300 import kda
    inp = KI.make_inputs(1, 150, 1, 2, seed=709, with_state=True, seqlens=[90, 60])
    do, dht = _grads(inp, 9)
    got = {k_: v_ for k_, v_ in _run_raw(inp, do, dht).items()}
    lib = kda.load()
    d = {n: (None if t is None else t.cuda()) for n, t in (("q", inp.q), ("k", inp.k), ("v", inp.v), ("g", inp.graw),
                                                          ("b", inp.b), ("a", inp.A_log), ("s", inp.initial_state),
                                                          ("cu", inp.cu_seqlens), ("do", do), ("dht", dht))}
    out = {n: torch.empty_like(t) for n, t in got.items()}
    p = lambda t: ctypes.c_void_p(0 if t is None else t.data_ptr())  # noqa: E731
    rc = lib.kda_bwd(p(d["q"]), p(d["k"]), p(d["v"]), p(d["g"]), p(d["b"]), p(d["a"]), ctypes.c_float(inp.scale),
                     p(d["s"]), p(d["cu"]), 2, 1, 150, 1, 2, 128, 128, p(d["do"]), p(d["dht"]), p(out["dq"]),
                     p(out["dk"]), p(out["dv"]), p(out["dgraw"]), p(out["db"]), p(out["dA_log"]), p(out["dh0"]),
                     ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == kda.KDA_OK
    torch.cuda.synchronize()
    for name in got:
        assert torch.equal(out[name], got[name]), name
