"""The allocation-free forward (kda_fwd_noalloc) against kda_fwd.

kda_fwd_noalloc serves callers that cannot allocate device memory where they
run the forward (under an allocator that owns every byte of device memory and
forbids allocations outside its pool, in serving loops that must never enter
the driver's allocator, in hosts that hand the library only their own
tensors): it uses the library's fixed 64 MiB device array as workspace.  It
runs the same kernels as kda_fwd, so its results must equal kda_fwd's bit for
bit.  This file runs last so that a failure here leaves every other test
already run.
"""
import ctypes

import pytest
import torch

import kda_inputs as KI
from kda_testutil import to_dev

pytestmark = pytest.mark.gpu


def _both(inp):
    from gated_delta_rule_40_gb300 import kda
    d = to_dev(inp)
    args = (d["q"], d["k"], d["v"], d["graw"], d["b"], d["A_log"], d["scale"])
    ref_out, ref_fin = kda.kda_fwd(*args, initial_state=d["initial_state"], cu_seqlens=d["cu_seqlens"])
    out = torch.empty_like(ref_out)
    fin = torch.empty_like(ref_fin)
    kda.kda_fwd_noalloc(*args, initial_state=d["initial_state"], cu_seqlens=d["cu_seqlens"], out=out,
                        final_state=fin)
    torch.cuda.synchronize()
    return ref_out, ref_fin, out, fin


def _rc_for_size(lib, B, T, H):
    """Return code of kda_fwd_noalloc for a problem size with every data pointer NULL:
    KDA_ERR_WORKSPACE when the size exceeds the array (checked before anything else that
    depends on the pointers), KDA_ERR_INVALID_ARG (the NULL inputs) when it fits.  No
    pointer is ever dereferenced and nothing is launched."""
    return lib.kda_fwd_noalloc(None, None, None, None, None, None, ctypes.c_float(0.1), None, None, None, 0, B, T,
                               H, H, 128, 128, None, None)


def test_noalloc_matches_kda_fwd_on_two_calls_in_a_row():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gated_delta_rule_40_gb300 import kda
    first = KI.make_inputs(1, 450, 2, 4, seed=201, with_state=True, seqlens=[100, 37, 250, 63])
    second = KI.make_inputs(2, 300, 1, 2, seed=202, with_state=True)
    for inp in (first, second):
        ref_out, ref_fin, out, fin = _both(inp)
        assert torch.equal(out, ref_out)
        assert torch.equal(fin, ref_fin)
    assert kda.kda_get_status() == 0


def test_noalloc_largest_accepted_size_and_first_rejected_one():
    """Binary search for the longest single sequence (4 value heads) whose workspace fits
    the array, run it (equal to kda_fwd), and check that one more token is rejected."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gated_delta_rule_40_gb300 import kda
    lib = kda.load()
    H = 4
    lo, hi = 1, 1 << 20          # lo fits, hi does not
    assert _rc_for_size(lib, 1, lo, H) == kda.KDA_ERR_INVALID_ARG
    assert _rc_for_size(lib, 1, hi, H) == kda.KDA_ERR_WORKSPACE
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if _rc_for_size(lib, 1, mid, H) == kda.KDA_ERR_WORKSPACE:
            hi = mid
        else:
            lo = mid
    # the array holds the workspace of more than a hundred 64-token chunks of four heads
    assert lo >= 100 * 64 and hi == lo + 1
    inp = KI.make_inputs(1, lo, H, H, seed=203, with_state=True)
    ref_out, ref_fin, out, fin = _both(inp)
    assert torch.equal(out, ref_out)
    assert torch.equal(fin, ref_fin)
    assert kda.kda_get_status() == 0


def test_noalloc_rejects_sizes_beyond_its_array():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gated_delta_rule_40_gb300 import kda
    lib = kda.load()
    # B=2, T=16384, H=32 needs far more workspace than the array holds: rejected before any
    # launch (NULL data pointers, so a regression of the size check fails argument validation
    # instead of touching memory)
    assert _rc_for_size(lib, 2, 16384, 32) == kda.KDA_ERR_WORKSPACE


def test_noalloc_replays_from_a_cuda_graph():
    """One warm-up call (the array's device address), then the allocation-free forward captured
    into a CUDA graph on a small varlen case; two replays on new inputs copied into the captured
    tensors each equal kda_fwd on those inputs bit for bit."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gated_delta_rule_40_gb300 import kda
    lens = [100, 37, 250, 63]
    base = KI.make_inputs(1, sum(lens), 2, 4, seed=211, with_state=True, seqlens=lens)
    d = to_dev(base)
    args = (d["q"], d["k"], d["v"], d["graw"], d["b"], d["A_log"], d["scale"])
    out = torch.empty((1, sum(lens), 4, 128), dtype=torch.bfloat16, device="cuda")
    fin = torch.empty_like(d["initial_state"])
    kda.kda_fwd_noalloc(*args, initial_state=d["initial_state"], cu_seqlens=d["cu_seqlens"], out=out,
                        final_state=fin)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        kda.kda_fwd_noalloc(*args, initial_state=d["initial_state"], cu_seqlens=d["cu_seqlens"], out=out,
                            final_state=fin)
    for seed in (212, 213):
        new = to_dev(KI.make_inputs(1, sum(lens), 2, 4, seed=seed, with_state=True, seqlens=lens))
        for n in ("q", "k", "v", "graw", "b", "A_log", "initial_state"):
            d[n].copy_(new[n])
        g.replay()
        torch.cuda.synchronize()
        ref_out, ref_fin = kda.kda_fwd(new["q"], new["k"], new["v"], new["graw"], new["b"], new["A_log"],
                                       new["scale"], initial_state=new["initial_state"],
                                       cu_seqlens=new["cu_seqlens"])
        torch.cuda.synchronize()
        assert torch.equal(out, ref_out)
        assert torch.equal(fin, ref_fin)
    assert kda.kda_get_status() == 0
