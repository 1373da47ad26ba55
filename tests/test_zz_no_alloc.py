"""The allocation-free forward (kda_fwd_noalloc) against kda_fwd.

kda_fwd_noalloc serves callers that cannot allocate device memory where they
run the forward (inside stream capture, under pool-only allocators, in
allocation-free serving loops): it uses the library's fixed 64 MiB device array
as workspace.  This file runs last so that a failure here leaves every other
test already run.
"""
import ctypes

import numpy as np
import pytest
import torch

import kda_inputs as KI
from kda_testutil import OUT_REL_L2, STATE_REL_L2, rel_l2, to_dev

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


def test_noalloc_matches_kda_fwd_on_two_calls_in_a_row():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gated_delta_rule_40_gb300 import kda
    first = KI.make_inputs(1, 450, 2, 4, seed=201, with_state=True, seqlens=[100, 37, 250, 63])
    second = KI.make_inputs(2, 300, 1, 2, seed=202, with_state=True)
    for inp in (first, second):
        ref_out, ref_fin, out, fin = _both(inp)
        o, ro = out.double().cpu().numpy(), ref_out.double().cpu().numpy()
        f, rf = fin.double().cpu().numpy(), ref_fin.double().cpu().numpy()
        assert rel_l2(o, ro) <= OUT_REL_L2 and np.abs(o - ro).max() <= 3e-2
        assert rel_l2(f, rf) <= STATE_REL_L2
    assert kda.kda_get_status() == 0


def test_noalloc_rejects_sizes_beyond_its_array():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gated_delta_rule_40_gb300 import kda
    lib = kda.load()
    fake = ctypes.c_void_p(0x100000)
    # B=2, T=16384, H=32 needs about 1.8 GB of workspace: rejected before any launch
    rc = lib.kda_fwd_noalloc(fake, fake, fake, fake, fake, fake, ctypes.c_float(0.1), None, None, None, 0, 2,
                             16384, 32, 32, 128, 128, fake, None)
    assert rc == kda.KDA_ERR_WORKSPACE
