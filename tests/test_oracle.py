"""CPU tests of the fp64 oracle against its pins (no GPU)."""
import functools

import numpy as np
import pytest
import torch

import kda_inputs as KI
import oracle
from oracle import chunk_model
from oracle_pins import PINS


@pytest.mark.parametrize("pin,tol", PINS, ids=[p.__name__ for p, _ in PINS])
def test_pin(pin, tol):
    err = pin(oracle.fwd)
    assert err <= tol, f"{pin.__name__}: {err:.3e} > {tol:.1e}"


MUTATIONS = {
    1: "decay dropped",
    2: "wrong sign of the erase term",
    3: "output read before the delta write",
    4: "state read transposed",
    5: "k not L2-normalised",
    6: "scale applied to k as well",
    7: "beta without the sigmoid",
    8: "softplus dropped from the gate",
    9: "decay channels reversed",
}


@pytest.mark.parametrize("m", sorted(MUTATIONS), ids=[MUTATIONS[m] for m in sorted(MUTATIONS)])
def test_pins_catch_planted_mistake(m):
    bad = functools.partial(oracle.fwd, mutation=m)
    failed = []
    with np.errstate(all="ignore"):
        for pin, tol in PINS:
            err = pin(bad)
            if not (err <= tol):
                failed.append(pin.__name__)
    assert failed, f"no pin catches mutation {m} ({MUTATIONS[m]})"


def _cmp(a, b):
    return np.abs(a - b).max() / max(np.abs(b).max(), 1e-300)


@pytest.mark.parametrize("case", ["random", "harsh", "partial", "varlen", "slow", "gva", "zero_len", "forget"])
def test_chunk_algebra_matches_oracle(case):
    """The chunked UT/WY form (with the sub-block decay references the GPU
    path uses) reproduces the token recurrence to fp64 rounding."""
    if case == "random":
        inp = KI.make_inputs(1, 192, 1, 2, seed=30, with_state=True)
    elif case == "harsh":
        inp = KI.make_inputs(1, 128, 1, 1, seed=31, with_state=True, graw_mean=3.0, A_log_value=1.0)
    elif case == "partial":
        inp = KI.make_inputs(2, 100, 1, 1, seed=32, with_state=True)
    elif case == "varlen":
        inp = KI.make_inputs(1, 200, 1, 1, seed=33, with_state=True, seqlens=[1, 63, 65, 71])
    elif case == "slow":
        inp = KI.make_inputs(1, 192, 1, 1, seed=34, with_state=True, graw_mean=-4.0, A_log_value=-1.0)
    elif case == "gva":
        inp = KI.make_inputs(1, 70, 1, 3, seed=35, with_state=True, scalar_gate=True)
    elif case == "forget":
        inp = KI.make_inputs(1, 100, 1, 1, seed=37, with_state=True)
        inp.graw.fill_(1e4)
        inp.b.fill_(float("inf"))
    else:
        inp = KI.make_inputs(1, 70, 1, 1, seed=36, with_state=True, seqlens=[0, 70, 0])
    o1, f1 = oracle.fwd_inputs(inp)
    o2, f2 = chunk_model.chunk_fwd_inputs(inp)
    assert _cmp(o2, o1) < 1e-10
    assert _cmp(f2, f1) < 1e-10


def test_zero_length_and_empty():
    """A zero-length sequence leaves its state unchanged; T = 0 writes no
    output and copies the initial state."""
    inp = KI.make_inputs(1, 10, 1, 1, seed=37, with_state=True, seqlens=[0, 10, 0])
    out, fin = oracle.fwd_inputs(inp)
    assert np.array_equal(fin[0], inp.initial_state[0].double().numpy())
    assert np.array_equal(fin[2], inp.initial_state[2].double().numpy())
    inp0 = KI.make_inputs(2, 0, 1, 1, seed=38, with_state=True)
    out0, fin0 = oracle.fwd_inputs(inp0)
    assert out0.shape == (2, 0, 1, 128)
    assert np.array_equal(fin0, inp0.initial_state.double().numpy())


def test_decode_is_one_step():
    d = KI.decode_inputs(B=3, H=4, H_qk=2, seed=39)
    out, new = oracle.decode(d)
    inp = KI.KdaInputs(q=d.q[:, None], k=d.k[:, None], v=d.v[:, None], graw=d.graw[:, None],
                       b=d.b[:, None], A_log=d.A_log, scale=d.scale, initial_state=d.state,
                       cu_seqlens=None)
    ro, rf = oracle.brute_force_inputs(inp)
    assert _cmp(out, ro[:, 0]) < 1e-12
    assert _cmp(new, rf) < 1e-12


def test_threads_do_not_change_result():
    inp = KI.make_inputs(1, 50, 2, 4, seed=40, with_state=True, seqlens=[20, 30])
    a = oracle.fwd_inputs(inp, nthreads=1)
    b = oracle.fwd_inputs(inp, nthreads=5)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_oracle_rejects_bad_args():
    inp = KI.make_inputs(1, 4, 2, 3, seed=41, with_state=False)
    with pytest.raises(ValueError):
        oracle.fwd_inputs(inp)   # H_v not a multiple of H_qk


def test_varlen_generator_shape():
    lens = KI.skewed_seqlens(16384, 20, 8192, 16, 4096, seed=1)
    assert len(lens) == 20 and sum(lens) == 16384 and 8192 in lens and min(lens) >= 1


def test_golden_fixture():
    """Stored oracle outputs for a small case (written by
    tests/golden/make_golden.py, which calls only the oracle) reproduce on this
    machine; guards the oracle build against compiler or platform drift."""
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "kda_small.txt")
    ref = np.loadtxt(path)
    from golden.make_golden import golden_case
    out, fin = oracle.fwd_inputs(golden_case())
    got = np.concatenate([out.ravel(), fin.ravel()])
    assert got.shape == ref.shape
    assert np.abs(got - ref).max() <= 1e-13 * np.abs(ref).max()
