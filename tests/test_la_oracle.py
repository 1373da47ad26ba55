"""CPU tests pinning the lightning-attention oracle (no GPU).

The oracle is the token recurrence S_t = lambda S_{t-1} + v_t k_t^T,
o_t = scale S_t q_t (lambda = exp(-slope[h])).  Its pins are facts that do not
go through that recurrence: the parallel (attention-matrix) form, the plain
cumulative sum that the method reduces to without decay, the closed form of a
decaying state with no writes, and exact retrieval with one-hot keys."""
import functools

import numpy as np
import pytest
import torch

import kda_inputs as KI
import oracle


def _rel(a, b):
    return np.abs(a - b).max() / max(np.abs(b).max(), 1e-300)


def _cases():
    return [
        KI.make_la_inputs(2, 150, 2, 4, seed=1),
        KI.make_la_inputs(1, 200, 1, 2, seed=2, seqlens=[0, 64, 1, 0, 70, 65]),
        KI.make_la_inputs(3, 40, 2, 2, seed=3, with_state=False),
        KI.make_la_inputs(1, 96, 1, 1, seed=4, slope=torch.tensor([3.0])),
    ]


def pin_parallel_form(fwd):
    """Largest relative deviation from the attention-matrix form over the cases."""
    err = 0.0
    for inp in _cases():
        o, f = fwd(inp.q, inp.k, inp.v, inp.slope, inp.scale, inp.initial_state, inp.cu_seqlens)
        ro, rf = oracle.la_quadratic_inputs(inp)
        err = max(err, _rel(o, ro), _rel(f, rf))
    return err


def pin_no_decay_cumsum(fwd):
    """slope = 0: S_t = S_0 + cumsum_j v_j k_j^T, o_t = scale S_t q_t."""
    inp = KI.make_la_inputs(1, 70, 1, 2, seed=5, slope=torch.zeros(2))
    o, f = fwd(inp.q, inp.k, inp.v, inp.slope, inp.scale, inp.initial_state, None)
    q, k, v = (t.double().numpy()[0] for t in (inp.q, inp.k, inp.v))
    err = 0.0
    for h in range(2):
        outer = np.einsum("tv,tk->tvk", v[:, h], k[:, 0])
        S = np.cumsum(outer, axis=0) + inp.initial_state[0, h].double().numpy()[None]
        ref = np.float32(inp.scale) * np.einsum("tvk,tk->tv", S, q[:, 0])
        err = max(err, _rel(o[0, :, h], ref), _rel(f[0, h], S[-1]))
    return err


def pin_decay_only(fwd):
    """v = 0: the state only decays, S_t = lambda^(t+1) S_0 and o_t = scale lambda^(t+1) S_0 q_t."""
    inp = KI.make_la_inputs(1, 50, 1, 3, seed=6)
    inp.v.zero_()
    o, f = fwd(inp.q, inp.k, inp.v, inp.slope, inp.scale, inp.initial_state, None)
    lam = np.exp(-inp.slope.double().numpy())
    q = inp.q.double().numpy()[0, :, 0]
    err = 0.0
    for h in range(3):
        S0 = inp.initial_state[0, h].double().numpy()
        p = lam[h] ** np.arange(1, 51)
        ref = np.float32(inp.scale) * p[:, None] * (q @ S0.T)
        err = max(err, _rel(o[0, :, h], ref), _rel(f[0, h], lam[h] ** 50 * S0))
    return err


def pin_one_hot_retrieval(fwd):
    """Token j writes v_j under the one-hot key e_j; the query e_i at step t >= i
    reads exactly scale lambda^(t-i) v_i, and 0 for i > t (zero initial state)."""
    T, K = 100, 128
    inp = KI.make_la_inputs(1, T, 1, 1, seed=7, with_state=False, slope=torch.tensor([0.05]))
    eye = torch.eye(K, dtype=torch.bfloat16)
    inp.k[0, :, 0] = eye[:T]
    perm = torch.randperm(T, generator=torch.Generator().manual_seed(8))
    inp.q[0, :, 0] = eye[perm]
    o, f = fwd(inp.q, inp.k, inp.v, inp.slope, inp.scale, None, None)
    lam = np.exp(-np.float64(np.float32(0.05)))
    v = inp.v.double().numpy()[0, :, 0]
    ref = np.zeros((T, K))
    for t in range(T):
        i = int(perm[t])
        if i <= t:
            ref[t] = np.float32(inp.scale) * lam ** (t - i) * v[i]
    return _rel(o[0, :, 0], ref)


PINS = [(pin_parallel_form, 1e-10), (pin_no_decay_cumsum, 1e-10), (pin_decay_only, 1e-10),
        (pin_one_hot_retrieval, 1e-12)]


@pytest.mark.parametrize("pin,tol", PINS, ids=[p.__name__ for p, _ in PINS])
def test_la_pin(pin, tol):
    err = pin(oracle.la_fwd)
    assert err <= tol, f"{pin.__name__}: {err:.3e} > {tol:.1e}"


MUTATIONS = {
    1: "decay applied after the write",
    2: "output read before the write",
    3: "q written instead of k",
    4: "scale dropped",
    5: "another head's decay",
    6: "value heads grouped the wrong way",
}


@pytest.mark.parametrize("m", sorted(MUTATIONS), ids=[MUTATIONS[m] for m in sorted(MUTATIONS)])
def test_la_pins_catch_planted_mistake(m):
    bad = functools.partial(oracle.la_fwd, mutation=m)
    failed = [p.__name__ for p, tol in PINS if not (p(bad) <= tol)]
    assert failed, f"no pin catches mutation {m} ({MUTATIONS[m]})"


def test_la_parallel_form_is_not_the_recurrence():
    """The parallel form is a separate formulation: it does not call the C oracle."""
    import inspect
    src = inspect.getsource(oracle.la_quadratic)
    assert "la_oracle_fwd" not in src and "_load" not in src


def test_la_state_handoff():
    """Running a sequence in two pieces, the second from the first's final state,
    equals one run (the recurrence carries everything in S)."""
    inp = KI.make_la_inputs(1, 130, 1, 2, seed=9)
    o, f = oracle.la_fwd_inputs(inp)
    o1, f1 = oracle.la_fwd(inp.q[:, :57], inp.k[:, :57], inp.v[:, :57], inp.slope, inp.scale, inp.initial_state)
    o2, f2 = oracle.la_fwd(inp.q[:, 57:], inp.k[:, 57:], inp.v[:, 57:], inp.slope, inp.scale,
                           torch.from_numpy(f1).float())
    # the hand-off rounds the state to fp32, so compare at fp32 precision
    assert _rel(np.concatenate([o1, o2], 1), o) <= 1e-6 and _rel(f2, f) <= 1e-6


def test_la_decode_is_one_forward_step():
    d = KI.la_decode_inputs(B=3, H=4, seed=10)
    out, st = oracle.la_decode(d)
    o, f = oracle.la_quadratic(d.q[:, None], d.k[:, None], d.v[:, None], d.slope, d.scale, d.state)
    assert _rel(out, o[:, 0]) <= 1e-12 and _rel(st, f) <= 1e-12
