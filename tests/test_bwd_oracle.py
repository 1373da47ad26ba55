"""CPU tests pinning the backward oracle (fp64 autograd through the token
recurrence) to central finite differences of the independent explicit-matrix
forward (``oracle.brute_force``), on small fp64 problems."""
import numpy as np
import pytest
import torch

import oracle
from oracle import backward as OB


def _problem(seed, B=1, T=4, H_qk=1, H_v=2, K=4, V=4, seqlens=None, with_state=True):
    g = torch.Generator().manual_seed(seed)
    r = lambda *s: torch.randn(*s, generator=g, dtype=torch.float64)  # noqa: E731
    if seqlens is not None:
        assert B == 1 and sum(seqlens) == T
        cu = torch.tensor([0] + list(np.cumsum(seqlens)), dtype=torch.int32)
        N = len(seqlens)
    else:
        cu, N = None, B
    x = dict(q=r(B, T, H_qk, K), k=r(B, T, H_qk, K), v=r(B, T, H_v, V), graw=r(B, T, H_v, K), b=r(B, T, H_v),
             A_log=0.5 * r(H_v), h0=0.3 * r(N, H_v, V, K) if with_state else None)
    do, dht = r(B, T, H_v, V), r(N, H_v, V, K)
    return x, cu, do, dht


def _loss(x, cu, do, dht, scale):
    o, f = oracle.brute_force(torch.as_tensor(x["q"]), torch.as_tensor(x["k"]), torch.as_tensor(x["v"]),
                              torch.as_tensor(x["graw"]), torch.as_tensor(x["b"]), torch.as_tensor(x["A_log"]),
                              scale, None if x["h0"] is None else torch.as_tensor(x["h0"]), cu)
    return float((o * do.numpy()).sum() + (f * dht.numpy()).sum())


def _fd(x, cu, do, dht, scale, name, h=1e-6):
    base = {k_: (None if v_ is None else v_.clone()) for k_, v_ in x.items()}
    grad = torch.zeros_like(base[name])
    flat = base[name].view(-1)
    gflat = grad.view(-1)
    for i in range(flat.numel()):
        old = float(flat[i])
        flat[i] = old + h
        lp = _loss(base, cu, do, dht, scale)
        flat[i] = old - h
        lm = _loss(base, cu, do, dht, scale)
        flat[i] = old
        gflat[i] = (lp - lm) / (2 * h)
    return grad


NAMES = {"q": "dq", "k": "dk", "v": "dv", "graw": "dgraw", "b": "db", "A_log": "dA_log", "h0": "dh0"}


def _max_rel(a, b):
    return float((a - b).abs().max() / max(float(b.abs().max()), 1e-300))


def _check(seed, mutation=0, **kw):
    scale = 0.5
    x, cu, do, dht = _problem(seed, **kw)
    got = OB.bwd(x["q"], x["k"], x["v"], x["graw"], x["b"], x["A_log"], scale, x["h0"], cu, do=do, dht=dht,
                 mutation=mutation)
    err = 0.0
    for name, gname in NAMES.items():
        if x[name] is None:
            continue
        err = max(err, _max_rel(got[gname], _fd(x, cu, do, dht, scale, name)))
    return err


@pytest.mark.parametrize("case", ["plain", "gva_varlen", "no_state"])
def test_bwd_oracle_matches_finite_differences(case):
    if case == "plain":
        err = _check(1)
    elif case == "gva_varlen":
        err = _check(2, T=5, H_qk=1, H_v=2, seqlens=[3, 0, 2])
    else:
        err = _check(3, with_state=False, B=2, T=3)
    assert err <= 1e-6, err


@pytest.mark.parametrize("m", [1, 2], ids=["decay gradient dropped", "erase-term gradient dropped"])
def test_fd_pin_catches_planted_mistake(m):
    assert _check(1, mutation=m) > 1e-3


def test_bwd_oracle_forward_equals_c_oracle():
    """The differentiable recurrence is the forward oracle's: same outputs on bf16 inputs."""
    import kda_inputs as KI
    inp = KI.make_inputs(1, 20, 1, 2, seed=5, with_state=True, seqlens=[12, 8])
    o, f = OB._recurrence(*(t.double() for t in (inp.q, inp.k, inp.v, inp.graw, inp.b, inp.A_log)),
                          float(torch.tensor(inp.scale, dtype=torch.float32)), inp.initial_state.double(),
                          inp.cu_seqlens, inp.H_qk)
    ro, rf = oracle.fwd_inputs(inp)
    assert np.abs(o.detach().numpy() - ro).max() <= 1e-9 * max(1.0, np.abs(ro).max())
    assert np.abs(f.detach().numpy() - rf).max() <= 1e-9 * max(1.0, np.abs(rf).max())


@pytest.mark.parametrize("case", ["plain", "gva_varlen", "no_state", "short_checkpoints"])
def test_recurrent_backward_matches_autograd(case):
    """The explicit reverse pass (for long sequences) equals the autograd oracle."""
    import kda_inputs as KI
    if case == "plain":
        inp, ck = KI.make_inputs(1, 70, 1, 2, seed=20, with_state=True), 64
    elif case == "gva_varlen":
        inp, ck = KI.make_inputs(1, 90, 1, 2, seed=21, with_state=True, seqlens=[40, 0, 1, 49]), 16
    elif case == "no_state":
        inp, ck = KI.make_inputs(2, 33, 2, 2, seed=22, with_state=False), 64
    else:
        inp, ck = KI.make_inputs(1, 50, 1, 1, seed=23, with_state=True, graw_mean=3.0, A_log_value=1.0), 7
    g = torch.Generator().manual_seed(30)
    do = torch.randn(inp.v.shape, generator=g).to(torch.bfloat16)
    dht = torch.randn((inp.N, inp.H_v, 128, 128), generator=g) * 0.1
    a = OB.bwd_inputs(inp, do, dht)
    r = OB.bwd_recurrent_inputs(inp, do, dht, checkpoint=ck)
    for name in a:
        err = _max_rel(r[name], a[name])
        assert err <= 1e-9, (name, err)


@pytest.mark.parametrize("case", ["plain", "gva_varlen", "no_state", "small_chunks"])
def test_chunked_backward_algebra_matches_autograd(case):
    """The chunked (UT/WY) backward formulas, the algebra a tensor-core backward
    uses, give the autograd oracle's gradients."""
    import kda_inputs as KI
    from oracle import chunk_bwd_model as CB
    if case == "plain":
        inp, C = KI.make_inputs(1, 150, 1, 2, seed=50, with_state=True), 64
    elif case == "gva_varlen":
        inp, C = KI.make_inputs(1, 140, 1, 2, seed=51, with_state=True, seqlens=[70, 0, 1, 69]), 64
    elif case == "no_state":
        inp, C = KI.make_inputs(2, 65, 2, 2, seed=52, with_state=False), 64
    else:
        inp, C = KI.make_inputs(1, 50, 1, 1, seed=53, with_state=True), 16
    g = torch.Generator().manual_seed(31)
    do = torch.randn(inp.v.shape, generator=g).to(torch.bfloat16)
    dht = torch.randn((inp.N, inp.H_v, 128, 128), generator=g) * 0.1
    a = OB.bwd_inputs(inp, do, dht)
    c = CB.chunk_bwd_inputs(inp, do, dht, C=C)
    for name in a:
        err = _max_rel(c[name], a[name])
        assert err <= 1e-9, (name, err)


def _rel_l2(x, ref):
    x, ref = np.asarray(x, dtype=np.float64), np.asarray(ref, dtype=np.float64)
    return float(np.linalg.norm(x - ref) / max(np.linalg.norm(ref), 1e-300))


@pytest.mark.parametrize("case", ["mha", "gva"])
def test_chunked_backward_operand_formats(case):
    """Operand formats for a tensor-core chunked backward, chosen on the blocked form of
    the chunk algebra (each product as a kernel forms it, operands rounded where they
    enter it, accumulators in fp32): bf16 for S0, W, dW, BV, T, dT and dA with
    nearest-rounded tf32 for the nine operands the gradients are most sensitive to (dS,
    Qg, P, Kd, Delta, dDelta, dP and the decayed keys and queries) keeps every gradient
    within rel-L2 6e-4 of the oracle (the GPU backward's bound is 1e-3); bf16 for all
    sixteen does not, and tf32 by truncation (the low bits dropped, a bias that adds up)
    comes out at about twice the nearest-rounded error."""
    import kda_inputs as KI
    from oracle import chunk_bwd_model as CB
    if case == "mha":
        inp = KI.make_inputs(1, 256, 1, 2, seed=60, with_state=True)
    else:
        inp = KI.make_inputs(1, 200, 2, 4, seed=80, with_state=True)
    g = torch.Generator().manual_seed(61)
    do = torch.randn(inp.v.shape, generator=g).to(torch.bfloat16)
    dht = torch.randn((inp.N, inp.H_v, 128, 128), generator=g) * 0.1
    ref = OB.bwd_recurrent_inputs(inp, do, dht)
    hi = ("dS", "Qg", "P", "Kd", "Delta", "dDelta", "dP", "Kdec", "Qdec")
    lo = ("S0", "W", "dW", "BV", "T", "dT", "dA")

    def worst(fmt_hi, fmt_lo):
        rounding = {**{n: fmt_lo for n in lo}, **{n: fmt_hi for n in hi}}
        got = CB.chunk_bwd_inputs(inp, do, dht, rounding=rounding, form="blocked")
        return max(_rel_l2(got[n], ref[n]) for n in ref)

    mixed = worst("tf32", "bf16")
    assert mixed <= 6e-4, mixed
    assert worst("bf16", "bf16") >= 1.5e-3
    assert worst("tf32_trunc", "bf16") >= 1.6 * mixed


def test_chunked_backward_blocked_form():
    """The blocked form (key products per pair of 16-row sub-blocks with reference
    points, as a kernel forms them) gives the pairwise form's gradients; at about 6 nats
    of decay per token (diagonal blocks inside the fp32 exponent clamp) and, with the
    clamp widened, at 22 nats per token it gives the reverse-pass oracle's (1e-9; 1e-8
    at 22 nats, where the gate gradients are about 1e-6 of the terms summed into them)."""
    import kda_inputs as KI
    from oracle import chunk_bwd_model as CB
    g = torch.Generator().manual_seed(34)
    inp = KI.make_inputs(1, 140, 1, 2, seed=51, with_state=True, seqlens=[70, 0, 1, 69])
    do = torch.randn(inp.v.shape, generator=g).to(torch.bfloat16)
    dht = torch.randn((inp.N, inp.H_v, 128, 128), generator=g) * 0.1
    a = CB.chunk_bwd_inputs(inp, do, dht, form="pairwise")
    b = CB.chunk_bwd_inputs(inp, do, dht, form="blocked")
    for name in a:
        assert _max_rel(b[name], a[name]) <= 1e-12, name
    for mean, alog, clamp in ((2.0, 1.0, 85.0), (3.0, 2.0, 400.0)):
        inp = KI.make_inputs(1, 100, 1, 2, seed=55, with_state=True, graw_mean=mean, graw_std=0.5, A_log_value=alog)
        do = torch.randn(inp.v.shape, generator=g).to(torch.bfloat16)
        dht = torch.randn((inp.N, inp.H_v, 128, 128), generator=g) * 0.1
        ref = OB.bwd_recurrent_inputs(inp, do, dht)
        got = CB.chunk_bwd_inputs(inp, do, dht, form="blocked", clamp=clamp)
        for name in ref:
            assert _max_rel(got[name], ref[name]) <= (1e-9 if clamp < 100 else 1e-8), (mean, name)


def test_chunk_model_rejects_key_side_rounding():
    import kda_inputs as KI
    from oracle import chunk_bwd_model as CB
    inp = KI.make_inputs(1, 8, 1, 1, seed=1, with_state=False)
    with pytest.raises(ValueError):
        CB.chunk_bwd_inputs(inp, torch.zeros(inp.v.shape), rounding={"Kn": "bf16"})


def test_chunked_backward_pairwise_form_equals_split():
    """The pairwise-decay form of the key products gives the split form's gradients."""
    import kda_inputs as KI
    from oracle import chunk_bwd_model as CB
    inp = KI.make_inputs(1, 140, 1, 2, seed=51, with_state=True, seqlens=[70, 0, 1, 69])
    g = torch.Generator().manual_seed(32)
    do = torch.randn(inp.v.shape, generator=g).to(torch.bfloat16)
    dht = torch.randn((inp.N, inp.H_v, 128, 128), generator=g) * 0.1
    a = CB.chunk_bwd_inputs(inp, do, dht)
    b = CB.chunk_bwd_inputs(inp, do, dht, form="pairwise")
    for name in a:
        assert _max_rel(b[name], a[name]) <= 1e-10, name


def test_chunked_backward_pairwise_form_survives_strong_gates():
    """A gate of about -22 nats per token (e^{A_log} = e^2, softplus(3)) takes a 64-token
    chunk's decay past 1400 nats: the split form's e^{-Gam} overflows, the pairwise form
    (every factor at most 1) still gives the reverse-pass oracle's gradients."""
    import kda_inputs as KI
    from oracle import chunk_bwd_model as CB
    inp = KI.make_inputs(1, 100, 1, 2, seed=54, with_state=True, graw_mean=3.0, graw_std=0.5, A_log_value=2.0)
    g = torch.Generator().manual_seed(33)
    do = torch.randn(inp.v.shape, generator=g).to(torch.bfloat16)
    dht = torch.randn((inp.N, inp.H_v, 128, 128), generator=g) * 0.1
    ref = OB.bwd_recurrent_inputs(inp, do, dht)
    got = CB.chunk_bwd_inputs(inp, do, dht, form="pairwise")
    for name in ref:
        assert torch.isfinite(got[name]).all(), name
        assert _max_rel(got[name], ref[name]) <= 1e-9, (name, _max_rel(got[name], ref[name]))
    with np.errstate(over="ignore", invalid="ignore", divide="ignore"):
        split = CB.chunk_bwd_inputs(inp, do, dht)
    assert not all(bool(torch.isfinite(split[n]).all()) for n in split)


def test_chunked_backward_intermediates():
    """What a phased backward passes between its phases, pinned independently: the state
    entering each chunk is the C oracle's final state of the prefix before it, and the
    gradient with respect to the state leaving a chunk is the reverse-pass oracle's dh0
    of the suffix problem after it (that state as its initial state, the same dO and dht)."""
    import kda_inputs as KI
    from oracle import chunk_bwd_model as CB
    inp = KI.make_inputs(1, 150, 1, 2, seed=56, with_state=True)       # chunks at 0, 64, 128
    g = torch.Generator().manual_seed(35)
    do = torch.randn(inp.v.shape, generator=g).to(torch.bfloat16)
    dht = torch.randn((inp.N, inp.H_v, 128, 128), generator=g) * 0.1
    grads, inter = CB.chunk_bwd_inputs(inp, do, dht, form="pairwise", return_intermediates=True)
    ref = OB.bwd_recurrent_inputs(inp, do, dht)
    for name in ref:
        assert _max_rel(grads[name], ref[name]) <= 1e-9, name
    cut = lambda t, a, b: t[:, a:b]  # noqa: E731
    for c0 in (64, 128):
        _, fin = oracle.fwd(cut(inp.q, 0, c0), cut(inp.k, 0, c0), cut(inp.v, 0, c0), cut(inp.graw, 0, c0),
                            cut(inp.b, 0, c0), inp.A_log, inp.scale, inp.initial_state)
        for h in range(inp.H_v):
            s0 = inter["S0"][(0, h, c0)]
            assert np.abs(s0 - fin[0, h]).max() <= 1e-12 * np.abs(fin[0, h]).max(), (c0, h)
    T = inp.q.shape[1]
    for c0, c1 in ((0, 64), (64, 128)):
        s_c1 = torch.from_numpy(np.stack([inter["S0"][(0, h, c1)] for h in range(inp.H_v)])[None])
        suf = OB.bwd_recurrent(cut(inp.q, c1, T), cut(inp.k, c1, T), cut(inp.v, c1, T), cut(inp.graw, c1, T),
                               cut(inp.b, c1, T), inp.A_log, inp.scale, s_c1, None, do=cut(do, c1, T), dht=dht)
        for h in range(inp.H_v):
            assert _max_rel(torch.from_numpy(inter["dS_end"][(0, h, c0)]), suf["dh0"][0, h]) <= 1e-9, (c0, h)
    for h in range(inp.H_v):
        assert np.array_equal(inter["dS_end"][(0, h, 128)], dht[0, h].double().numpy())
        assert inter["dDelta"][(0, h, 128)].shape == (T - 128, 128)


def test_operand_rounding_helper():
    """The model's roundings: bf16 equals torch's nearest-even conversion; tf32 keeps 10
    fraction bits, nearest with ties to even, or truncated."""
    from oracle import chunk_bwd_model as CB
    x = torch.randn(4096, generator=torch.Generator().manual_seed(7), dtype=torch.float64) * 10.0
    got = CB._round(x.numpy(), "bf16")
    want = x.to(torch.float32).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(got, want)
    u = 2.0 ** -10                       # one tf32 unit in the last place at 1.0
    cases = {1.0 + u / 2: 1.0,           # halfway, even neighbour below
             1.0 + 3 * u / 2: 1.0 + 2 * u,   # halfway, even neighbour above
             1.0 + u / 2 + u / 8: 1.0 + u,   # above halfway
             1.0 + u / 2 - u / 8: 1.0,       # below halfway
             -(1.0 + 3 * u / 4): -(1.0 + u)}
    for v, r in cases.items():
        assert CB._round(np.array([v]), "tf32")[0] == r, v
    assert CB._round(np.array([1.0 + 3 * u / 4]), "tf32_trunc")[0] == 1.0
    assert CB._round(np.array([-(1.0 + 3 * u / 4)]), "tf32_trunc")[0] == -1.0
    assert CB._round(np.array([1.0 + u]), "tf32_trunc")[0] == 1.0 + u
    with pytest.raises(ValueError):
        CB._round(np.array([1.0]), "fp8")
