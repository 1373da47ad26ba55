"""CPU tests of the C-ABI library: it loads, exports every symbol the header
declares, and its host-side validation rejects bad arguments before touching
any device (the pointers below are never dereferenced)."""
import ctypes

import pytest

from gated_delta_rule_40_gb300 import kda


@pytest.fixture(scope="module")
def lib():
    return kda.load()


def test_exports_every_declared_symbol(lib):
    names = kda.declared_symbols()
    assert {"kda_fwd", "kda_fwd_ws", "kda_fwd_workspace_size", "kda_decode_step", "kda_status_string",
            "kda_get_status", "kda_last_launch_count"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for code in (0, -1, -2, -3, -4, -5, -6):
        assert kda.status_string(code) and kda.status_string(code) != "unknown status"
    assert kda.status_string(17) == "unknown status"


def test_workspace_size(lib):
    assert kda.kda_fwd_workspace_size(0, 2, 16384, 32, 32) > 2 * 16384 * 32 * 1700
    assert kda.kda_fwd_workspace_size(20, 1, 16384, 32, 32) >= kda.kda_fwd_workspace_size(0, 1, 16384, 32, 32)
    assert kda.kda_fwd_workspace_size(0, 1, 64, 1, 1, K=64) == 0


FAKE = ctypes.c_void_p(0x100000)
FAKE_ODD = ctypes.c_void_p(0x100008)


def _fwd(lib, K=128, V=128, H_qk=1, H_v=1, B=1, T=4, N=0, cu=None, out=FAKE):
    return lib.kda_fwd(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.c_float(0.1), None, None, cu, N, B, T,
                       H_qk, H_v, K, V, out, None)


def test_fwd_rejects_unsupported_dims(lib):
    assert _fwd(lib, K=64) == kda.KDA_ERR_UNSUPPORTED
    assert _fwd(lib, V=256) == kda.KDA_ERR_UNSUPPORTED


def test_fwd_rejects_bad_heads_and_sizes(lib):
    assert _fwd(lib, H_qk=2, H_v=3) == kda.KDA_ERR_INVALID_ARG
    assert _fwd(lib, T=-1) == kda.KDA_ERR_INVALID_ARG
    assert _fwd(lib, B=2, N=1, cu=FAKE) == kda.KDA_ERR_INVALID_ARG
    assert _fwd(lib, out=FAKE_ODD) == kda.KDA_ERR_INVALID_ARG
    assert _fwd(lib, out=None) == kda.KDA_ERR_INVALID_ARG


def test_fwd_ws_rejects_small_workspace(lib):
    rc = lib.kda_fwd_ws(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.c_float(0.1), None, None, None, 0, 1, 64,
                        1, 1, 128, 128, FAKE, FAKE, ctypes.c_size_t(16), None)
    assert rc == kda.KDA_ERR_WORKSPACE


def test_decode_rejects_bad_args(lib):
    rc = lib.kda_decode_step(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.c_float(0.1), FAKE, 1, 1, 1, 128, 64,
                             FAKE, None)
    assert rc == kda.KDA_ERR_UNSUPPORTED
    rc = lib.kda_decode_step(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.c_float(0.1), None, 1, 1, 1, 128, 128,
                             FAKE, None)
    assert rc == kda.KDA_ERR_INVALID_ARG
    rc = lib.kda_decode_step(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.c_float(0.1), FAKE, 0, 1, 1, 128, 128,
                             FAKE, None)
    assert rc == kda.KDA_OK


def test_la_fwd_rejects_bad_args(lib):
    f = ctypes.c_float(0.1)
    la = lambda K=128, V=128, H_qk=1, H_v=1, B=1, T=4, N=0, cu=None, q=FAKE, slope=FAKE: lib.kda_la_fwd(  # noqa: E731
        q, FAKE, FAKE, slope, f, None, None, cu, N, B, T, H_qk, H_v, K, V, FAKE, None)
    assert la(K=64) == kda.KDA_ERR_UNSUPPORTED
    assert la(H_qk=2, H_v=3) == kda.KDA_ERR_INVALID_ARG
    assert la(T=-1) == kda.KDA_ERR_INVALID_ARG
    assert la(B=2, N=1, cu=FAKE) == kda.KDA_ERR_INVALID_ARG
    assert la(q=FAKE_ODD) == kda.KDA_ERR_INVALID_ARG     # TMA needs 16-byte aligned tensors
    assert la(slope=None) == kda.KDA_ERR_INVALID_ARG


def test_la_decode_rejects_bad_args(lib):
    f = ctypes.c_float(0.1)
    assert lib.kda_la_decode(FAKE, FAKE, FAKE, FAKE, f, FAKE, 1, 1, 1, 128, 64, FAKE, None) == kda.KDA_ERR_UNSUPPORTED
    assert lib.kda_la_decode(FAKE, FAKE, FAKE, None, f, FAKE, 1, 1, 1, 128, 128, FAKE, None) == kda.KDA_ERR_INVALID_ARG
    assert lib.kda_la_decode(FAKE, FAKE, FAKE, FAKE, f, FAKE, 1, 2, 3, 128, 128, FAKE, None) == kda.KDA_ERR_INVALID_ARG
    assert lib.kda_la_decode(FAKE, FAKE, FAKE, FAKE, f, FAKE, 0, 1, 1, 128, 128, FAKE, None) == kda.KDA_OK


def test_bwd_rejects_bad_args(lib):
    f = ctypes.c_float(0.1)

    def bwd(K=128, H_qk=1, H_v=1, dout=FAKE, dq=FAKE, dA=FAKE, dh0=FAKE):
        return lib.kda_bwd(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, f, None, None, 0, 1, 4, H_qk, H_v, K, 128, dout, None,
                           dq, FAKE, FAKE, FAKE, FAKE, dA, dh0, None)
    assert bwd(K=64) == kda.KDA_ERR_UNSUPPORTED
    assert bwd(H_qk=2, H_v=3) == kda.KDA_ERR_INVALID_ARG
    assert bwd(dout=None) == kda.KDA_ERR_INVALID_ARG
    assert bwd(dq=None) == kda.KDA_ERR_INVALID_ARG
    assert bwd(dq=FAKE_ODD) == kda.KDA_ERR_INVALID_ARG
    assert bwd(dA=None) == kda.KDA_ERR_INVALID_ARG
    assert bwd(dh0=None) == kda.KDA_ERR_INVALID_ARG


def test_work_item_limits(lib):
    """Calls whose 32-bit work-item indices would overflow are rejected before any device
    call: 2^28 sequences x 2 value heads x 4 row blocks, and 2^30 x 2 decode pairs."""
    f = ctypes.c_float(0.1)
    big = 1 << 28
    assert _fwd(lib, H_v=2, B=1, T=4, N=big, cu=FAKE) == kda.KDA_ERR_INVALID_ARG
    assert _fwd(lib, H_v=2, B=big, T=1) == kda.KDA_ERR_INVALID_ARG
    assert lib.kda_fwd_host(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, f, None, None, FAKE, big, 1, 4, 1, 2, 128, 128,
                            FAKE, None) == kda.KDA_ERR_INVALID_ARG
    assert lib.kda_la_fwd(FAKE, FAKE, FAKE, FAKE, f, None, None, FAKE, big, 1, 4, 1, 2, 128, 128, FAKE,
                          None) == kda.KDA_ERR_INVALID_ARG
    assert lib.kda_bwd(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, f, None, None, 0, big, 1, 1, 2, 128, 128, FAKE, None,
                       FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None) == kda.KDA_ERR_INVALID_ARG
    pairs = 1 << 30
    assert lib.kda_decode_step(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, f, FAKE, pairs, 1, 2, 128, 128, FAKE,
                               None) == kda.KDA_ERR_INVALID_ARG
    assert lib.kda_decode_tokens(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, f, FAKE, 0, pairs, 1, 1, 2, 128, 128, FAKE,
                                 None) == kda.KDA_ERR_INVALID_ARG
    assert lib.kda_la_decode(FAKE, FAKE, FAKE, FAKE, f, FAKE, pairs, 1, 2, 128, 128, FAKE,
                             None) == kda.KDA_ERR_INVALID_ARG
