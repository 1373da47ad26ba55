"""CPU tests of the C-ABI library: it loads, exports every symbol the header
declares, and its host-side validation rejects bad arguments before touching
any device.

Where only a rejection is asserted the data pointers are NULL.  A check that
needs non-NULL pointers (alignment, workspace size, cu_seqlens with B > 1)
gets the address of a real 16 MiB device buffer when a GPU is present, so
that a regression of the check would run on valid memory instead of faulting;
on a host without a GPU the address is a stand-in that nothing can
dereference (there is no device)."""
import ctypes

import pytest
import torch

from gated_delta_rule_40_gb300 import kda

if torch.cuda.is_available():
    _BUF = torch.zeros(16 << 20, dtype=torch.uint8, device="cuda")
    _BASE = _BUF.data_ptr()
else:
    _BASE = 0x100000


@pytest.fixture(scope="module")
def lib():
    return kda.load()


def test_exports_every_declared_symbol(lib):
    names = kda.declared_symbols()
    assert {"kda_fwd", "kda_fwd_ws", "kda_fwd_workspace_size", "kda_decode_step", "kda_status_string",
            "kda_get_status", "kda_last_launch_count", "kda_bwd", "kda_bwd_ws", "kda_bwd_workspace_size",
            "kda_release_cached_memory"} <= set(names)
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


# a valid, 16-byte aligned address (zeros: read as an int32 cu_seqlens it is [0, 0, ...])
FAKE = ctypes.c_void_p(_BASE)
FAKE_ODD = ctypes.c_void_p(_BASE + 8)


def _fwd(lib, K=128, V=128, H_qk=1, H_v=1, B=1, T=4, N=0, cu=None, out=None, data=None):
    return lib.kda_fwd(data, data, data, data, data, data, ctypes.c_float(0.1), None, None, cu, N, B, T,
                       H_qk, H_v, K, V, out, None)


def test_fwd_rejects_unsupported_dims(lib):
    assert _fwd(lib, K=64) == kda.KDA_ERR_UNSUPPORTED
    assert _fwd(lib, V=256) == kda.KDA_ERR_UNSUPPORTED


def test_fwd_rejects_bad_heads_and_sizes(lib):
    # T = 0: no token is read, so only the checked condition can reject the call
    assert _fwd(lib, H_qk=2, H_v=3, T=0) == kda.KDA_ERR_INVALID_ARG
    assert _fwd(lib, T=-1) == kda.KDA_ERR_INVALID_ARG
    assert _fwd(lib, B=2, N=1, T=0, cu=FAKE) == kda.KDA_ERR_INVALID_ARG
    assert _fwd(lib, out=None, data=FAKE) == kda.KDA_ERR_INVALID_ARG


# A regressed alignment check would launch kernels whose vector accesses fault on a
# misaligned address, so these run only where no GPU can execute anything.
no_device = pytest.mark.skipif(torch.cuda.is_available(), reason="misaligned pointers: host-only check")


@no_device
def test_fwd_rejects_misaligned_pointers(lib):
    assert _fwd(lib, out=FAKE_ODD, data=FAKE) == kda.KDA_ERR_INVALID_ARG
    assert _fwd(lib, out=FAKE, data=FAKE_ODD) == kda.KDA_ERR_INVALID_ARG


def test_fwd_ws_rejects_small_workspace(lib):
    rc = lib.kda_fwd_ws(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.c_float(0.1), None, None, None, 0, 1, 64,
                        1, 1, 128, 128, FAKE, FAKE, ctypes.c_size_t(16), None)
    assert rc == kda.KDA_ERR_WORKSPACE


def test_bwd_workspace_size(lib):
    # per (chunk, value head) about 434 KiB, plus 1 KiB per token and value head
    dense = kda.kda_bwd_workspace_size(0, 2, 16384, 32, 32)
    assert 8.0e9 < dense < 9.0e9
    assert kda.kda_bwd_workspace_size(20, 1, 16384, 32, 32) >= kda.kda_bwd_workspace_size(0, 1, 16384, 32, 32)
    assert kda.kda_bwd_workspace_size(0, 1, 64, 1, 1, K=64) == 0


def test_bwd_ws_rejects_small_workspace(lib):
    # T = 0 with NULL token tensors: only dA_log, dh0 and the workspace are real addresses, so a
    # regressed size check could touch nothing but the 16 MiB buffer behind FAKE
    f = ctypes.c_float(0.1)
    rc = lib.kda_bwd_ws(None, None, None, None, None, FAKE, f, None, None, 0, 1, 0, 1, 1, 128, 128, None, None,
                        None, None, None, None, None, FAKE, FAKE, FAKE, ctypes.c_size_t(16), None)
    assert rc == kda.KDA_ERR_WORKSPACE


def test_decode_rejects_bad_args(lib):
    rc = lib.kda_decode_step(None, None, None, None, None, None, ctypes.c_float(0.1), None, 1, 1, 1, 128, 64,
                             None, None)
    assert rc == kda.KDA_ERR_UNSUPPORTED
    rc = lib.kda_decode_step(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.c_float(0.1), None, 1, 1, 1, 128, 128,
                             FAKE, None)
    assert rc == kda.KDA_ERR_INVALID_ARG
    rc = lib.kda_decode_step(None, None, None, None, None, None, ctypes.c_float(0.1), None, 0, 1, 1, 128, 128,
                             None, None)
    assert rc == kda.KDA_OK


def test_la_fwd_rejects_bad_args(lib):
    f = ctypes.c_float(0.1)
    la = lambda K=128, V=128, H_qk=1, H_v=1, B=1, T=4, N=0, cu=None, q=FAKE, slope=FAKE: lib.kda_la_fwd(  # noqa: E731
        q, FAKE, FAKE, slope, f, None, None, cu, N, B, T, H_qk, H_v, K, V, FAKE, None)
    assert la(K=64, q=None) == kda.KDA_ERR_UNSUPPORTED
    assert la(H_qk=2, H_v=3, T=0) == kda.KDA_ERR_INVALID_ARG
    assert la(T=-1) == kda.KDA_ERR_INVALID_ARG
    assert la(B=2, N=1, T=0, cu=FAKE) == kda.KDA_ERR_INVALID_ARG
    assert la(slope=None, q=None) == kda.KDA_ERR_INVALID_ARG
    if not torch.cuda.is_available():
        assert la(q=FAKE_ODD) == kda.KDA_ERR_INVALID_ARG     # TMA needs 16-byte aligned tensors


def test_la_decode_rejects_bad_args(lib):
    f = ctypes.c_float(0.1)
    assert lib.kda_la_decode(None, None, None, None, f, None, 1, 1, 1, 128, 64, None, None) == kda.KDA_ERR_UNSUPPORTED
    assert lib.kda_la_decode(FAKE, FAKE, FAKE, None, f, FAKE, 1, 1, 1, 128, 128, FAKE, None) == kda.KDA_ERR_INVALID_ARG
    assert lib.kda_la_decode(None, None, None, None, f, None, 1, 2, 3, 128, 128, None, None) == kda.KDA_ERR_INVALID_ARG
    assert lib.kda_la_decode(None, None, None, None, f, None, 0, 1, 1, 128, 128, None, None) == kda.KDA_OK


def test_bwd_rejects_bad_args(lib):
    f = ctypes.c_float(0.1)

    def bwd(K=128, H_qk=1, H_v=1, T=4, dout=FAKE, dq=FAKE, dA=FAKE, dh0=FAKE):
        return lib.kda_bwd(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, f, None, None, 0, 1, T, H_qk, H_v, K, 128, dout, None,
                           dq, FAKE, FAKE, FAKE, FAKE, dA, dh0, None)
    assert bwd(K=64) == kda.KDA_ERR_UNSUPPORTED
    assert bwd(H_qk=2, H_v=3, T=0) == kda.KDA_ERR_INVALID_ARG
    assert bwd(dout=None) == kda.KDA_ERR_INVALID_ARG
    assert bwd(dq=None) == kda.KDA_ERR_INVALID_ARG
    assert bwd(dA=None) == kda.KDA_ERR_INVALID_ARG
    assert bwd(dh0=None) == kda.KDA_ERR_INVALID_ARG
    if not torch.cuda.is_available():
        assert bwd(dq=FAKE_ODD) == kda.KDA_ERR_INVALID_ARG


def test_work_item_limits(lib):
    """Calls whose 32-bit work-item indices would overflow are rejected before any device
    call: 2^28 sequences x 2 value heads x 4 row blocks, and 2^30 x 2 decode pairs.  The
    data pointers are NULL (a regressed size check then fails the pointer checks)."""
    f = ctypes.c_float(0.1)
    big = 1 << 28
    assert _fwd(lib, H_v=2, B=1, T=4, N=big, cu=FAKE) == kda.KDA_ERR_INVALID_ARG
    assert _fwd(lib, H_v=2, B=big, T=1) == kda.KDA_ERR_INVALID_ARG
    assert lib.kda_fwd_host(None, None, None, None, None, None, f, None, None, FAKE, big, 1, 4, 1, 2, 128, 128,
                            None, None) == kda.KDA_ERR_INVALID_ARG
    assert lib.kda_la_fwd(None, None, None, FAKE, f, None, None, FAKE, big, 1, 4, 1, 2, 128, 128, None,
                          None) == kda.KDA_ERR_INVALID_ARG
    assert lib.kda_bwd(None, None, None, None, None, FAKE, f, None, None, 0, big, 1, 1, 2, 128, 128, None, None,
                       None, None, None, None, None, FAKE, FAKE, None) == kda.KDA_ERR_INVALID_ARG
    pairs = 1 << 30
    assert lib.kda_decode_step(None, None, None, None, None, None, f, None, pairs, 1, 2, 128, 128, None,
                               None) == kda.KDA_ERR_INVALID_ARG
    assert lib.kda_decode_tokens(None, None, None, None, None, None, f, None, 0, pairs, 1, 1, 2, 128, 128, None,
                                 None) == kda.KDA_ERR_INVALID_ARG
    assert lib.kda_la_decode(None, None, None, None, f, None, pairs, 1, 2, 128, 128, None,
                             None) == kda.KDA_ERR_INVALID_ARG
