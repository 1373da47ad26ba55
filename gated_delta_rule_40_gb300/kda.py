"""Python binding of libkda (include/kda.h): argument marshalling only.

Every function here takes torch tensors, checks dtype / device / layout (CUDA
tensors and a given stream must be on the current device, where the library
launches), passes raw pointers and the current CUDA stream to the C ABI and
raises on a non-zero return code.  All arithmetic runs in the CUDA kernels of libkda.so;
there is no other code path.  If the library is missing the first call raises
``KdaLibraryError``.
"""
from __future__ import annotations

import ctypes
import os
import re
from typing import Optional, Tuple

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkda.so")
HEADER_PATH = os.path.join(os.path.dirname(_HERE), "include", "kda.h")

KDA_OK = 0
KDA_ERR_INVALID_ARG = -1
KDA_ERR_UNSUPPORTED = -2
KDA_ERR_CUDA = -3
KDA_ERR_DEVICE_TIMEOUT = -4
KDA_ERR_BAD_SEQLENS = -5
KDA_ERR_WORKSPACE = -6


class KdaLibraryError(RuntimeError):
    pass


class KdaError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where}: {status_string(code)} ({code})")
        self.code = code


_lib = None


def load() -> ctypes.CDLL:
    """Load libkda.so (built in-tree by ``gated_delta_rule_40_gb300.build``)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise KdaLibraryError(f"{LIB_PATH} is missing; run __graft_entry__.build() first")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, F, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    fwd_args = [P, P, P, P, P, P, F, P, P, P, I, I, I, I, I, I, I, P]
    lib.kda_fwd.argtypes = fwd_args + [P]
    lib.kda_fwd.restype = I
    lib.kda_fwd_ws.argtypes = fwd_args + [P, Z, P]
    lib.kda_fwd_ws.restype = I
    lib.kda_fwd_noalloc.argtypes = fwd_args + [P]
    lib.kda_fwd_noalloc.restype = I
    lib.kda_fwd_host.argtypes = fwd_args + [P]
    lib.kda_fwd_host.restype = I
    lib.kda_fwd_scalar_gate.argtypes = fwd_args + [P]
    lib.kda_fwd_scalar_gate.restype = I
    lib.kda_fwd_workspace_size.argtypes = [I] * 7
    lib.kda_fwd_workspace_size.restype = Z
    lib.kda_decode_step.argtypes = [P, P, P, P, P, P, F, P, I, I, I, I, I, P, P]
    lib.kda_decode_step.restype = I
    lib.kda_decode_tokens.argtypes = [P, P, P, P, P, P, F, P, I, I, I, I, I, I, I, P, P]
    lib.kda_decode_tokens.restype = I
    lib.kda_fwd_bf16_state.argtypes = [P, P, P, P, P, P, F, P, P, P, I, I, I, I, I, I, I, P, P]
    lib.kda_fwd_bf16_state.restype = I
    bwd_args = [P, P, P, P, P, P, F, P, P, I, I, I, I, I, I, I, P, P, P, P, P, P, P, P, P]
    lib.kda_bwd.argtypes = bwd_args + [P]
    lib.kda_bwd.restype = I
    lib.kda_bwd_ws.argtypes = bwd_args + [P, Z, P]
    lib.kda_bwd_ws.restype = I
    lib.kda_bwd_workspace_size.argtypes = [I] * 7
    lib.kda_bwd_workspace_size.restype = Z
    lib.kda_la_fwd.argtypes = [P, P, P, P, F, P, P, P, I, I, I, I, I, I, I, P, P]
    lib.kda_la_fwd.restype = I
    lib.kda_la_decode.argtypes = [P, P, P, P, F, P, I, I, I, I, I, P, P]
    lib.kda_la_decode.restype = I
    lib.kda_status_string.argtypes = [I]
    lib.kda_status_string.restype = ctypes.c_char_p
    lib.kda_get_status.argtypes = [P]
    lib.kda_get_status.restype = I
    lib.kda_selftest_wait_timeout.argtypes = [P]
    lib.kda_selftest_wait_timeout.restype = I
    lib.kda_last_launch_count.argtypes = []
    lib.kda_last_launch_count.restype = I
    lib.kda_set_kernel_timing.argtypes = [I]
    lib.kda_set_kernel_timing.restype = I
    lib.kda_kernel_times.argtypes = [ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_char_p), I]
    lib.kda_kernel_times.restype = I
    lib.kda_release_cached_memory.argtypes = []
    lib.kda_release_cached_memory.restype = I
    _lib = lib
    return lib


def declared_symbols() -> list:
    """Names of the functions include/kda.h declares."""
    txt = open(HEADER_PATH).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w\s\*]*?\b(kda_\w+)\s*\(", txt, re.M)))


def status_string(code: int) -> str:
    return load().kda_status_string(int(code)).decode()


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    elif stream.device.index != torch.cuda.current_device():
        raise ValueError(f"stream is on {stream.device}, but the current CUDA device is "
                         f"cuda:{torch.cuda.current_device()}")
    return ctypes.c_void_p(stream.cuda_stream)


def _check(t: Optional[torch.Tensor], name: str, dtype, shape=None, optional=False, device: str = "cuda"):
    if t is None:
        if optional:
            return
        raise ValueError(f"{name} is required")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.device.type != device:
        raise ValueError(f"{name} must be a {'CUDA' if device == 'cuda' else 'host'} tensor")
    if device == "cuda" and t.device.index != torch.cuda.current_device():
        # the library launches on the calling thread's current device
        raise ValueError(f"{name} is on {t.device}, but the current CUDA device is "
                         f"cuda:{torch.cuda.current_device()} (select it with torch.cuda.set_device "
                         f"or torch.cuda.device)")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def _raise(rc: int, where: str):
    if rc != KDA_OK:
        raise KdaError(rc, where)


def kda_fwd_workspace_size(N: int, B: int, T: int, H_qk: int, H_v: int, K: int = 128, V: int = 128) -> int:
    return int(load().kda_fwd_workspace_size(N, B, T, H_qk, H_v, K, V))


def kda_fwd(q, k, v, graw, b, A_log, scale: float, initial_state=None, cu_seqlens=None,
            output_final_state: bool = True, out=None, final_state=None, workspace=None,
            stream=None) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """KDA forward.  Shapes: q, k [B,T,H_qk,K]; v, graw [B,T,H_v,*]; b [B,T,H_v]
    (bf16); A_log [H_v] fp32; initial_state [N,H_v,V,K] fp32 or None;
    cu_seqlens int32 [N+1] (device) or None.  Returns (out, final_state)."""
    lib = load()
    B, T, H_qk, K = q.shape
    H_v, V = v.shape[2], v.shape[3]
    N = cu_seqlens.numel() - 1 if cu_seqlens is not None else B
    bf = torch.bfloat16
    _check(q, "q", bf, (B, T, H_qk, K))
    _check(k, "k", bf, (B, T, H_qk, K))
    _check(v, "v", bf, (B, T, H_v, V))
    _check(graw, "graw", bf, (B, T, H_v, K))
    _check(b, "b", bf, (B, T, H_v))
    _check(A_log, "A_log", torch.float32, (H_v,))
    _check(initial_state, "initial_state", torch.float32, (N, H_v, V, K), optional=True)
    _check(cu_seqlens, "cu_seqlens", torch.int32, optional=True)
    if out is None:
        out = torch.empty((B, T, H_v, V), dtype=bf, device=q.device)
    _check(out, "out", bf, (B, T, H_v, V))
    if final_state is None and output_final_state:
        final_state = torch.empty((N, H_v, V, K), dtype=torch.float32, device=q.device)
    _check(final_state, "final_state", torch.float32, (N, H_v, V, K), optional=True)
    args = [_ptr(q), _ptr(k), _ptr(v), _ptr(graw), _ptr(b), _ptr(A_log), ctypes.c_float(scale),
            _ptr(initial_state), _ptr(final_state), _ptr(cu_seqlens), N, B, T, H_qk, H_v, K, V, _ptr(out)]
    if workspace is None:
        rc = lib.kda_fwd(*args, _stream(stream))
        _raise(rc, "kda_fwd")
    else:
        _check(workspace, "workspace", torch.uint8)
        rc = lib.kda_fwd_ws(*args, _ptr(workspace), ctypes.c_size_t(workspace.numel()), _stream(stream))
        _raise(rc, "kda_fwd_ws")
    return out, final_state


def kda_fwd_scalar_gate(q, k, v, graw, b, A_log, scale: float, initial_state=None, cu_seqlens=None,
                        output_final_state: bool = True, out=None, final_state=None,
                        stream=None) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """KDA forward with one gate value per token and value head: graw [B,T,H_v]
    (bf16).  Other shapes as ``kda_fwd``; equals ``kda_fwd`` with graw broadcast
    along K."""
    lib = load()
    B, T, H_qk, K = q.shape
    H_v, V = v.shape[2], v.shape[3]
    N = cu_seqlens.numel() - 1 if cu_seqlens is not None else B
    bf = torch.bfloat16
    _check(q, "q", bf, (B, T, H_qk, K))
    _check(k, "k", bf, (B, T, H_qk, K))
    _check(v, "v", bf, (B, T, H_v, V))
    _check(graw, "graw", bf, (B, T, H_v))
    _check(b, "b", bf, (B, T, H_v))
    _check(A_log, "A_log", torch.float32, (H_v,))
    _check(initial_state, "initial_state", torch.float32, (N, H_v, V, K), optional=True)
    _check(cu_seqlens, "cu_seqlens", torch.int32, optional=True)
    if out is None:
        out = torch.empty((B, T, H_v, V), dtype=bf, device=q.device)
    _check(out, "out", bf, (B, T, H_v, V))
    if final_state is None and output_final_state:
        final_state = torch.empty((N, H_v, V, K), dtype=torch.float32, device=q.device)
    _check(final_state, "final_state", torch.float32, (N, H_v, V, K), optional=True)
    rc = lib.kda_fwd_scalar_gate(_ptr(q), _ptr(k), _ptr(v), _ptr(graw), _ptr(b), _ptr(A_log), ctypes.c_float(scale),
                                 _ptr(initial_state), _ptr(final_state), _ptr(cu_seqlens), N, B, T, H_qk, H_v, K, V,
                                 _ptr(out), _stream(stream))
    _raise(rc, "kda_fwd_scalar_gate")
    return out, final_state


def kda_fwd_host(q, k, v, graw, b, A_log, scale: float, initial_state=None, cu_seqlens=None,
                 output_final_state: bool = True, out=None, final_state=None, stream=None,
                 synchronize: bool = True) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """``kda_fwd`` on host (CPU) tensors: the library copies the inputs to the
    GPU, runs the forward and copies ``out`` / ``final_state`` back, overlapping
    the copies of one token piece with the kernels of the previous one.  Pinned inputs
    (``tensor.pin_memory()``) run at the host link's bandwidth; outputs are
    allocated pinned when not given.  With ``synchronize`` the call waits for
    ``stream``, so the returned host tensors hold the results; without it they
    are valid once the stream has passed the call."""
    lib = load()
    B, T, H_qk, K = q.shape
    H_v, V = v.shape[2], v.shape[3]
    N = cu_seqlens.numel() - 1 if cu_seqlens is not None else B
    bf, cpu = torch.bfloat16, "cpu"
    _check(q, "q", bf, (B, T, H_qk, K), device=cpu)
    _check(k, "k", bf, (B, T, H_qk, K), device=cpu)
    _check(v, "v", bf, (B, T, H_v, V), device=cpu)
    _check(graw, "graw", bf, (B, T, H_v, K), device=cpu)
    _check(b, "b", bf, (B, T, H_v), device=cpu)
    _check(A_log, "A_log", torch.float32, (H_v,), device=cpu)
    _check(initial_state, "initial_state", torch.float32, (N, H_v, V, K), optional=True, device=cpu)
    _check(cu_seqlens, "cu_seqlens", torch.int32, optional=True, device=cpu)
    if out is None:
        out = torch.empty((B, T, H_v, V), dtype=bf).pin_memory()
    _check(out, "out", bf, (B, T, H_v, V), device=cpu)
    if final_state is None and output_final_state:
        final_state = torch.empty((N, H_v, V, K), dtype=torch.float32).pin_memory()
    _check(final_state, "final_state", torch.float32, (N, H_v, V, K), optional=True, device=cpu)
    s = _stream(stream)
    rc = lib.kda_fwd_host(_ptr(q), _ptr(k), _ptr(v), _ptr(graw), _ptr(b), _ptr(A_log), ctypes.c_float(scale),
                          _ptr(initial_state), _ptr(final_state), _ptr(cu_seqlens), N, B, T, H_qk, H_v, K, V,
                          _ptr(out), s)
    _raise(rc, "kda_fwd_host")
    if synchronize:
        (stream if stream is not None else torch.cuda.current_stream()).synchronize()
    return out, final_state


NOALLOC_WS_BYTES = 64 << 20


def kda_fwd_noalloc(q, k, v, graw, b, A_log, scale: float, initial_state=None, cu_seqlens=None,
                    out=None, final_state=None, stream=None) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """``kda_fwd`` for callers that cannot allocate device memory where they
    call it: the workspace is the library's fixed 64 MiB device array, shared
    by every call on the device (calls that overlap on the GPU race).  The
    caller still provides ``out`` and ``final_state`` (allocated here only if
    not given).  Raises KdaError(KDA_ERR_WORKSPACE) when the sizes need more
    workspace than the array holds."""
    lib = load()
    B, T, H_qk, K = q.shape
    H_v, V = v.shape[2], v.shape[3]
    N = cu_seqlens.numel() - 1 if cu_seqlens is not None else B
    bf = torch.bfloat16
    _check(q, "q", bf, (B, T, H_qk, K))
    _check(k, "k", bf, (B, T, H_qk, K))
    _check(v, "v", bf, (B, T, H_v, V))
    _check(graw, "graw", bf, (B, T, H_v, K))
    _check(b, "b", bf, (B, T, H_v))
    _check(A_log, "A_log", torch.float32, (H_v,))
    _check(initial_state, "initial_state", torch.float32, (N, H_v, V, K), optional=True)
    _check(cu_seqlens, "cu_seqlens", torch.int32, optional=True)
    if out is None:
        out = torch.empty((B, T, H_v, V), dtype=bf, device=q.device)
    _check(out, "out", bf, (B, T, H_v, V))
    _check(final_state, "final_state", torch.float32, (N, H_v, V, K), optional=True)
    rc = lib.kda_fwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(graw), _ptr(b), _ptr(A_log), ctypes.c_float(scale),
                             _ptr(initial_state), _ptr(final_state), _ptr(cu_seqlens), N, B, T, H_qk, H_v, K, V,
                             _ptr(out), _stream(stream))
    _raise(rc, "kda_fwd_noalloc")
    return out, final_state


def kda_decode_step(q, k, v, graw, b, A_log, scale: float, state, out=None, stream=None) -> torch.Tensor:
    """One decode step; ``state`` [B,H_v,V,K] fp32 is updated in place.
    Shapes: q, k [B,H_qk,K]; v, graw [B,H_v,*]; b [B,H_v] (bf16)."""
    lib = load()
    B, H_qk, K = q.shape
    H_v, V = v.shape[1], v.shape[2]
    bf = torch.bfloat16
    _check(q, "q", bf, (B, H_qk, K))
    _check(k, "k", bf, (B, H_qk, K))
    _check(v, "v", bf, (B, H_v, V))
    _check(graw, "graw", bf, (B, H_v, K))
    _check(b, "b", bf, (B, H_v))
    _check(A_log, "A_log", torch.float32, (H_v,))
    _check(state, "state", torch.float32, (B, H_v, V, K))
    if out is None:
        out = torch.empty((B, H_v, V), dtype=bf, device=q.device)
    _check(out, "out", bf, (B, H_v, V))
    rc = lib.kda_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(graw), _ptr(b), _ptr(A_log),
                             ctypes.c_float(scale), _ptr(state), B, H_qk, H_v, K, V, _ptr(out),
                             _stream(stream))
    _raise(rc, "kda_decode_step")
    return out


def kda_get_status(stream=None) -> int:
    return int(load().kda_get_status(_stream(stream)))


def kda_last_launch_count() -> int:
    return int(load().kda_last_launch_count())


def kda_set_kernel_timing(enable: bool) -> None:
    _raise(load().kda_set_kernel_timing(1 if enable else 0), "kda_set_kernel_timing")


def kda_kernel_times() -> list:
    """[(kernel name, ms)] for the most recent call on this thread (timing on)."""
    lib = load()
    ms = (ctypes.c_float * 8)()
    names = (ctypes.c_char_p * 8)()
    n = lib.kda_kernel_times(ms, names, 8)
    if n < 0:
        raise KdaError(n, "kda_kernel_times")
    return [(names[i].decode(), float(ms[i])) for i in range(n)]


def kda_release_cached_memory() -> None:
    """Hand the workspace pool's unused device memory back to the driver (the allocating
    entry points keep their largest workspace mapped between calls)."""
    _raise(load().kda_release_cached_memory(), "kda_release_cached_memory")


DECODE_MAX_TOKENS = 8


def kda_decode_tokens(q, k, v, graw, b, A_log, scale: float, state, out=None, stream=None) -> torch.Tensor:
    """Decode of Tq <= 8 consecutive tokens per (b, h) in one pass over ``state``
    [B,H_v,V,K] (fp32 or bf16, updated in place).  Shapes: q, k [B,Tq,H_qk,K];
    v, graw [B,Tq,H_v,*]; b [B,Tq,H_v] (bf16).  Returns out [B,Tq,H_v,V]."""
    lib = load()
    B, Tq, H_qk, K = q.shape
    H_v, V = v.shape[2], v.shape[3]
    bf = torch.bfloat16
    _check(q, "q", bf, (B, Tq, H_qk, K))
    _check(k, "k", bf, (B, Tq, H_qk, K))
    _check(v, "v", bf, (B, Tq, H_v, V))
    _check(graw, "graw", bf, (B, Tq, H_v, K))
    _check(b, "b", bf, (B, Tq, H_v))
    _check(A_log, "A_log", torch.float32, (H_v,))
    if state.dtype not in (torch.float32, bf):
        raise TypeError(f"state must be float32 or bfloat16, got {state.dtype}")
    _check(state, "state", state.dtype, (B, H_v, V, K))
    if out is None:
        out = torch.empty((B, Tq, H_v, V), dtype=bf, device=q.device)
    _check(out, "out", bf, (B, Tq, H_v, V))
    rc = lib.kda_decode_tokens(_ptr(q), _ptr(k), _ptr(v), _ptr(graw), _ptr(b), _ptr(A_log), ctypes.c_float(scale),
                               _ptr(state), 1 if state.dtype == bf else 0, B, Tq, H_qk, H_v, K, V, _ptr(out),
                               _stream(stream))
    _raise(rc, "kda_decode_tokens")
    return out


def kda_selftest_wait_timeout(stream=None) -> None:
    """Queue the self-test whose bounded device wait gives up and records
    KDA_ERR_DEVICE_TIMEOUT in the status word (see ``kda_get_status``)."""
    _raise(load().kda_selftest_wait_timeout(_stream(stream)), "kda_selftest_wait_timeout")


def kda_la_fwd(q, k, v, slope, scale: float, initial_state=None, cu_seqlens=None,
               output_final_state: bool = True, out=None, final_state=None,
               stream=None) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """Lightning-attention forward (fixed per-head decay exp(-slope[h])).
    Shapes: q, k [B,T,H_qk,K]; v [B,T,H_v,V] (bf16); slope [H_v] fp32;
    initial_state [N,H_v,V,K] fp32 or None; cu_seqlens int32 [N+1] (device) or
    None.  Returns (out, final_state)."""
    lib = load()
    B, T, H_qk, K = q.shape
    H_v, V = v.shape[2], v.shape[3]
    N = cu_seqlens.numel() - 1 if cu_seqlens is not None else B
    bf = torch.bfloat16
    _check(q, "q", bf, (B, T, H_qk, K))
    _check(k, "k", bf, (B, T, H_qk, K))
    _check(v, "v", bf, (B, T, H_v, V))
    _check(slope, "slope", torch.float32, (H_v,))
    _check(initial_state, "initial_state", torch.float32, (N, H_v, V, K), optional=True)
    _check(cu_seqlens, "cu_seqlens", torch.int32, optional=True)
    if out is None:
        out = torch.empty((B, T, H_v, V), dtype=bf, device=q.device)
    _check(out, "out", bf, (B, T, H_v, V))
    if final_state is None and output_final_state:
        final_state = torch.empty((N, H_v, V, K), dtype=torch.float32, device=q.device)
    _check(final_state, "final_state", torch.float32, (N, H_v, V, K), optional=True)
    rc = lib.kda_la_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(slope), ctypes.c_float(scale), _ptr(initial_state),
                        _ptr(final_state), _ptr(cu_seqlens), N, B, T, H_qk, H_v, K, V, _ptr(out), _stream(stream))
    _raise(rc, "kda_la_fwd")
    return out, final_state


def kda_la_decode(q, k, v, slope, scale: float, state, out=None, stream=None) -> torch.Tensor:
    """One lightning-attention decode step; ``state`` [B,H_v,V,K] fp32 is
    updated in place.  Shapes: q, k [B,H_qk,K]; v [B,H_v,V] (bf16); slope [H_v]."""
    lib = load()
    B, H_qk, K = q.shape
    H_v, V = v.shape[1], v.shape[2]
    bf = torch.bfloat16
    _check(q, "q", bf, (B, H_qk, K))
    _check(k, "k", bf, (B, H_qk, K))
    _check(v, "v", bf, (B, H_v, V))
    _check(slope, "slope", torch.float32, (H_v,))
    _check(state, "state", torch.float32, (B, H_v, V, K))
    if out is None:
        out = torch.empty((B, H_v, V), dtype=bf, device=q.device)
    _check(out, "out", bf, (B, H_v, V))
    rc = lib.kda_la_decode(_ptr(q), _ptr(k), _ptr(v), _ptr(slope), ctypes.c_float(scale), _ptr(state), B, H_qk,
                           H_v, K, V, _ptr(out), _stream(stream))
    _raise(rc, "kda_la_decode")
    return out


def kda_bwd_workspace_size(N: int, B: int, T: int, H_qk: int, H_v: int, K: int = 128, V: int = 128) -> int:
    return int(load().kda_bwd_workspace_size(N, B, T, H_qk, H_v, K, V))


def kda_bwd(q, k, v, graw, b, A_log, scale: float, dout, initial_state=None, cu_seqlens=None, dht=None,
            stream=None, workspace=None) -> dict:
    """Backward of ``kda_fwd``: returns fp32 gradients ``dq, dk`` [B,T,H_qk,K],
    ``dv`` [B,T,H_v,V], ``dgraw`` [B,T,H_v,K], ``db`` [B,T,H_v], ``dA_log``
    [H_v] and ``dh0`` [N,H_v,V,K] of a loss given ``dout`` (bf16, shape of
    out) and optionally ``dht`` (fp32, shape of the final state).  The
    workspace (``kda_bwd_workspace_size`` bytes, uint8 on the device) is
    ``workspace`` if given, else taken from torch's caching allocator, so that
    repeated calls reuse the same memory (kda_bwd_ws)."""
    lib = load()
    B, T, H_qk, K = q.shape
    H_v, V = v.shape[2], v.shape[3]
    N = cu_seqlens.numel() - 1 if cu_seqlens is not None else B
    bf, f32 = torch.bfloat16, torch.float32
    _check(q, "q", bf, (B, T, H_qk, K))
    _check(k, "k", bf, (B, T, H_qk, K))
    _check(v, "v", bf, (B, T, H_v, V))
    _check(graw, "graw", bf, (B, T, H_v, K))
    _check(b, "b", bf, (B, T, H_v))
    _check(A_log, "A_log", f32, (H_v,))
    _check(dout, "dout", bf, (B, T, H_v, V))
    _check(initial_state, "initial_state", f32, (N, H_v, V, K), optional=True)
    _check(dht, "dht", f32, (N, H_v, V, K), optional=True)
    _check(cu_seqlens, "cu_seqlens", torch.int32, optional=True)
    dev = q.device
    g = {"dq": torch.empty((B, T, H_qk, K), dtype=f32, device=dev),
         "dk": torch.empty((B, T, H_qk, K), dtype=f32, device=dev),
         "dv": torch.empty((B, T, H_v, V), dtype=f32, device=dev),
         "dgraw": torch.empty((B, T, H_v, K), dtype=f32, device=dev),
         "db": torch.empty((B, T, H_v), dtype=f32, device=dev),
         "dA_log": torch.empty((H_v,), dtype=f32, device=dev),
         "dh0": torch.empty((N, H_v, V, K), dtype=f32, device=dev)}
    if workspace is None:
        nbytes = int(lib.kda_bwd_workspace_size(N, B, T, H_qk, H_v, K, V))
        workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=dev)
    _check(workspace, "workspace", torch.uint8)
    rc = lib.kda_bwd_ws(_ptr(q), _ptr(k), _ptr(v), _ptr(graw), _ptr(b), _ptr(A_log), ctypes.c_float(scale),
                        _ptr(initial_state), _ptr(cu_seqlens), N, B, T, H_qk, H_v, K, V, _ptr(dout), _ptr(dht),
                        _ptr(g["dq"]), _ptr(g["dk"]), _ptr(g["dv"]), _ptr(g["dgraw"]), _ptr(g["db"]),
                        _ptr(g["dA_log"]), _ptr(g["dh0"]), _ptr(workspace), ctypes.c_size_t(workspace.numel()),
                        _stream(stream))
    _raise(rc, "kda_bwd_ws")
    return g


def kda_fwd_bf16_state(q, k, v, graw, b, A_log, scale: float, initial_state=None, cu_seqlens=None,
                       output_final_state: bool = True, out=None, final_state=None,
                       stream=None) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """``kda_fwd`` with the initial / final states in bf16 ([N,H_v,V,K]); the
    recurrence itself keeps an fp32 state."""
    lib = load()
    B, T, H_qk, K = q.shape
    H_v, V = v.shape[2], v.shape[3]
    N = cu_seqlens.numel() - 1 if cu_seqlens is not None else B
    bf = torch.bfloat16
    _check(q, "q", bf, (B, T, H_qk, K))
    _check(k, "k", bf, (B, T, H_qk, K))
    _check(v, "v", bf, (B, T, H_v, V))
    _check(graw, "graw", bf, (B, T, H_v, K))
    _check(b, "b", bf, (B, T, H_v))
    _check(A_log, "A_log", torch.float32, (H_v,))
    _check(initial_state, "initial_state", bf, (N, H_v, V, K), optional=True)
    _check(cu_seqlens, "cu_seqlens", torch.int32, optional=True)
    if out is None:
        out = torch.empty((B, T, H_v, V), dtype=bf, device=q.device)
    _check(out, "out", bf, (B, T, H_v, V))
    if final_state is None and output_final_state:
        final_state = torch.empty((N, H_v, V, K), dtype=bf, device=q.device)
    _check(final_state, "final_state", bf, (N, H_v, V, K), optional=True)
    rc = lib.kda_fwd_bf16_state(_ptr(q), _ptr(k), _ptr(v), _ptr(graw), _ptr(b), _ptr(A_log), ctypes.c_float(scale),
                                _ptr(initial_state), _ptr(final_state), _ptr(cu_seqlens), N, B, T, H_qk, H_v, K, V,
                                _ptr(out), _stream(stream))
    _raise(rc, "kda_fwd_bf16_state")
    return out, final_state
