"""Thin Python binding of libfa.so (exact attention on GB300).

The functions carry the C entry points' names and only marshal arguments: torch tensors give device
pointers and the current CUDA stream; every step of the computation runs in the library's kernels.
There is no fallback: if ``libfa.so`` is missing or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfa.so")

FA_OK, FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED, FA_ERR_CUDA, FA_ERR_TIMEOUT = range(5)
STATUS_NAMES = {0: "FA_OK", 1: "FA_ERR_INVALID_ARG", 2: "FA_ERR_UNSUPPORTED", 3: "FA_ERR_CUDA", 4: "FA_ERR_TIMEOUT"}

# Every symbol include/fa.h declares.
EXPORTS = ("fa_fwd", "fa_fwd_stepnorm", "fa_fwd_f32", "fa_bwd_workspace_size", "fa_bwd", "fa_bwd_noalloc",
           "fa_last_error_string", "fa_check_status", "fa_kernel_launches", "fa_test_force_wait_timeout",
           "fa_debug_time_bwd_main")

# Bytes of the static scratch that fa_bwd_noalloc uses (FA_BWD_NOALLOC_MAX_SCRATCH_BYTES).
NOALLOC_MAX_SCRATCH_BYTES = 32 << 20

_lib = None


class FAError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Loads libfa.so and declares the C signatures; raises if the library is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with `python -m exact_io_aware_17_gb300.build`")
    lib = ctypes.CDLL(path)
    P, I, F, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.fa_fwd.argtypes = [P, P, P, P, P, I, I, I, I, F, P]
    lib.fa_fwd.restype = I
    lib.fa_fwd_stepnorm.argtypes = [P, P, P, P, P, I, I, I, I, F, P]
    lib.fa_fwd_stepnorm.restype = I
    lib.fa_fwd_f32.argtypes = [P, P, P, P, P, I, I, I, I, F, P]
    lib.fa_fwd_f32.restype = I
    lib.fa_bwd_workspace_size.argtypes = [I, I, I, I]
    lib.fa_bwd_workspace_size.restype = Z
    lib.fa_bwd.argtypes = [P, P, P, P, P, P, P, P, P, I, I, I, I, F, P, Z, P]
    lib.fa_bwd.restype = I
    lib.fa_bwd_noalloc.argtypes = [P, P, P, P, P, P, P, P, P, I, I, I, I, F, P]
    lib.fa_bwd_noalloc.restype = I
    lib.fa_last_error_string.argtypes = []
    lib.fa_last_error_string.restype = ctypes.c_char_p
    lib.fa_check_status.argtypes = [P]
    lib.fa_check_status.restype = I
    lib.fa_kernel_launches.argtypes = []
    lib.fa_kernel_launches.restype = ctypes.c_ulonglong
    lib.fa_debug_time_bwd_main.argtypes = [P, P]
    lib.fa_debug_time_bwd_main.restype = None
    lib.fa_test_force_wait_timeout.argtypes = [I]
    lib.fa_test_force_wait_timeout.restype = None
    _lib = lib
    return lib


def _check(status: int):
    if status != FA_OK:
        msg = load_library().fa_last_error_string().decode(errors="replace")
        raise FAError(status, msg)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream, device=None):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _shape(q):
    if q.dim() != 4:
        raise ValueError("expected [B, H, N, d] tensors")
    return tuple(int(x) for x in q.shape)


def _default_scale(d, scale):
    return 1.0 / math.sqrt(d) if scale is None else float(scale)


def _check_tensor(name, t, shape, dtype, device=None):
    if t.dtype != dtype or tuple(t.shape) != tuple(shape) or not t.is_contiguous() or not t.is_cuda:
        raise ValueError(f"{name}: expected a contiguous CUDA {dtype} tensor of shape {tuple(shape)}")
    if device is not None and t.device != device:
        raise ValueError(f"{name}: on {t.device}, expected {device} (every tensor of a call on one GPU)")


def fa_fwd(q, k, v, scale=None, o=None, lse=None, stream=None, _entry="fa_fwd"):
    """bf16 forward: returns (o bf16 [B,H,N,d], lse fp32 [B,H,N])."""
    B, H, N, d = _shape(q)
    dev = q.device
    for name, t in (("q", q), ("k", k), ("v", v)):
        _check_tensor(name, t, (B, H, N, d), torch.bfloat16, dev)
    o = torch.empty_like(q) if o is None else o
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev) if lse is None else lse
    _check_tensor("o", o, (B, H, N, d), torch.bfloat16, dev)
    _check_tensor("lse", lse, (B, H, N), torch.float32, dev)
    with torch.cuda.device(dev):
        _check(getattr(load_library(), _entry)(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, d,
                                               _default_scale(d, scale), _stream(stream, dev)))
    return o, lse


def fa_fwd_stepnorm(q, k, v, scale=None, o=None, lse=None, stream=None):
    """bf16 forward with the per-step normalised accumulator (ablation of fa_fwd's update rule)."""
    return fa_fwd(q, k, v, scale, o, lse, stream, _entry="fa_fwd_stepnorm")


def fa_fwd_f32(q, k, v, scale=None, o=None, lse=None, stream=None):
    """fp32 forward: returns (o fp32 [B,H,N,d], lse fp32 [B,H,N])."""
    B, H, N, d = _shape(q)
    dev = q.device
    for name, t in (("q", q), ("k", k), ("v", v)):
        _check_tensor(name, t, (B, H, N, d), torch.float32, dev)
    o = torch.empty_like(q) if o is None else o
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev) if lse is None else lse
    _check_tensor("o", o, (B, H, N, d), torch.float32, dev)
    _check_tensor("lse", lse, (B, H, N), torch.float32, dev)
    with torch.cuda.device(dev):
        _check(load_library().fa_fwd_f32(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, d,
                                         _default_scale(d, scale), _stream(stream, dev)))
    return o, lse


def fa_bwd_workspace_size(B, H, N, d) -> int:
    return int(load_library().fa_bwd_workspace_size(B, H, N, d))


def fa_bwd(q, k, v, o, do, lse, scale=None, dq=None, dk=None, dv=None, workspace=None, stream=None):
    """bf16 backward: returns (dq, dk, dv), bf16 [B,H,N,d].  ``workspace`` is a uint8 CUDA tensor of at
    least fa_bwd_workspace_size(B,H,N,d) bytes; one is allocated by torch if not given."""
    B, H, N, d = _shape(q)
    dev = q.device
    dq, dk, dv = _bwd_outputs(q, k, v, o, do, lse, dq, dk, dv)
    if workspace is None:
        workspace = torch.empty(fa_bwd_workspace_size(B, H, N, d), dtype=torch.uint8, device=dev)
    if not workspace.is_cuda or workspace.device != dev or not workspace.is_contiguous():
        raise ValueError(f"workspace: expected a contiguous tensor on {dev}")
    with torch.cuda.device(dev):
        _check(load_library().fa_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(dq), _ptr(dk),
                                     _ptr(dv), B, H, N, d, _default_scale(d, scale), _ptr(workspace),
                                     workspace.numel() * workspace.element_size(), _stream(stream, dev)))
    return dq, dk, dv


def _bwd_outputs(q, k, v, o, do, lse, dq, dk, dv):
    """Checks the backward's inputs and caller-given outputs (dtype, shape, contiguity, one device) and
    allocates the outputs not given."""
    B, H, N, d = _shape(q)
    dev = q.device
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("do", do)):
        _check_tensor(name, t, (B, H, N, d), torch.bfloat16, dev)
    _check_tensor("lse", lse, (B, H, N), torch.float32, dev)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    for name, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        _check_tensor(name, t, (B, H, N, d), torch.bfloat16, dev)
    return dq, dk, dv


def fa_bwd_noalloc(q, k, v, o, do, lse, scale=None, dq=None, dk=None, dv=None, stream=None):
    """bf16 backward that allocates no scratch: the library's static scratch array stands in for the
    workspace (for callers that cannot allocate device memory).  Pass preallocated dq, dk, dv to make
    the call allocate nothing at all; shapes needing more than NOALLOC_MAX_SCRATCH_BYTES of scratch
    raise FAError (FA_ERR_INVALID_ARG)."""
    B, H, N, d = _shape(q)
    dev = q.device
    dq, dk, dv = _bwd_outputs(q, k, v, o, do, lse, dq, dk, dv)
    with torch.cuda.device(dev):
        _check(load_library().fa_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(dq),
                                             _ptr(dk), _ptr(dv), B, H, N, d, _default_scale(d, scale),
                                             _stream(stream, dev)))
    return dq, dk, dv


def fa_check_status(stream=None):
    _check(load_library().fa_check_status(_stream(stream)))


def fa_kernel_launches() -> int:
    """Kernels libfa.so has launched in this process so far (a diagnostic; see include/fa.h)."""
    return int(load_library().fa_kernel_launches())


def fa_debug_time_bwd_main(start, stop) -> None:
    """Timing diagnostic: the next fa_bwd / fa_bwd_noalloc on this thread records the torch.cuda.Events
    `start` and `stop` (already recorded once, so that they exist) around its main kernel only."""
    load_library().fa_debug_time_bwd_main(ctypes.c_void_p(start.cuda_event), ctypes.c_void_p(stop.cuda_event))


def fa_test_force_wait_timeout(enable: bool) -> None:
    """Test switch of the failure path: while enabled, the tensor-core kernels withhold their Q loads and
    their bounded waits run out after ~10 ms (fa_check_status then raises FA_ERR_TIMEOUT).  Tests only."""
    load_library().fa_test_force_wait_timeout(1 if enable else 0)


def fa_last_error_string() -> str:
    return load_library().fa_last_error_string().decode(errors="replace")


__all__ = ["fa_fwd", "fa_fwd_stepnorm", "fa_fwd_f32", "fa_bwd", "fa_bwd_workspace_size", "fa_bwd_noalloc",
           "fa_check_status", "fa_last_error_string", "fa_kernel_launches", "fa_test_force_wait_timeout",
           "fa_debug_time_bwd_main", "load_library", "FAError", "EXPORTS", "LIB_PATH"]
