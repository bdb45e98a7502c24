"""Thin Python binding over libssm_b300.so (C ABI in include/ssm.h).

Argument marshalling only: every step of the scan and the decode step runs in the library's CUDA
kernels.  PyTorch supplies device memory and the current stream.  There is no CPU fallback: if the
library is missing or a tensor is not on a CUDA device, the call raises.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
from typing import Iterator, Optional, Tuple

import torch

from . import build as _build

SSM_OK, SSM_ERR_INVALID_ARG, SSM_ERR_UNSUPPORTED, SSM_ERR_CUDA, SSM_ERR_TIMEOUT, SSM_ERR_CHECK = range(6)
SSM_F32, SSM_BF16 = 0, 1
ALGORITHMS = {"auto": 0, "single_pass": 1, "chunked": 2}
DISCRETIZATIONS = {"delta_b": 0, "zoh": 1}

_lib = None


class SSMError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{_status_name(status)}: {message}")
        self.status = status


class ScanOptions(ctypes.Structure):
    _fields_ = [("struct_size", ctypes.c_int), ("algorithm", ctypes.c_int), ("chunk_len", ctypes.c_int64),
                ("discretization", ctypes.c_int), ("h0", ctypes.c_void_p)]


class ScanPlan(ctypes.Structure):
    _fields_ = [("struct_size", ctypes.c_int), ("path", ctypes.c_int), ("schedule", ctypes.c_int),
                ("nchunks", ctypes.c_int), ("chunk_len", ctypes.c_int64), ("ctas", ctypes.c_int),
                ("kernel_launches", ctypes.c_int), ("workspace_bytes", ctypes.c_size_t)]


def library_path() -> str:
    return _build.LIB


def load_library(path: Optional[str] = None) -> ctypes.CDLL:
    """Loads the in-tree library (built beforehand by ``build.py``); raises if it is missing."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    path = path or _build.LIB
    if not os.path.exists(path):
        raise ImportError(f"libssm_b300.so not found at {path}; build it with "
                          f"`python -m selective_state_space_139_b300.build`")
    lib = ctypes.CDLL(path)
    vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
    lib.ssm_abi_version.restype = i32
    lib.ssm_abi_version.argtypes = []
    lib.ssm_checked_build.restype = i32
    lib.ssm_checked_build.argtypes = []
    lib.ssm_status_string.restype = ctypes.c_char_p
    lib.ssm_status_string.argtypes = [i32]
    lib.ssm_last_error_message.restype = ctypes.c_char_p
    lib.ssm_last_error_message.argtypes = []
    lib.ssm_scan_fwd_workspace_size.restype = sz
    lib.ssm_scan_fwd_workspace_size.argtypes = [i32, i32, i32, i64, i32]
    lib.ssm_scan_fwd_workspace_size_ex.restype = sz
    lib.ssm_scan_fwd_workspace_size_ex.argtypes = [i32, i32, i32, i64, i32, ctypes.POINTER(ScanOptions)]
    scan = [vp, vp, vp, vp, vp, vp, vp, vp, i32, vp, vp, i32, i32, i32, i64, i32, vp, sz]
    lib.ssm_scan_fwd.restype = i32
    lib.ssm_scan_fwd.argtypes = scan + [vp]
    lib.ssm_scan_fwd_ex.restype = i32
    lib.ssm_scan_fwd_ex.argtypes = scan + [ctypes.POINTER(ScanOptions), vp]
    lib.ssm_state_update.restype = i32
    lib.ssm_state_update.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i32, vp]
    lib.ssm_selftest_bounded_wait.restype = i32
    lib.ssm_selftest_bounded_wait.argtypes = [i32, i64, vp]
    lib.ssm_selftest_withhold_carry.restype = i32
    lib.ssm_selftest_withhold_carry.argtypes = [i32, i64]
    lib.ssm_selftest_index_check.restype = i32
    lib.ssm_selftest_index_check.argtypes = [vp]
    lib.ssm_scan_fwd_describe.restype = i32
    lib.ssm_scan_fwd_describe.argtypes = [i32, i32, i32, i64, i32, ctypes.POINTER(ScanOptions), ctypes.POINTER(ScanPlan)]
    lib.ssm_causal_conv1d_fwd.restype = i32
    lib.ssm_causal_conv1d_fwd.argtypes = [vp, vp, vp, vp, vp, i32, i32, i64, i32, i32, i32, vp]
    lib.ssm_device_status.restype = i32
    lib.ssm_device_status.argtypes = [vp]
    lib.ssm_ssd_state_update.restype = i32
    lib.ssm_ssd_state_update.argtypes = [vp] * 7 + [i32, vp, vp, i32, i32, i32, i32, i32, i32, vp]
    lib.ssm_ssd_fwd.restype = i32
    lib.ssm_ssd_fwd.argtypes = [vp] * 7 + [i32, vp, vp, vp, i32, i64, i32, i32, i32, i32, i32, vp]
    lib.ssm_ssd_fwd_ex.restype = i32
    lib.ssm_ssd_fwd_ex.argtypes = [vp] * 7 + [i32, vp, vp, vp, i32, i64, i32, i32, i32, i32, i32, vp, sz, i32, vp]
    lib.ssm_ssd_fwd_workspace_size.restype = sz
    lib.ssm_ssd_fwd_workspace_size.argtypes = [i32, i64, i32, i32]
    lib.ssm_scan_bwd_workspace_size.restype = sz
    lib.ssm_scan_bwd_workspace_size.argtypes = [i32, i32, i32, i64, i32]
    lib.ssm_scan_bwd.restype = i32
    lib.ssm_scan_bwd.argtypes = [vp] * 8 + [i32] + [vp] * 9 + [i32, i32, i32, i64, i32, vp, sz, vp]
    if path == _build.LIB:
        _lib = lib
    return lib


@contextlib.contextmanager
def use_checked_library() -> Iterator[ctypes.CDLL]:
    """Routes every call in the block through the checked debug build (libssm_b300_check.so).

    Its kernels check each global index against the buffer's size; a failed check is reported by
    ``device_status()`` as SSM_ERR_CHECK instead of touching memory outside the buffer.
    """
    global _lib
    plain = load_library()
    checked = load_library(_build.LIB_CHECK)
    if checked.ssm_checked_build() != 1:
        raise ImportError(f"{_build.LIB_CHECK} is not a checked build")
    _lib = checked
    try:
        yield checked
    finally:
        _lib = plain


def _status_name(s: int) -> str:
    return {0: "SSM_OK", 1: "SSM_ERR_INVALID_ARG", 2: "SSM_ERR_UNSUPPORTED", 3: "SSM_ERR_CUDA",
            4: "SSM_ERR_TIMEOUT", 5: "SSM_ERR_CHECK"}.get(s, f"status {s}")


def _check(lib, status: int):
    if status != SSM_OK:
        raise SSMError(status, lib.ssm_last_error_message().decode(errors="replace"))


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _io_code(dtype) -> int:
    if dtype == torch.bfloat16:
        return SSM_BF16
    if dtype == torch.float32:
        return SSM_F32
    raise TypeError(f"io dtype must be bfloat16 or float32, got {dtype}")


def _need(t: Optional[torch.Tensor], name: str, shape, dtype, device, optional=False):
    if t is None:
        if optional:
            return
        raise ValueError(f"{name} is required")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (no CPU path exists)")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _stream_handle(stream) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _options(algorithm: str, chunk_len: int, discretization: str, h0: Optional[torch.Tensor]) -> ScanOptions:
    o = ScanOptions()
    o.struct_size = ctypes.sizeof(ScanOptions)
    o.algorithm = ALGORITHMS[algorithm]
    o.chunk_len = int(chunk_len)
    o.discretization = DISCRETIZATIONS[discretization]
    o.h0 = _ptr(h0)
    return o


def scan_workspace_size(batch: int, dim: int, dstate: int, seqlen: int, dtype=torch.bfloat16,
                        algorithm: str = "auto", chunk_len: int = 0, discretization: str = "delta_b") -> int:
    lib = load_library()
    o = _options(algorithm, chunk_len, discretization, None)
    return int(lib.ssm_scan_fwd_workspace_size_ex(batch, dim, dstate, seqlen, _io_code(dtype), ctypes.byref(o)))


def describe_scan(batch: int, dim: int, dstate: int, seqlen: int, dtype=torch.bfloat16, algorithm: str = "auto",
                  chunk_len: int = 0, discretization: str = "delta_b") -> dict:
    """The plan a prefill call with these sizes would run (kernel path, schedule, launches, workspace)."""
    lib = load_library()
    o = _options(algorithm, chunk_len, discretization, None)
    pl = ScanPlan()
    pl.struct_size = ctypes.sizeof(ScanPlan)
    _check(lib, lib.ssm_scan_fwd_describe(batch, dim, dstate, seqlen, _io_code(dtype), ctypes.byref(o), ctypes.byref(pl)))
    return {"path": ("general", "fast")[pl.path], "schedule": ("grid", "balanced", "chunked")[pl.schedule],
            "nchunks": pl.nchunks, "chunk_len": pl.chunk_len, "ctas": pl.ctas, "kernel_launches": pl.kernel_launches,
            "workspace_bytes": pl.workspace_bytes}


def selective_scan_fwd(u: torch.Tensor, delta: torch.Tensor, A: torch.Tensor, B: torch.Tensor, C: torch.Tensor,
                       D: Optional[torch.Tensor] = None, z: Optional[torch.Tensor] = None,
                       delta_bias: Optional[torch.Tensor] = None, delta_softplus: bool = True,
                       return_last_state: bool = True, *, algorithm: str = "auto", chunk_len: int = 0,
                       discretization: str = "delta_b", h0: Optional[torch.Tensor] = None,
                       out: Optional[torch.Tensor] = None, last_state: Optional[torch.Tensor] = None,
                       workspace: Optional[torch.Tensor] = None, stream=None
                       ) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """Prefill scan.  u, delta, z: (batch, dim, L); A: (dim, N) f32; B, C: (batch, N, L);
    D, delta_bias: (dim,) f32; h0: (batch, dim, N) f32.  Returns (y, last_state)."""
    lib = load_library()
    batch, dim, L = u.shape
    N = A.shape[1]
    dev = u.device
    io = u.dtype
    _need(u, "u", (batch, dim, L), io, dev)
    _need(delta, "delta", (batch, dim, L), io, dev)
    _need(z, "z", (batch, dim, L), io, dev, optional=True)
    _need(A, "A", (dim, N), torch.float32, dev)
    _need(B, "B", (batch, N, L), io, dev)
    _need(C, "C", (batch, N, L), io, dev)
    _need(D, "D", (dim,), torch.float32, dev, optional=True)
    _need(delta_bias, "delta_bias", (dim,), torch.float32, dev, optional=True)
    _need(h0, "h0", (batch, dim, N), torch.float32, dev, optional=True)
    y = torch.empty_like(u) if out is None else out
    _need(y, "out", (batch, dim, L), io, dev)
    if return_last_state and last_state is None:
        last_state = torch.empty((batch, dim, N), dtype=torch.float32, device=dev)
    if last_state is not None:
        _need(last_state, "last_state", (batch, dim, N), torch.float32, dev)
    o = _options(algorithm, chunk_len, discretization, h0)
    ws_bytes = int(lib.ssm_scan_fwd_workspace_size_ex(batch, dim, N, L, _io_code(io), ctypes.byref(o)))
    if ws_bytes and (workspace is None or workspace.numel() < ws_bytes):
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    with torch.cuda.device(dev):
        st = lib.ssm_scan_fwd_ex(_ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z), _ptr(delta_bias),
                                 int(bool(delta_softplus)), _ptr(y), _ptr(last_state), batch, dim, N, L, _io_code(io),
                                 _ptr(workspace) if ws_bytes else None, ws_bytes, ctypes.byref(o),
                                 _stream_handle(stream))
    _check(lib, st)
    return y, last_state


def selective_state_update(x_t: torch.Tensor, delta_t: torch.Tensor, A: torch.Tensor, B_t: torch.Tensor,
                           C_t: torch.Tensor, D: Optional[torch.Tensor], z_t: Optional[torch.Tensor],
                           state: torch.Tensor, conv_state: torch.Tensor, conv_w: torch.Tensor,
                           delta_bias: Optional[torch.Tensor] = None, delta_softplus: bool = True,
                           out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """One decode step; updates ``state`` (batch, dim, N) and ``conv_state`` (batch, dim, 3) in place.
    x_t, delta_t, z_t: (batch, dim); B_t, C_t: (batch, N); conv_w: (dim, 4) f32.  Returns y_t."""
    lib = load_library()
    batch, dim = x_t.shape
    N = A.shape[1]
    K = conv_w.shape[1]
    dev = x_t.device
    io = x_t.dtype
    _need(x_t, "x_t", (batch, dim), io, dev)
    _need(delta_t, "delta_t", (batch, dim), io, dev)
    _need(z_t, "z_t", (batch, dim), io, dev, optional=True)
    _need(A, "A", (dim, N), torch.float32, dev)
    _need(B_t, "B_t", (batch, N), io, dev)
    _need(C_t, "C_t", (batch, N), io, dev)
    _need(D, "D", (dim,), torch.float32, dev, optional=True)
    _need(delta_bias, "delta_bias", (dim,), torch.float32, dev, optional=True)
    _need(state, "state", (batch, dim, N), torch.float32, dev)
    _need(conv_state, "conv_state", (batch, dim, K - 1), torch.float32, dev)
    _need(conv_w, "conv_w", (dim, K), torch.float32, dev)
    y = torch.empty_like(x_t) if out is None else out
    _need(y, "out", (batch, dim), io, dev)
    with torch.cuda.device(dev):
        st = lib.ssm_state_update(_ptr(x_t), _ptr(delta_t), _ptr(A), _ptr(B_t), _ptr(C_t), _ptr(D), _ptr(z_t),
                                  _ptr(state), _ptr(conv_state), _ptr(conv_w), _ptr(delta_bias),
                                  int(bool(delta_softplus)), _ptr(y), batch, dim, N, K, _io_code(io),
                                  _stream_handle(stream))
    _check(lib, st)
    return y


def causal_conv1d_fwd(x: torch.Tensor, conv_w: torch.Tensor, conv_state: Optional[torch.Tensor] = None,
                      silu: bool = True, return_final_state: bool = True, out: Optional[torch.Tensor] = None,
                      final_state: Optional[torch.Tensor] = None, stream=None
                      ) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """Causal depthwise conv (width 4) + SiLU over x (batch, dim, L) with weights (dim, 4) and an optional
    incoming conv state (batch, dim, 3).  Returns (u, final conv state)."""
    lib = load_library()
    batch, dim, L = x.shape
    K = conv_w.shape[1]
    dev = x.device
    _need(x, "x", (batch, dim, L), x.dtype, dev)
    _need(conv_w, "conv_w", (dim, K), torch.float32, dev)
    _need(conv_state, "conv_state", (batch, dim, K - 1), torch.float32, dev, optional=True)
    u = torch.empty_like(x) if out is None else out
    _need(u, "out", (batch, dim, L), x.dtype, dev)
    if return_final_state and final_state is None:
        final_state = torch.empty((batch, dim, K - 1), dtype=torch.float32, device=dev)
    if final_state is not None:
        _need(final_state, "final_state", (batch, dim, K - 1), torch.float32, dev)
    with torch.cuda.device(dev):
        st = lib.ssm_causal_conv1d_fwd(_ptr(x), _ptr(conv_w), _ptr(conv_state), _ptr(u), _ptr(final_state), batch, dim, L,
                                       K, int(bool(silu)), _io_code(x.dtype), _stream_handle(stream))
    _check(lib, st)
    return u, final_state


def scan_bwd_workspace_size(batch: int, dim: int, dstate: int, seqlen: int, dtype=torch.bfloat16) -> int:
    lib = load_library()
    return int(lib.ssm_scan_bwd_workspace_size(batch, dim, dstate, seqlen, _io_code(dtype)))


def selective_scan_bwd(u: torch.Tensor, delta: torch.Tensor, A: torch.Tensor, B: torch.Tensor, C: torch.Tensor,
                       dy: torch.Tensor, D: Optional[torch.Tensor] = None, z: Optional[torch.Tensor] = None,
                       delta_bias: Optional[torch.Tensor] = None, delta_softplus: bool = True, *,
                       workspace: Optional[torch.Tensor] = None, stream=None) -> dict:
    """Gradients of sum(dy * y) for the prefill scan (zero initial state).  Returns a dict with du,
    ddelta, dz (batch, dim, L) in the io dtype (dz None without z), dA (dim, N), dB, dC (batch, N, L),
    dD and ddelta_bias (dim,) in float32 (dD / ddelta_bias None when D / delta_bias is None)."""
    lib = load_library()
    batch, dim, L = u.shape
    N = A.shape[1]
    dev = u.device
    io = u.dtype
    _need(u, "u", (batch, dim, L), io, dev)
    _need(delta, "delta", (batch, dim, L), io, dev)
    _need(z, "z", (batch, dim, L), io, dev, optional=True)
    _need(A, "A", (dim, N), torch.float32, dev)
    _need(B, "B", (batch, N, L), io, dev)
    _need(C, "C", (batch, N, L), io, dev)
    _need(dy, "dy", (batch, dim, L), io, dev)
    _need(D, "D", (dim,), torch.float32, dev, optional=True)
    _need(delta_bias, "delta_bias", (dim,), torch.float32, dev, optional=True)
    f32 = dict(dtype=torch.float32, device=dev)
    g = {"du": torch.empty_like(u), "ddelta": torch.empty_like(u),
         "dz": None if z is None else torch.empty_like(u),
         "dA": torch.empty((dim, N), **f32), "dB": torch.empty((batch, N, L), **f32),
         "dC": torch.empty((batch, N, L), **f32),
         "dD": None if D is None else torch.empty((dim,), **f32),
         "ddelta_bias": None if delta_bias is None else torch.empty((dim,), **f32)}
    ws_bytes = int(lib.ssm_scan_bwd_workspace_size(batch, dim, N, L, _io_code(io)))
    if ws_bytes and (workspace is None or workspace.numel() < ws_bytes):
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    with torch.cuda.device(dev):
        st = lib.ssm_scan_bwd(_ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z), _ptr(delta_bias),
                              int(bool(delta_softplus)), _ptr(dy), _ptr(g["du"]), _ptr(g["ddelta"]), _ptr(g["dz"]),
                              _ptr(g["dA"]), _ptr(g["dB"]), _ptr(g["dC"]), _ptr(g["dD"]), _ptr(g["ddelta_bias"]),
                              batch, dim, N, L, _io_code(io), _ptr(workspace) if ws_bytes else None, ws_bytes,
                              _stream_handle(stream))
    _check(lib, st)
    return g


def ssd_fwd(x: torch.Tensor, dt: torch.Tensor, A: torch.Tensor, B: torch.Tensor, C: torch.Tensor,
            D: Optional[torch.Tensor] = None, dt_bias: Optional[torch.Tensor] = None, dt_softplus: bool = True,
            h0: Optional[torch.Tensor] = None, return_final_state: bool = True, *, out: Optional[torch.Tensor] = None,
            final_state: Optional[torch.Tensor] = None, balanced: bool = True, ctas: int = 0,
            workspace: Optional[torch.Tensor] = None, stream=None) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """Mamba-2 SSD forward.  x (batch, L, nheads, headdim), dt (batch, L, nheads), B, C (batch, L,
    ngroups, dstate) in bf16; A, D, dt_bias (nheads,) f32; h0 (batch, nheads, headdim, dstate) f32.
    balanced: the balanced schedule of ssm_ssd_fwd_ex where it applies (ctas: at most that many ranges,
    0 = one per co-resident CTA; workspace: a uint8 device tensor reused if large enough, else one is
    allocated); False: one CTA per sequence (ssm_ssd_fwd).  Returns (y, final state)."""
    lib = load_library()
    batch, L, nheads, headdim = x.shape
    ngroups, dstate = B.shape[2], B.shape[3]
    dev = x.device
    io = x.dtype
    _need(x, "x", (batch, L, nheads, headdim), io, dev)
    _need(dt, "dt", (batch, L, nheads), io, dev)
    _need(B, "B", (batch, L, ngroups, dstate), io, dev)
    _need(C, "C", (batch, L, ngroups, dstate), io, dev)
    _need(A, "A", (nheads,), torch.float32, dev)
    _need(D, "D", (nheads,), torch.float32, dev, optional=True)
    _need(dt_bias, "dt_bias", (nheads,), torch.float32, dev, optional=True)
    _need(h0, "h0", (batch, nheads, headdim, dstate), torch.float32, dev, optional=True)
    y = torch.empty_like(x) if out is None else out
    _need(y, "out", (batch, L, nheads, headdim), io, dev)
    if return_final_state and final_state is None:
        final_state = torch.empty((batch, nheads, headdim, dstate), dtype=torch.float32, device=dev)
    if final_state is not None:
        _need(final_state, "final_state", (batch, nheads, headdim, dstate), torch.float32, dev)
    with torch.cuda.device(dev):
        ws_bytes = int(lib.ssm_ssd_fwd_workspace_size(batch, L, nheads, int(ctas))) if balanced else 0
        if ws_bytes and (workspace is None or workspace.numel() < ws_bytes):
            workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
        st = lib.ssm_ssd_fwd_ex(_ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(dt_bias),
                                int(bool(dt_softplus)), _ptr(h0), _ptr(y), _ptr(final_state), batch, L, nheads,
                                headdim, dstate, ngroups, _io_code(io), _ptr(workspace) if ws_bytes else None,
                                ws_bytes, int(ctas), _stream_handle(stream))
    _check(lib, st)
    return y, final_state


def ssd_workspace_size(batch: int, seqlen: int, nheads: int, ctas: int = 0) -> int:
    """Bytes of workspace the balanced SSD schedule needs on the current device (0: one CTA per sequence)."""
    return int(load_library().ssm_ssd_fwd_workspace_size(batch, seqlen, nheads, ctas))


def ssd_state_update(x_t: torch.Tensor, dt_t: torch.Tensor, A: torch.Tensor, B_t: torch.Tensor, C_t: torch.Tensor,
                     state: torch.Tensor, D: Optional[torch.Tensor] = None, dt_bias: Optional[torch.Tensor] = None,
                     dt_softplus: bool = True, out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """One Mamba-2 decode step; updates ``state`` (batch, nheads, headdim, dstate) f32 in place.
    x_t (batch, nheads, headdim), dt_t (batch, nheads), B_t, C_t (batch, ngroups, dstate) in bf16;
    A, D, dt_bias (nheads,) f32.  Returns y_t (batch, nheads, headdim)."""
    lib = load_library()
    batch, nheads, headdim = x_t.shape
    ngroups, dstate = B_t.shape[1], B_t.shape[2]
    dev = x_t.device
    io = x_t.dtype
    _need(x_t, "x_t", (batch, nheads, headdim), io, dev)
    _need(dt_t, "dt_t", (batch, nheads), io, dev)
    _need(B_t, "B_t", (batch, ngroups, dstate), io, dev)
    _need(C_t, "C_t", (batch, ngroups, dstate), io, dev)
    _need(A, "A", (nheads,), torch.float32, dev)
    _need(D, "D", (nheads,), torch.float32, dev, optional=True)
    _need(dt_bias, "dt_bias", (nheads,), torch.float32, dev, optional=True)
    _need(state, "state", (batch, nheads, headdim, dstate), torch.float32, dev)
    y = torch.empty_like(x_t) if out is None else out
    _need(y, "out", (batch, nheads, headdim), io, dev)
    with torch.cuda.device(dev):
        st = lib.ssm_ssd_state_update(_ptr(x_t), _ptr(dt_t), _ptr(A), _ptr(B_t), _ptr(C_t), _ptr(D), _ptr(dt_bias),
                                      int(bool(dt_softplus)), _ptr(state), _ptr(y), batch, nheads, headdim, dstate,
                                      ngroups, _io_code(io), _stream_handle(stream))
    _check(lib, st)
    return y


def device_status(stream=None) -> int:
    """Reads and clears the library's device status word (synchronises the stream)."""
    lib = load_library()
    return int(lib.ssm_device_status(_stream_handle(stream)))
