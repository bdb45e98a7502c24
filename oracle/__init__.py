"""Plain fp64 CPU oracle for the selective state-space scan (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import this package.  It shares no code with the CUDA implementation: the arithmetic lives in
``ssm_oracle.c`` (plain C, double precision, one channel at a time in the pages' order) and
this module only converts numpy arrays and calls it.

What it computes (page title, section):

* ``selective_scan`` -- the sequential selective recurrence of "Mamba и State Space Models",
  "Selective Scan (core algorithm)": Δ = softplus(Δ_raw + bias), h_t = exp(Δ_t A) ⊙ h_{t-1}
  + Δ_t B_t x_t, y_t = C_t·h_t, plus the D skip and the SiLU gate of "State Space Models: Mamba
  и альтернатива Transformer", "Mamba: Selective State Space".  ``discretization="zoh"``
  replaces the input term by the exact zero-order hold of "Модуль 8. Альтернативы
  Transformer", §4.
* ``chunked_scan`` -- the same operator through per-chunk affine aggregates and a carry
  ("Модуль 8", §7); pinned against the sequential form.
* ``causal_conv1d`` -- the depthwise causal conv (width K, K-1 leading pad values) with SiLU.
* ``state_update`` -- one decode step with the conv cache and the SSM cache ("Модуль 8", §6, §14).
* ``compose_affine`` -- (a2, b2) ∘ (a1, b1) = (a2 a1, a2 b1 + b2), "later after earlier".
* ``scan_backward`` -- gradients of sum(dy * y) by reverse-mode differentiation of the recurrence
  (the pages' hardware-aware scan recomputes states for its backward; here the plain form).
* ``ssd_scan`` -- Mamba-2 state space duality: a scalar decay per head and a (headdim, dstate) state
  ("Mamba и State Space Models", "Mamba-2: State Space Duality (SSD)"; "Модуль 8", §7, §14), as the
  recurrence and as the chunked block form.

Pins: every function is checked in ``tests/test_oracle_pins.py`` against closed forms, brute
force and the pages' worked examples (see the test module's docstring for the list).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ssm_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libssm_oracle.so")
_lib = None

_D = ctypes.POINTER(ctypes.c_double)
_I64 = ctypes.POINTER(ctypes.c_int64)


def build(force: bool = False) -> str:
    """Compile ``ssm_oracle.c`` with gcc (-O2, no fast-math, no FMA contraction)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    cmd = ["gcc", "-O2", "-std=c99", "-D_POSIX_C_SOURCE=200809L", "-fno-fast-math", "-ffp-contract=off",
           "-fPIC", "-shared", "-pthread", "-o", _LIB_PATH + ".tmp", _SRC, "-lm"]
    subprocess.check_call(cmd)
    os.replace(_LIB_PATH + ".tmp", _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        scan_args = [_D, _D, _D, _D, _D, _D, _D, _D, ctypes.c_int, ctypes.c_int, _D, _I64, _D, _D,
                     ctypes.c_int64, ctypes.c_int, ctypes.c_int64]
        lib.oracle_selective_scan.argtypes = scan_args + [ctypes.c_int]
        lib.oracle_selective_scan.restype = ctypes.c_int
        lib.oracle_chunked_scan.argtypes = scan_args + [ctypes.c_int64, ctypes.c_int]
        lib.oracle_chunked_scan.restype = ctypes.c_int
        lib.oracle_causal_conv1d.argtypes = [_D, _D, _D, _D, _D, ctypes.c_int64, ctypes.c_int64,
                                             ctypes.c_int, ctypes.c_int]
        lib.oracle_causal_conv1d.restype = ctypes.c_int
        lib.oracle_state_update.argtypes = [_D, _D, _D, _D, _D, _D, _D, _D, ctypes.c_int, _D, _D, _D,
                                            _D, _I64, ctypes.c_int64, ctypes.c_int, ctypes.c_int]
        lib.oracle_state_update.restype = ctypes.c_int
        lib.oracle_scan_backward.argtypes = [_D, _D, _D, _D, _D, _D, _D, _D, ctypes.c_int, _D, _I64, _D, _D, _D, _D,
                                             _D, _D, _D, _D, _D, ctypes.c_int64, ctypes.c_int, ctypes.c_int64,
                                             ctypes.c_int]
        lib.oracle_scan_backward.restype = ctypes.c_int
        lib.oracle_ssd_scan.argtypes = [_D] * 7 + [ctypes.c_int, _D, _D, _D, ctypes.c_int64, ctypes.c_int64,
                                                   ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                   ctypes.c_int64, ctypes.c_int]
        lib.oracle_ssd_scan.restype = ctypes.c_int
        lib.oracle_compose_affine.argtypes = [ctypes.c_double] * 4 + [_D, _D]
        lib.oracle_compose_affine.restype = None
        _lib = lib
    return _lib


def _f64(a, shape=None) -> Optional[np.ndarray]:
    if a is None:
        return None
    a = np.ascontiguousarray(np.asarray(a, dtype=np.float64))
    if shape is not None and a.shape != tuple(shape):
        raise ValueError(f"expected shape {tuple(shape)}, got {a.shape}")
    return a


def _p(a):
    return None if a is None else a.ctypes.data_as(_D)


_DISC = {"delta_b": 0, "zoh": 1}


def compose_affine(later: Tuple[float, float], earlier: Tuple[float, float]) -> Tuple[float, float]:
    """(a2, b2) ∘ (a1, b1): apply ``earlier`` first, then ``later``."""
    a, b = ctypes.c_double(), ctypes.c_double()
    _load().oracle_compose_affine(float(later[0]), float(later[1]), float(earlier[0]), float(earlier[1]),
                                  ctypes.byref(a), ctypes.byref(b))
    return a.value, b.value


def selective_scan_channels(u, delta, A, B, C, bidx, D=None, z=None, delta_bias=None,
                            delta_softplus: bool = True, h0=None, discretization: str = "delta_b",
                            chunk: Optional[int] = None, threads: int = 0):
    """Channel-list form: per-channel rows ``u, delta, z`` (n, L), ``A`` (n, N), ``D, delta_bias`` (n),
    ``h0`` (n, N); ``B, C`` keep their (batch, N, L) layout and ``bidx`` (n) names each channel's batch.

    Returns ``(y (n, L), last_state (n, N))`` in float64.  ``chunk`` selects the chunked form.
    """
    u = _f64(u)
    n, L = u.shape
    A = _f64(A)
    N = A.shape[1]
    delta = _f64(delta, (n, L))
    A = _f64(A, (n, N))
    B = _f64(B)
    C = _f64(C, B.shape)
    if B.ndim != 3 or B.shape[1] != N or B.shape[2] != L:
        raise ValueError("B, C must be (batch, N, L)")
    bidx = np.ascontiguousarray(np.asarray(bidx, dtype=np.int64))
    if bidx.shape != (n,) or (n and (bidx.min() < 0 or bidx.max() >= B.shape[0])):
        raise ValueError("bad bidx")
    D = _f64(D, (n,))
    z = _f64(z, (n, L))
    delta_bias = _f64(delta_bias, (n,))
    h0 = _f64(h0, (n, N))
    y = np.empty((n, L), dtype=np.float64)
    hL = np.empty((n, N), dtype=np.float64)
    lib = _load()
    args = [_p(u), _p(delta), _p(A), _p(B), _p(C), _p(D), _p(z), _p(delta_bias), int(bool(delta_softplus)),
            _DISC[discretization], _p(h0), bidx.ctypes.data_as(_I64), _p(y), _p(hL), n, N, L]
    if chunk is None:
        rc = lib.oracle_selective_scan(*args, threads)
    else:
        rc = lib.oracle_chunked_scan(*args, int(chunk), threads)
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    return y, hL


def _expand(u, A, D, delta_bias, z, h0):
    batch, dim, L = u.shape
    n = batch * dim
    A_c = np.broadcast_to(np.asarray(A, dtype=np.float64), (batch,) + np.shape(A)).reshape(n, -1)
    D_c = None if D is None else np.broadcast_to(np.asarray(D, dtype=np.float64), (batch, dim)).reshape(n)
    b_c = None if delta_bias is None else np.broadcast_to(np.asarray(delta_bias, dtype=np.float64),
                                                          (batch, dim)).reshape(n)
    z_c = None if z is None else np.asarray(z, dtype=np.float64).reshape(n, L)
    h_c = None if h0 is None else np.asarray(h0, dtype=np.float64).reshape(n, -1)
    bidx = np.repeat(np.arange(batch, dtype=np.int64), dim)
    return A_c, D_c, b_c, z_c, h_c, bidx


def selective_scan(u, delta, A, B, C, D=None, z=None, delta_bias=None, delta_softplus: bool = True,
                   h0=None, discretization: str = "delta_b", threads: int = 0):
    """Full-tensor form: ``u, delta, z`` (batch, dim, L); ``A`` (dim, N); ``B, C`` (batch, N, L);
    ``D, delta_bias`` (dim); ``h0`` (batch, dim, N).  Returns ``y`` (batch, dim, L) and
    ``last_state`` (batch, dim, N), float64."""
    u = np.asarray(u, dtype=np.float64)
    batch, dim, L = u.shape
    A_c, D_c, b_c, z_c, h_c, bidx = _expand(u, A, D, delta_bias, z, h0)
    y, hL = selective_scan_channels(u.reshape(batch * dim, L), np.asarray(delta, np.float64).reshape(batch * dim, L),
                                    A_c, B, C, bidx, D=D_c, z=z_c, delta_bias=b_c,
                                    delta_softplus=delta_softplus, h0=h_c, discretization=discretization,
                                    threads=threads)
    return y.reshape(batch, dim, L), hL.reshape(batch, dim, -1)


def chunked_scan(u, delta, A, B, C, chunk: int, D=None, z=None, delta_bias=None, delta_softplus: bool = True,
                 h0=None, discretization: str = "delta_b", threads: int = 0):
    """Full-tensor form of the chunked (aggregate, carry, re-run) scan."""
    u = np.asarray(u, dtype=np.float64)
    batch, dim, L = u.shape
    A_c, D_c, b_c, z_c, h_c, bidx = _expand(u, A, D, delta_bias, z, h0)
    y, hL = selective_scan_channels(u.reshape(batch * dim, L), np.asarray(delta, np.float64).reshape(batch * dim, L),
                                    A_c, B, C, bidx, D=D_c, z=z_c, delta_bias=b_c,
                                    delta_softplus=delta_softplus, h0=h_c, discretization=discretization,
                                    chunk=chunk, threads=threads)
    return y.reshape(batch, dim, L), hL.reshape(batch, dim, -1)


def causal_conv1d(x, w, state=None, silu: bool = True):
    """Depthwise causal conv over rows of ``x`` (n, L) with weights ``w`` (n, K) and optional
    initial pad ``state`` (n, K-1), oldest first.  Returns ``(out (n, L), state_out (n, K-1))``."""
    x = _f64(x)
    n, L = x.shape
    w = _f64(w)
    K = w.shape[1]
    w = _f64(w, (n, K))
    state = _f64(state, (n, K - 1))
    out = np.empty((n, L), dtype=np.float64)
    st = np.empty((n, K - 1), dtype=np.float64)
    rc = _load().oracle_causal_conv1d(_p(x), _p(w), _p(state), _p(out), _p(st), n, L, K, int(bool(silu)))
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    return out, st


def state_update(x_t, delta_t, A, B_t, C_t, bidx, state, conv_state, conv_w, D=None, z_t=None,
                 delta_bias=None, delta_softplus: bool = True):
    """One decode step over channels: ``x_t, delta_t, z_t, D, delta_bias`` (n); ``A`` (n, N);
    ``B_t, C_t`` (batch, N); ``state`` (n, N); ``conv_state`` (n, K-1); ``conv_w`` (n, K).
    Returns ``(y_t, new_state, new_conv_state)``; the inputs are not modified."""
    x_t = _f64(x_t)
    n = x_t.shape[0]
    A = _f64(A)
    N = A.shape[1]
    conv_w = _f64(conv_w)
    K = conv_w.shape[1]
    st = np.array(_f64(state, (n, N)), copy=True)
    cs = np.array(_f64(conv_state, (n, K - 1)), copy=True)
    B_t = _f64(B_t)
    C_t = _f64(C_t, B_t.shape)
    bidx = np.ascontiguousarray(np.asarray(bidx, dtype=np.int64))
    y = np.empty(n, dtype=np.float64)
    delta_t = _f64(delta_t, (n,))
    A = _f64(A, (n, N))
    D = _f64(D, (n,))
    z_t = _f64(z_t, (n,))
    delta_bias = _f64(delta_bias, (n,))
    conv_w = _f64(conv_w, (n, K))
    rc = _load().oracle_state_update(_p(x_t), _p(delta_t), _p(A), _p(B_t), _p(C_t), _p(D), _p(z_t),
                                     _p(delta_bias), int(bool(delta_softplus)), _p(st), _p(cs), _p(conv_w),
                                     _p(y), bidx.ctypes.data_as(_I64), n, N, K)
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    return y, st, cs


def scan_backward_channels(u, delta, A, B, C, bidx, dy, D=None, z=None, delta_bias=None,
                           delta_softplus: bool = True, h0=None, threads: int = 0, block: int = 512):
    """Backward in channel-list form: rows ``u, delta, dy, z`` (n, L), ``A`` (n, N), ``D, delta_bias``
    (n), ``h0`` (n, N), channel c reading ``B[bidx[c]], C[bidx[c]]`` (batch, N, L).  Returns per-channel
    du, ddelta, dz (n, L), dA (n, N), dD, ddelta_bias (n), and dB, dC (batch, N, L) summed over the listed
    channels of each batch row.  Channels are processed ``block`` at a time to bound memory."""
    uu = np.ascontiguousarray(u, dtype=np.float64)
    n, L = uu.shape
    B = _f64(B)
    C = _f64(C)
    batch, N = B.shape[0], B.shape[1]
    A = np.ascontiguousarray(A, dtype=np.float64)
    dl = np.ascontiguousarray(delta, dtype=np.float64)
    dyc = np.ascontiguousarray(dy, dtype=np.float64)
    bidx = np.ascontiguousarray(bidx, dtype=np.int64)
    opt = lambda a, shape: None if a is None else np.ascontiguousarray(np.asarray(a, np.float64).reshape(shape))
    D = opt(D, (n,))
    z = opt(z, (n, L))
    delta_bias = opt(delta_bias, (n,))
    h0 = opt(h0, (n, N))
    out = {"du": np.empty((n, L)), "ddelta": np.empty((n, L)), "dz": None if z is None else np.empty((n, L)),
           "dA": np.empty((n, N)), "dD": np.empty(n), "ddelta_bias": np.empty(n),
           "dB": np.zeros((batch, N, L)), "dC": np.zeros((batch, N, L))}
    for c0 in range(0, n, block):
        c1 = min(n, c0 + block)
        m = c1 - c0
        sl = lambda a: None if a is None else np.ascontiguousarray(a[c0:c1])
        dB = np.empty((m, N, L))
        dC = np.empty((m, N, L))
        du, dd, dA, dD, db = np.empty((m, L)), np.empty((m, L)), np.empty((m, N)), np.empty(m), np.empty(m)
        dz = None if z is None else np.empty((m, L))
        rc = _load().oracle_scan_backward(_p(sl(uu)), _p(sl(dl)), _p(sl(A)), _p(B), _p(C), _p(sl(D)), _p(sl(z)),
                                          _p(sl(delta_bias)), int(bool(delta_softplus)), _p(sl(h0)),
                                          sl(bidx).ctypes.data_as(_I64), _p(sl(dyc)), _p(du), _p(dd), _p(dz), _p(dA),
                                          _p(dD), _p(db), _p(dB), _p(dC), m, N, L, threads)
        if rc != 0:
            raise ValueError("oracle rejected its arguments")
        out["du"][c0:c1], out["ddelta"][c0:c1], out["dA"][c0:c1] = du, dd, dA
        out["dD"][c0:c1], out["ddelta_bias"][c0:c1] = dD, db
        if dz is not None:
            out["dz"][c0:c1] = dz
        bb = bidx[c0:c1]
        for b in np.unique(bb):
            out["dB"][b] += dB[bb == b].sum(0)
            out["dC"][b] += dC[bb == b].sum(0)
    return out


def scan_backward(u, delta, A, B, C, dy, D=None, z=None, delta_bias=None, delta_softplus: bool = True, h0=None,
                  threads: int = 0):
    """Gradients of sum(dy * y) for the full-tensor scan (Δ·B input term).  Shapes as in
    ``selective_scan``; returns a dict with du, ddelta, dz (batch, dim, L), dA (dim, N), dB, dC
    (batch, N, L), dD, ddelta_bias (dim), summed over the batch where a parameter is shared."""
    u = np.asarray(u, dtype=np.float64)
    batch, dim, L = u.shape
    A_c, D_c, b_c, z_c, h_c, bidx = _expand(u, A, D, delta_bias, z, h0)
    n = batch * dim
    g = scan_backward_channels(u.reshape(n, L), np.asarray(delta, np.float64).reshape(n, L), A_c, B, C, bidx,
                               np.asarray(dy, np.float64).reshape(n, L), D=D_c, z=z_c, delta_bias=b_c,
                               delta_softplus=delta_softplus, h0=h_c, threads=threads)
    N = g["dA"].shape[1]
    return {"du": g["du"].reshape(batch, dim, L), "ddelta": g["ddelta"].reshape(batch, dim, L),
            "dz": None if g["dz"] is None else g["dz"].reshape(batch, dim, L),
            "dA": g["dA"].reshape(batch, dim, N).sum(0), "dD": g["dD"].reshape(batch, dim).sum(0),
            "ddelta_bias": g["ddelta_bias"].reshape(batch, dim).sum(0), "dB": g["dB"], "dC": g["dC"]}


def ssd_scan(x, dt, A, B, C, D=None, dt_bias=None, dt_softplus: bool = True, h0=None, chunk: Optional[int] = None,
             threads: int = 0):
    """Mamba-2 SSD with a scalar decay per head.  ``x`` (batch, L, nheads, headdim); ``dt`` (batch, L,
    nheads) before bias and softplus; ``A, D, dt_bias`` (nheads); ``B, C`` (batch, L, ngroups, dstate);
    ``h0`` (batch, nheads, headdim, dstate).  ``chunk=None`` runs the recurrence, an integer the
    chunked block form.  Returns ``y`` (batch, L, nheads, headdim) and the final state, float64."""
    x = _f64(x)
    batch, L, nheads, headdim = x.shape
    B = _f64(B)
    ngroups, dstate = B.shape[2], B.shape[3]
    dt = _f64(dt, (batch, L, nheads))
    A = _f64(A, (nheads,))
    B = _f64(B, (batch, L, ngroups, dstate))
    C = _f64(C, (batch, L, ngroups, dstate))
    D = _f64(D, (nheads,))
    dt_bias = _f64(dt_bias, (nheads,))
    h0 = _f64(h0, (batch, nheads, headdim, dstate))
    y = np.empty((batch, L, nheads, headdim))
    hT = np.empty((batch, nheads, headdim, dstate))
    rc = _load().oracle_ssd_scan(_p(x), _p(dt), _p(A), _p(B), _p(C), _p(D), _p(dt_bias), int(bool(dt_softplus)),
                                 _p(h0), _p(y), _p(hT), batch, L, nheads, headdim, dstate, ngroups,
                                 int(chunk or 0), threads)
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    return y, hT
