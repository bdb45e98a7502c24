"""The allocation-free prefill entry point, called through the C ABI.

ssm_scan_fwd_noalloc exists for callers that cannot allocate device memory or hand the library a
workspace (allocation forbidden or owned by someone else on their code path).  These tests call it
twice in a row through ctypes and check both results against the regular entry point's, within the
parity tolerances of the other tests (1e-2 for bf16 io, 2e-5 for float32 io).  The file is named to
be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

from selective_state_space_139_b300 import ssm
from selective_state_space_139_b300 import workloads as W
from tests._helpers import max_rel_err, to64

import oracle

pytestmark = pytest.mark.gpu


def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib = ssm.load_library()
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
    lib.ssm_scan_fwd_noalloc.restype = i32
    lib.ssm_scan_fwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i32, vp, vp, i32, i32, i32, i64, i32,
                                         ctypes.POINTER(ssm.ScanOptions), vp]
    lib.ssm_scan_fwd_noalloc_max_scratch.restype = ctypes.c_size_t
    lib.ssm_scan_fwd_noalloc_max_scratch.argtypes = []
    return lib


def _noalloc(lib, inp, y, hL, algorithm="auto", chunk_len=0):
    P = lambda t: None if t is None else t.data_ptr()
    batch, dim, L = inp["u"].shape
    N = inp["A"].shape[1]
    o = ssm._options(algorithm, chunk_len, "delta_b", None)
    io = ssm.SSM_BF16 if inp["u"].dtype == torch.bfloat16 else ssm.SSM_F32
    return lib.ssm_scan_fwd_noalloc(P(inp["u"]), P(inp["delta"]), P(inp["A"]), P(inp["B"]), P(inp["C"]), P(inp["D"]),
                                    P(inp["z"]), P(inp["delta_bias"]), 1, P(y), P(hL), batch, dim, N, L, io,
                                    ctypes.byref(o), torch.cuda.current_stream().cuda_stream)


CASES = [  # (batch, dim, dstate, L, io, algorithm): balanced, chunked and single-pass schedules
    (4, 5120, 16, 4096, "bf16", "auto"),
    (2, 256, 16, 2048, "bf16", "auto"),
    (2, 256, 16, 1000, "f32", "chunked"),
    (1, 64, 16, 256, "f32", "auto"),
]


@pytest.mark.parametrize("case", CASES)
def test_noalloc_matches_regular_entry_twice(case):
    lib = _lib()
    b, d, n, L, io, algo = case
    inp = W.random_scan_inputs(b, d, n, L, io, seed=L + d, a_scale=(0.5, 2.0), device="cuda")
    need = ssm.scan_workspace_size(b, d, n, L, inp["u"].dtype, algorithm=algo)
    assert need <= lib.ssm_scan_fwd_noalloc_max_scratch()
    y_ref, h_ref = ssm.selective_scan_fwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], D=inp["D"],
                                          z=inp["z"], delta_bias=inp["delta_bias"], algorithm=algo)
    tol = 1e-2 if io == "bf16" else 2e-5
    for _ in range(2):
        y = torch.full_like(y_ref, float("nan"))
        hL = torch.full_like(h_ref, float("nan"))
        st = _noalloc(lib, inp, y, hL, algorithm=algo)
        assert st == ssm.SSM_OK, lib.ssm_last_error_message()
        torch.cuda.synchronize()
        assert torch.isfinite(y).all() and torch.isfinite(hL).all()
        assert max_rel_err(to64(y), to64(y_ref)) <= tol
        assert max_rel_err(to64(hL), to64(h_ref)) <= tol
    assert ssm.device_status() == ssm.SSM_OK


def test_noalloc_schedules_interleaved_share_the_array():
    """Different schedules one after another on the shared array: balanced, chunked bf16, chunked
    float32, single pass, then balanced again.  Each call's scratch words are written before they
    are read in that call, so none of the earlier calls' contents may show in a result: every output
    matches the regular entry point's, and the tiny float32 case the oracle."""
    lib = _lib()
    order = [CASES[0], CASES[1], CASES[2], CASES[3], CASES[0], CASES[2], CASES[1]]
    refs = {}
    for case in order:
        b, d, n, L, io, algo = case
        if case not in refs:
            inp = W.random_scan_inputs(b, d, n, L, io, seed=L + d, a_scale=(0.5, 2.0), device="cuda")
            y_ref, h_ref = ssm.selective_scan_fwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], D=inp["D"],
                                                  z=inp["z"], delta_bias=inp["delta_bias"], algorithm=algo)
            refs[case] = (inp, y_ref, h_ref)
        inp, y_ref, h_ref = refs[case]
        y = torch.full_like(y_ref, float("nan"))
        hL = torch.full_like(h_ref, float("nan"))
        assert _noalloc(lib, inp, y, hL, algorithm=algo) == ssm.SSM_OK, lib.ssm_last_error_message()
        torch.cuda.synchronize()
        tol = 1e-2 if io == "bf16" else 2e-5
        assert max_rel_err(to64(y), to64(y_ref)) <= tol, case
        assert max_rel_err(to64(hL), to64(h_ref)) <= tol, case
        if (b, d, n, L) == (1, 64, 16, 256):
            ry, rh = oracle.selective_scan(to64(inp["u"]), to64(inp["delta"]), to64(inp["A"]), to64(inp["B"]),
                                           to64(inp["C"]), D=to64(inp["D"]), z=to64(inp["z"]),
                                           delta_bias=to64(inp["delta_bias"]))
            assert max_rel_err(to64(y), ry) <= 2e-5 and max_rel_err(to64(hL), rh) <= 2e-5
    assert ssm.device_status() == ssm.SSM_OK


def test_noalloc_refuses_shapes_beyond_its_scratch():
    lib = _lib()
    b, d, n, L = 64, 1024, 16, 4096
    need = ssm.scan_workspace_size(b, d, n, L, torch.bfloat16, algorithm="chunked", chunk_len=64)
    assert need > lib.ssm_scan_fwd_noalloc_max_scratch()
    inp = W.random_scan_inputs(1, 64, 16, 64, "bf16", seed=0, device="cuda")   # buffers are never read
    o = ssm._options("chunked", 64, "delta_b", None)
    P = lambda t: t.data_ptr()
    y = torch.empty_like(inp["u"])
    st = lib.ssm_scan_fwd_noalloc(P(inp["u"]), P(inp["delta"]), P(inp["A"]), P(inp["B"]), P(inp["C"]), None, None, None,
                                  1, P(y), None, b, d, n, L, ssm.SSM_BF16, ctypes.byref(o), None)
    assert st == ssm.SSM_ERR_UNSUPPORTED
    assert b"scratch" in lib.ssm_last_error_message()
