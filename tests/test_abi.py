"""The C ABI without a GPU: the library loads, exports every entry point include/ssm.h declares,
and rejects bad arguments on the host (before any CUDA call) with the documented status codes."""
import ctypes
import os
import re

import pytest

from selective_state_space_139_b300 import build, ssm

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return ssm.load_library()


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "ssm.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S).replace("SSM_API", "")
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z_0-9]*\s*\*?\s*([a-z_][a-z_0-9]*)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n.startswith("ssm_")))


def test_every_declared_symbol_is_exported(lib):
    names = _declared_functions()
    assert "ssm_scan_fwd" in names and "ssm_state_update" in names and len(names) >= 9
    for n in names:
        assert hasattr(lib, n), f"{n} declared in ssm.h but not exported"


def test_version_and_status_strings(lib):
    assert lib.ssm_abi_version() == 1
    assert lib.ssm_status_string(0) == b"SSM_OK"
    assert lib.ssm_status_string(2) == b"SSM_ERR_UNSUPPORTED"


# Fake device addresses: validation never dereferences them.
P = 0x7f0000000000


def _scan(lib, **kw):
    a = dict(u=P, delta=P + 0x10000000, A=P + 0x20000000, B=P + 0x30000000, C=P + 0x40000000, D=None, z=None,
             bias=None, softplus=1, y=P + 0x50000000, last=None, batch=2, dim=8, dstate=16, seqlen=64, io=ssm.SSM_BF16,
             ws=None, wsb=0, opts=None, stream=None)
    a.update(kw)
    return lib.ssm_scan_fwd_ex(a["u"], a["delta"], a["A"], a["B"], a["C"], a["D"], a["z"], a["bias"], a["softplus"],
                               a["y"], a["last"], a["batch"], a["dim"], a["dstate"], a["seqlen"], a["io"], a["ws"],
                               a["wsb"], a["opts"], a["stream"])


def test_scan_rejects_bad_arguments_on_host(lib):
    assert _scan(lib, dstate=17) == ssm.SSM_ERR_UNSUPPORTED
    assert _scan(lib, dstate=0) == ssm.SSM_ERR_INVALID_ARG
    assert _scan(lib, batch=0) == ssm.SSM_ERR_INVALID_ARG
    assert _scan(lib, seqlen=-1) == ssm.SSM_ERR_INVALID_ARG
    assert _scan(lib, io=7) == ssm.SSM_ERR_INVALID_ARG
    assert _scan(lib, u=None) == ssm.SSM_ERR_INVALID_ARG
    assert _scan(lib, y=None) == ssm.SSM_ERR_INVALID_ARG
    assert _scan(lib, u=P + 1) == ssm.SSM_ERR_INVALID_ARG                 # misaligned bf16
    assert _scan(lib, A=P + 0x20000002) == ssm.SSM_ERR_INVALID_ARG        # misaligned float32
    assert _scan(lib, y=P + 0x10) == ssm.SSM_ERR_INVALID_ARG              # y overlaps u
    assert b"overlaps" in lib.ssm_last_error_message()
    bad = ssm.ScanOptions()
    bad.struct_size = 3
    assert _scan(lib, opts=ctypes.pointer(bad)) == ssm.SSM_ERR_INVALID_ARG
    o = ssm.ScanOptions()
    o.struct_size = ctypes.sizeof(ssm.ScanOptions)
    o.algorithm = 2
    o.chunk_len = 100                                                     # not a multiple of 64
    assert _scan(lib, opts=ctypes.pointer(o)) == ssm.SSM_ERR_INVALID_ARG
    o.chunk_len = 64
    assert _scan(lib, seqlen=256, opts=ctypes.pointer(o)) == ssm.SSM_ERR_INVALID_ARG   # chunked needs a workspace
    assert b"workspace" in lib.ssm_last_error_message()
    o.discretization = 5
    o.chunk_len = 0
    o.algorithm = 1
    assert _scan(lib, opts=ctypes.pointer(o)) == ssm.SSM_ERR_INVALID_ARG


def test_workspace_query(lib):
    o = ssm.ScanOptions()
    o.struct_size = ctypes.sizeof(ssm.ScanOptions)
    o.algorithm = 2
    o.chunk_len = 64
    n = lib.ssm_scan_fwd_workspace_size_ex(2, 8, 16, 64 * 5, ssm.SSM_BF16, ctypes.pointer(o))
    per_chunk = 2 * 8 * 16 * 4
    # aggregates P and Q for the first 4 chunks, carried-in states for all 5 chunks
    assert n == per_chunk * (4 + 4 + 5)
    o.algorithm = 1
    assert lib.ssm_scan_fwd_workspace_size_ex(2, 8, 16, 64 * 5, ssm.SSM_BF16, ctypes.pointer(o)) == 0
    assert lib.ssm_scan_fwd_workspace_size(2, 8, 17, 64, ssm.SSM_BF16) == 0


def _upd(lib, **kw):
    a = dict(x=P, dl=P + 0x1000000, A=P + 0x2000000, B=P + 0x3000000, C=P + 0x4000000, D=None, z=None,
             state=P + 0x5000000, cs=P + 0x6000000, w=P + 0x7000000, bias=None, softplus=1, y=P + 0x8000000,
             batch=2, dim=8, dstate=16, dconv=4, io=ssm.SSM_BF16, stream=None)
    a.update(kw)
    return lib.ssm_state_update(a["x"], a["dl"], a["A"], a["B"], a["C"], a["D"], a["z"], a["state"], a["cs"], a["w"],
                                a["bias"], a["softplus"], a["y"], a["batch"], a["dim"], a["dstate"], a["dconv"],
                                a["io"], a["stream"])


def test_state_update_rejects_bad_arguments_on_host(lib):
    assert _upd(lib, dconv=3) == ssm.SSM_ERR_UNSUPPORTED
    assert _upd(lib, dstate=32) == ssm.SSM_ERR_UNSUPPORTED
    assert _upd(lib, state=None) == ssm.SSM_ERR_INVALID_ARG
    assert _upd(lib, cs=None) == ssm.SSM_ERR_INVALID_ARG
    assert _upd(lib, x=P + 1) == ssm.SSM_ERR_INVALID_ARG
    assert _upd(lib, y=P + 0x5000000) == ssm.SSM_ERR_INVALID_ARG          # y aliases state
    assert _upd(lib, state=P + 0x2000000) == ssm.SSM_ERR_INVALID_ARG      # state aliases A


def test_conv1d_rejects_bad_arguments_on_host(lib):
    f = lib.ssm_causal_conv1d_fwd
    assert f(P, P + 0x1000000, None, P + 0x2000000, None, 2, 8, 64, 3, 1, ssm.SSM_BF16, None) == ssm.SSM_ERR_UNSUPPORTED
    assert f(P, None, None, P + 0x2000000, None, 2, 8, 64, 4, 1, ssm.SSM_BF16, None) == ssm.SSM_ERR_INVALID_ARG
    assert f(P, P + 0x1000000, None, P + 0x10, None, 2, 8, 64, 4, 1, ssm.SSM_BF16, None) == ssm.SSM_ERR_INVALID_ARG
    assert f(P + 1, P + 0x1000000, None, P + 0x2000000, None, 2, 8, 64, 4, 1, ssm.SSM_BF16, None) == ssm.SSM_ERR_INVALID_ARG
    # the outgoing state may not alias the incoming one
    assert f(P, P + 0x1000000, P + 0x3000000, P + 0x2000000, P + 0x3000000, 2, 8, 64, 4, 1, ssm.SSM_BF16,
             None) == ssm.SSM_ERR_INVALID_ARG


def _bwd(lib, **kw):
    a = dict(u=P, delta=P + 0x1000000, A=P + 0x2000000, B=P + 0x3000000, C=P + 0x4000000, D=None, z=None, bias=None,
             softplus=1, dy=P + 0x5000000, du=P + 0x6000000, dd=P + 0x7000000, dz=None, dA=P + 0x8000000,
             dB=P + 0x9000000, dC=P + 0xa000000, dD=None, dbias=None, batch=2, dim=8, dstate=16, seqlen=64,
             io=ssm.SSM_BF16, ws=P + 0x10000000, wsb=1 << 24, stream=None)
    a.update(kw)
    return lib.ssm_scan_bwd(a["u"], a["delta"], a["A"], a["B"], a["C"], a["D"], a["z"], a["bias"], a["softplus"],
                            a["dy"], a["du"], a["dd"], a["dz"], a["dA"], a["dB"], a["dC"], a["dD"], a["dbias"],
                            a["batch"], a["dim"], a["dstate"], a["seqlen"], a["io"], a["ws"], a["wsb"], a["stream"])


def test_scan_bwd_rejects_bad_arguments_on_host(lib):
    assert _bwd(lib, dstate=17) == ssm.SSM_ERR_UNSUPPORTED
    assert _bwd(lib, batch=0) == ssm.SSM_ERR_INVALID_ARG
    assert _bwd(lib, io=5) == ssm.SSM_ERR_INVALID_ARG
    assert _bwd(lib, dy=None) == ssm.SSM_ERR_INVALID_ARG
    assert _bwd(lib, dA=None) == ssm.SSM_ERR_INVALID_ARG
    assert _bwd(lib, z=P + 0xb000000) == ssm.SSM_ERR_INVALID_ARG                    # z without dz
    assert _bwd(lib, dz=P + 0xb000000) == ssm.SSM_ERR_INVALID_ARG                   # dz without z
    assert _bwd(lib, du=P + 1) == ssm.SSM_ERR_INVALID_ARG                           # misaligned
    assert _bwd(lib, du=P + 0x10) == ssm.SSM_ERR_INVALID_ARG                        # du overlaps u
    assert _bwd(lib, dB=P + 0xa000010) == ssm.SSM_ERR_INVALID_ARG                   # dB overlaps dC
    assert _bwd(lib, wsb=16) == ssm.SSM_ERR_INVALID_ARG                             # short workspace
    assert _bwd(lib, ws=P + 0x10000010) == ssm.SSM_ERR_INVALID_ARG                  # unaligned workspace
    assert _bwd(lib, ws=P + 0x400) == ssm.SSM_ERR_INVALID_ARG                       # workspace overlaps u


def test_scan_bwd_workspace_query(lib):
    # bf16, one 64-step chunk: per channel 8 float checkpoints of 16 states and a Δ sum, and one
    # 48-float chunk aggregate (each region rounded up to 256 bytes)
    assert lib.ssm_scan_bwd_workspace_size(2, 8, 16, 64, ssm.SSM_BF16) == 2 * 8 * 8 * 16 * 4 + 512 + 2 * 8 * 48 * 4
    assert lib.ssm_scan_bwd_workspace_size(2, 8, 16, 0, ssm.SSM_BF16) == 0
    assert lib.ssm_scan_bwd_workspace_size(2, 8, 17, 64, ssm.SSM_BF16) == 0
    # float32: double checkpoints plus double accumulators
    assert lib.ssm_scan_bwd_workspace_size(1, 128, 16, 64, ssm.SSM_F32) >= 128 * 8 * 16 * 8 + 2 * 16 * 64 * 8


def test_ssd_rejects_bad_arguments_on_host(lib):
    f = lib.ssm_ssd_fwd
    base = dict(x=P, dt=P + 0x1000000, A=P + 0x2000000, B=P + 0x3000000, C=P + 0x4000000, D=None, bias=None, sp=1,
                h0=None, y=P + 0x5000000, hT=None, batch=2, L=64, H=4, hd=64, N=128, G=1, io=ssm.SSM_BF16)

    def call(**kw):
        a = dict(base)
        a.update(kw)
        return f(a["x"], a["dt"], a["A"], a["B"], a["C"], a["D"], a["bias"], a["sp"], a["h0"], a["y"], a["hT"],
                 a["batch"], a["L"], a["H"], a["hd"], a["N"], a["G"], a["io"], None)
    assert call(io=ssm.SSM_F32) == ssm.SSM_ERR_UNSUPPORTED
    assert call(hd=32) == ssm.SSM_ERR_UNSUPPORTED
    assert call(N=64) == ssm.SSM_ERR_UNSUPPORTED
    assert call(G=3) == ssm.SSM_ERR_INVALID_ARG          # 4 heads do not split into 3 groups
    assert call(H=0) == ssm.SSM_ERR_INVALID_ARG
    assert call(x=P + 8) == ssm.SSM_ERR_INVALID_ARG      # not 16-byte aligned
    assert call(y=P + 0x100) == ssm.SSM_ERR_INVALID_ARG  # y overlaps x
    assert call(dt=None) == ssm.SSM_ERR_INVALID_ARG
    assert call(hT=P + 0x5000004) == ssm.SSM_ERR_INVALID_ARG   # misaligned final state


def test_ssd_state_update_rejects_bad_arguments_on_host(lib):
    f = lib.ssm_ssd_state_update
    base = dict(x=P, dt=P + 0x100000, A=P + 0x200000, B=P + 0x300000, C=P + 0x400000, D=None, bias=None, sp=1,
                st=P + 0x1000000, y=P + 0x500000, batch=2, H=4, hd=64, N=128, G=1, io=ssm.SSM_BF16)

    def call(**kw):
        a = dict(base)
        a.update(kw)
        return f(a["x"], a["dt"], a["A"], a["B"], a["C"], a["D"], a["bias"], a["sp"], a["st"], a["y"], a["batch"],
                 a["H"], a["hd"], a["N"], a["G"], a["io"], None)
    assert call(io=ssm.SSM_F32) == ssm.SSM_ERR_UNSUPPORTED
    assert call(N=16) == ssm.SSM_ERR_UNSUPPORTED
    assert call(G=3) == ssm.SSM_ERR_INVALID_ARG
    assert call(st=None) == ssm.SSM_ERR_INVALID_ARG
    assert call(st=P + 0x1000008) == ssm.SSM_ERR_INVALID_ARG   # state not 16-byte aligned
    assert call(y=P + 0x1000000) == ssm.SSM_ERR_INVALID_ARG    # y overlaps the state


def test_selftest_rejects_unknown_wait_kind_on_host(lib):
    assert lib.ssm_selftest_bounded_wait(2, 1000000, None) == ssm.SSM_ERR_INVALID_ARG
    assert lib.ssm_selftest_bounded_wait(-1, 1000000, None) == ssm.SSM_ERR_INVALID_ARG


def test_checked_build_exports_the_same_entry_points(lib):
    """libssm_b300_check.so (-DSSM_CHECK=1) is a drop-in for the ordinary library."""
    build.build(checked=True)
    chk = ssm.load_library(build.LIB_CHECK)
    for n in _declared_functions():
        assert hasattr(chk, n), f"{n} declared in ssm.h but not exported by the checked build"
    assert lib.ssm_checked_build() == 0
    assert chk.ssm_checked_build() == 1
    assert chk.ssm_status_string(ssm.SSM_ERR_CHECK) == b"SSM_ERR_CHECK"


def test_index_check_selftest_needs_the_checked_build(lib):
    # the ordinary build has no checks to exercise: refused before any CUDA call
    assert lib.ssm_selftest_index_check(None) == ssm.SSM_ERR_UNSUPPORTED
