"""The small and ragged parity cases again, through the checked debug build (libssm_b300_check.so).

In that build every global load and store of the kernels goes through an index check against its
buffer's element count; a failed check redirects the access to a sink and makes ssm_device_status()
return SSM_ERR_CHECK (nothing traps).  Each case below must match the fp64 oracle with the same
tolerance as in the ordinary build AND leave the status word clean, so an index that strays outside
its buffer on any of these shapes (ragged tails, dstate < 16, partial channel groups, every schedule
of the prefill) fails here instead of reading or writing memory it does not own.
"""
import pytest
import torch

from selective_state_space_139_b300 import ssm
from selective_state_space_139_b300 import workloads as W
from tests._helpers import max_rel_err, to64
from tests import test_conv1d_parity as conv_t
from tests import test_decode_parity as decode_t
from tests import test_scan_bwd_parity as bwd_t
from tests import test_scan_parity as scan_t
from tests import test_ssd_parity as ssd_t

pytestmark = pytest.mark.gpu


@pytest.fixture
def checked():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    with ssm.use_checked_library() as lib:
        assert ssm.device_status() == ssm.SSM_OK
        yield lib
        assert ssm.device_status() == ssm.SSM_OK, "an index check failed"


def test_the_checks_report_a_stray_index(checked):
    # a store one past a 32-element buffer, through the check: redirected, reported once, cleared
    assert checked.ssm_selftest_index_check(None) == ssm.SSM_OK
    assert ssm.device_status() == ssm.SSM_ERR_CHECK
    assert ssm.device_status() == ssm.SSM_OK


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("shape", scan_t.SHAPES)
def test_scan_ragged_shapes(checked, shape, dtype):
    scan_t.test_ragged_shapes(shape, dtype)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_scan_options_general_A_and_zoh(checked, dtype):
    scan_t.test_optional_operands_and_softplus_off(dtype)
    scan_t.test_general_A(dtype)
    scan_t.test_zoh_discretization(dtype)
    scan_t.test_chunked_with_initial_state(64, dtype)


@pytest.mark.parametrize("shape", [scan_t.ZOH_FAST_SHAPES[2], scan_t.ZOH_FAST_SHAPES[3]])
def test_scan_zoh_fast_path(checked, shape):
    scan_t.test_zoh_fast_path(shape)


@pytest.mark.parametrize("discretization", ["delta_b", "zoh"])
def test_scan_fast_kernel_flag_instances(checked, discretization):
    for use_z in (True, False):
        for softplus in (True, False):
            scan_t.test_fast_kernel_flag_instances(discretization, use_z, softplus)


def test_scan_zoh_fast_path_general_A_chunked_balanced(checked):
    scan_t.test_zoh_fast_path_general_A_and_zero_rows()
    scan_t.test_zoh_fast_path_chunked(64)
    scan_t.test_zoh_fast_path_balanced_sampled()


@pytest.mark.parametrize("shape,chunk", [((2, 140, 16, 512), 256), ((3, 100, 7, 1000), 192),
                                         ((1, 130, 16, 136), 64)])
def test_scan_bf16_chunked_schedule(checked, shape, chunk):
    """The fast kernel's aggregate and main passes, ragged last chunk and channel group included."""
    b, d, n, L = shape
    inp = W.random_scan_inputs(b, d, n, L, "bf16", seed=L + chunk, device=torch.device("cuda:0"))
    h0 = torch.randn((b, d, n), device="cuda:0")
    y, hL = scan_t._run(inp, algorithm="chunked", chunk_len=chunk, h0=h0)
    scan_t._check_full(inp, y, hL, scan_t.TOL[torch.bfloat16], h0=h0)


@pytest.mark.parametrize("shape", [scan_t.BALANCED_SHAPES[2], scan_t.BALANCED_SHAPES[3]])
def test_scan_balanced_schedule(checked, shape):
    scan_t.test_balanced_schedule_sampled(shape)


def test_scan_grid_schedule_130m_layer(checked):
    scan_t.test_mamba130m_layer_full("auto")


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("shape", [(3, 37, 16), (2, 20, 5), (5, 130, 1)])
def test_decode_small_shapes(checked, shape, io):
    decode_t.test_decode_small_shapes_every_channel(shape, io)


def test_decode_flag_instances(checked):
    for use_z in (True, False):
        for softplus in (True, False):
            decode_t.test_decode_flag_instances(use_z, softplus)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("shape", [(2, 130, 256), (1, 64, 33), (3, 20, 1), (1, 5, 2), (1, 16, 3)])
def test_conv1d_small_shapes(checked, shape, dtype):
    conv_t.test_conv1d_every_element(shape, dtype, True, True)
    conv_t.test_conv1d_every_element(shape, dtype, False, False)


@pytest.mark.parametrize("L", [1, 63, 65, 200])
def test_ssd_ragged_lengths(checked, L):
    ssd_t.test_ssd_ragged_lengths(L)


def test_ssd_groups_h0_and_options(checked):
    ssd_t.test_ssd_groups_h0_and_options()


@pytest.mark.parametrize("ctas", [1, 3, 7])
def test_ssd_balanced_ranges(checked, ctas):
    ssd_t.test_ssd_balanced_ranges_match_one_cta_per_sequence(ctas)


@pytest.mark.parametrize("groups", [1, 2])
def test_ssd_decode_steps(checked, groups):
    ssd_t.test_ssd_decode_steps_match_the_recurrence(groups)


@pytest.mark.parametrize("L", [200, 203])
def test_backward_flag_instances(checked, L):
    for use_z in (True, False):
        for softplus in (True, False):
            bwd_t.test_backward_flag_instances(use_z, softplus, L)


@pytest.mark.parametrize("shape,io", [((2, 200, 13, 333), "f32"), ((3, 130, 16, 77), "bf16"),
                                      ((2, 256, 16, 512), "bf16"), ((1, 5, 1, 9), "f32"), ((2, 129, 16, 1), "bf16")])
def test_backward_small_and_ragged(checked, shape, io):
    bwd_t.test_backward_small_and_ragged(shape, io)


def _close(a, b, tol):
    assert max_rel_err(to64(a), to64(b)) <= tol


def test_full_size_workloads_stay_in_bounds():
    """The full-size workloads through the checked build: every global index of the prefill (balanced
    and chunked schedules, exact ZOH), the backward, conv1d, the decode step, the SSD forward (balanced
    and one CTA per sequence) and its decode step stays inside its buffer, and the results agree with the ordinary build's (the same
    arithmetic: equal up to the order of the backward's cross-channel atomics)."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dev = torch.device("cuda:0")
    w = W.WORKLOADS["mamba2.8b-layer"]
    inp = W.make_scan_inputs(w, device=dev)
    dy = W.make_cotangent(w.batch, w.dim, w.seqlen, inp["u"].dtype, w.seed, device=dev)
    conv_w = torch.randn((w.dim, 4), device=dev) * 0.5
    conv_s = torch.randn((w.batch, w.dim, 3), device=dev)
    sw = W.WORKLOADS["mamba2-ssd-layer"]
    sin = W.make_ssd_inputs(sw, device=dev)
    dw = W.WORKLOADS["decode-2.8b"]
    din = W.make_decode_inputs(dw, steps=3, device=dev)
    mw = W.WORKLOADS["mamba2-decode"]
    mdin = W.make_ssd_decode_inputs(mw, device=dev)

    def run_all():
        a = dict(D=inp["D"], z=inp["z"], delta_bias=inp["delta_bias"])
        out = {"scan": ssm.selective_scan_fwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], **a),
               "chunked": ssm.selective_scan_fwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"],
                                                 algorithm="chunked", **a),
               "zoh": ssm.selective_scan_fwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"],
                                             discretization="zoh", **a),
               "bwd": ssm.selective_scan_bwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], dy, **a),
               "conv": ssm.causal_conv1d_fwd(inp["u"], conv_w, conv_state=conv_s),
               "ssd": ssm.ssd_fwd(sin["x"], sin["dt"], sin["A"], sin["B"], sin["C"], D=sin["D"],
                                  dt_bias=sin["dt_bias"]),
               "ssd_grid": ssm.ssd_fwd(sin["x"], sin["dt"], sin["A"], sin["B"], sin["C"], D=sin["D"],
                                       dt_bias=sin["dt_bias"], balanced=False)}
        state = torch.zeros((dw.batch, dw.dim, dw.dstate), device=dev)
        cst = torch.zeros((dw.batch, dw.dim, 3), device=dev)
        out["decode"] = [ssm.selective_state_update(din["x"][t], din["delta"][t], din["A"], din["B"][t], din["C"][t],
                                                    din["D"], din["z"][t], state, cst, din["conv_w"],
                                                    delta_bias=din["delta_bias"]) for t in range(3)] + [state, cst]
        mstate = torch.zeros((mw.batch, mw.nheads, mw.headdim, mw.dstate), device=dev)
        out["ssd_decode"] = [ssm.ssd_state_update(mdin["x"][t], mdin["dt"][t], mdin["A"], mdin["B"][t], mdin["C"][t],
                                                  mstate, D=mdin["D"], dt_bias=mdin["dt_bias"]) for t in range(3)]
        out["ssd_decode"].append(mstate)
        torch.cuda.synchronize()
        return out

    ref = run_all()
    assert ssm.device_status() == ssm.SSM_OK
    with ssm.use_checked_library():
        assert ssm.device_status() == ssm.SSM_OK
        got = run_all()
        assert ssm.device_status() == ssm.SSM_OK, "an index check failed at full size"
    for a, b in zip(ref["ssd"], ref["ssd_grid"]):   # the two SSD schedules: the same arithmetic
        assert torch.equal(a, b)
    for k in ("scan", "chunked", "zoh", "conv", "ssd", "ssd_grid"):
        for a, b in zip(got[k], ref[k]):
            if a is not None:
                _close(a, b, 1e-5)
    for name, g in got["bwd"].items():
        if g is not None:
            _close(g, ref["bwd"][name], 1e-3)
    for a, b in zip(got["decode"], ref["decode"]):
        _close(a, b, 1e-5)
    for a, b in zip(got["ssd_decode"], ref["ssd_decode"]):
        _close(a, b, 1e-5)
