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
