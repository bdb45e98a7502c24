"""GPU test of the device failure path, without faulting a GPU.

The library's kernels bound every device wait (an mbarrier phase of a TMA pipeline, the flag of the
CTA-to-CTA carry): when a wait runs out, the kernel records a timeout in a status word and returns.
ssm_selftest_bounded_wait runs each kind of wait against a condition that nothing satisfies; the
timeout must reach the host through ssm_device_status, the word must be cleared by that read, and the
context must remain usable (a scan afterwards still matches the oracle).  ssm_selftest_withhold_carry
makes the real prefill and SSD kernels' CTA-to-CTA carry waits run out: one CTA of a balanced
schedule writes its carry but never raises the flag that publishes it.
"""
import time

import pytest
import torch

from selective_state_space_139_b300 import ssm
from selective_state_space_139_b300 import workloads as W
from tests._helpers import max_rel_err, oracle_channels, sample_channels, to64

import oracle

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("which", [0, 1])   # 0: mbarrier phase, 1: global flag
def test_bounded_wait_timeout_reaches_the_host_and_clears(which):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib = ssm.load_library()
    stream = torch.cuda.current_stream().cuda_stream
    assert lib.ssm_device_status(stream) == ssm.SSM_OK            # nothing pending before the test
    t0 = time.monotonic()
    assert lib.ssm_selftest_bounded_wait(which, 50_000_000, stream) == ssm.SSM_OK   # 50 ms limit
    assert lib.ssm_device_status(stream) == ssm.SSM_ERR_TIMEOUT
    assert time.monotonic() - t0 < 10.0                            # the wait ended by itself
    assert lib.ssm_device_status(stream) == ssm.SSM_OK            # the read cleared the word
    # the context is still usable: a scan afterwards matches the oracle
    inp = W.make_scan_inputs(W.WORKLOADS["tiny-f32"], device=torch.device("cuda:0"))
    y, hL = ssm.selective_scan_fwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], D=inp["D"], z=inp["z"],
                                   delta_bias=inp["delta_bias"])
    torch.cuda.synchronize()
    ry, rh = oracle.selective_scan(to64(inp["u"]), to64(inp["delta"]), to64(inp["A"]), to64(inp["B"]),
                                   to64(inp["C"]), D=to64(inp["D"]), z=to64(inp["z"]),
                                   delta_bias=to64(inp["delta_bias"]))
    assert max_rel_err(to64(y), ry) <= 2e-5 and max_rel_err(to64(hL), rh) <= 2e-5
    assert lib.ssm_device_status(stream) == ssm.SSM_OK


def test_withheld_carry_times_out_in_the_prefill_kernel():
    """The balanced schedule of the 2.8B layer (160 groups of 128 channels on 148 CTAs, ranges of 70
    tiles): CTA 0 runs group 0 and the head of group 1 (tiles 0..5), CTA 1 continues group 1 from tile
    6 with the state CTA 0 publishes.  With that publication withheld, CTA 1's wait gives up after the
    armed 50 ms, the call returns, the status read reports the timeout once, and the next call (not
    armed) matches the oracle, group 1 included."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib = ssm.load_library()
    dev = torch.device("cuda:0")
    b, d, n, L = 4, 5120, 16, 4096
    plan = ssm.describe_scan(b, d, n, L, dtype=torch.bfloat16)
    assert plan["schedule"] == "balanced" and plan["ctas"] >= 2
    inp = W.random_scan_inputs(b, d, n, L, "bf16", seed=77, a_scale=(0.5, 2.0), device=dev)
    args = dict(D=inp["D"], z=inp["z"], delta_bias=inp["delta_bias"])
    assert ssm.device_status() == ssm.SSM_OK
    assert lib.ssm_selftest_withhold_carry(0, 50_000_000) == ssm.SSM_OK
    t0 = time.monotonic()
    ssm.selective_scan_fwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], **args)
    assert ssm.device_status() == ssm.SSM_ERR_TIMEOUT
    assert time.monotonic() - t0 < 10.0                            # the wait ended by itself
    assert ssm.device_status() == ssm.SSM_OK                       # the read cleared the word
    y, hL = ssm.selective_scan_fwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], **args)
    assert ssm.device_status() == ssm.SSM_OK
    chans = sample_channels(b, d, 24, seed=3) + [(0, 128), (0, 200), (0, 255)]   # group 1: CTA 1's tail
    ry, rh = oracle_channels(inp, sorted(set(chans)))
    bi = torch.tensor([c[0] for c in sorted(set(chans))])
    di = torch.tensor([c[1] for c in sorted(set(chans))])
    assert max_rel_err(to64(y[bi, di]), ry) <= 1e-2
    assert max_rel_err(to64(hL[bi, di]), rh) <= 1e-2


def test_withheld_carry_times_out_in_the_ssd_kernel():
    """The SSD forward's balanced schedule on 8 sequences of 5 chunks in 3 ranges: CTA 0 runs the head
    of sequence 2 (chunks 0..3), CTA 1 its tail.  With CTA 0's publication withheld, CTA 1's wait gives
    up after the armed 50 ms, the status read reports the timeout once, and the next call matches the
    oracle."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib = ssm.load_library()
    dev = torch.device("cuda:0")
    w = W.SsdWorkload("adhoc", 2, 293, 4, 64, 128, 2, 2402)
    inp = W.make_ssd_inputs(w, device=dev)
    args = dict(D=inp["D"], dt_bias=inp["dt_bias"], ctas=3)
    assert ssm.device_status() == ssm.SSM_OK
    assert lib.ssm_selftest_withhold_carry(0, 50_000_000) == ssm.SSM_OK
    t0 = time.monotonic()
    ssm.ssd_fwd(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], **args)
    assert ssm.device_status() == ssm.SSM_ERR_TIMEOUT
    assert time.monotonic() - t0 < 10.0                            # the wait ended by itself
    assert ssm.device_status() == ssm.SSM_OK                       # the read cleared the word
    y, hT = ssm.ssd_fwd(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], **args)
    assert ssm.device_status() == ssm.SSM_OK
    ry, rh = oracle.ssd_scan(to64(inp["x"]), to64(inp["dt"]), to64(inp["A"]), to64(inp["B"]), to64(inp["C"]),
                             D=to64(inp["D"]), dt_bias=to64(inp["dt_bias"]))
    assert max_rel_err(to64(y), ry) <= 1e-2 and max_rel_err(to64(hT), rh) <= 1e-2


def test_withhold_carry_rejects_a_negative_cta():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib = ssm.load_library()
    assert lib.ssm_selftest_withhold_carry(-1, 50_000_000) == ssm.SSM_ERR_INVALID_ARG
