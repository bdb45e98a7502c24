"""GPU test of the device failure path, without faulting a GPU.

The library's kernels bound every device wait (an mbarrier phase of a TMA pipeline, the flag of the
CTA-to-CTA carry): when a wait runs out, the kernel records a timeout in a status word and returns.
ssm_selftest_bounded_wait runs each kind of wait against a condition that nothing satisfies; the
timeout must reach the host through ssm_device_status, the word must be cleared by that read, and the
context must remain usable (a scan afterwards still matches the oracle).
"""
import time

import pytest
import torch

from selective_state_space_139_b300 import ssm
from selective_state_space_139_b300 import workloads as W
from tests._helpers import max_rel_err, to64

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
