"""The prefill planner (ssm_scan_fwd_describe): which kernel path and schedule a call runs, and the
workspace it needs.  The CPU tests check what does not depend on a device; the GPU test checks the
schedules the full-size workloads run with the device's resident-CTA count."""
import ctypes

import pytest
import torch

from selective_state_space_139_b300 import ssm

BF16, F32 = torch.bfloat16, torch.float32


def _ws_ex(batch, dim, N, L, dtype, algorithm="auto", chunk_len=0, discretization="delta_b"):
    lib = ssm.load_library()
    o = ssm._options(algorithm, chunk_len, discretization, None)
    return lib.ssm_scan_fwd_workspace_size_ex(batch, dim, N, L, 1 if dtype == BF16 else 0, ctypes.byref(o))


@pytest.mark.parametrize("shape", [(4, 5120, 16, 4096), (8, 1536, 16, 2048), (1, 64, 16, 256), (4, 512, 16, 1000),
                                   (3, 130, 5, 777)])
@pytest.mark.parametrize("dtype", [BF16, F32])
@pytest.mark.parametrize("algorithm", ["auto", "single_pass", "chunked"])
def test_plan_workspace_matches_the_workspace_query(shape, dtype, algorithm):
    pl = ssm.describe_scan(*shape, dtype=dtype, algorithm=algorithm)
    assert pl["workspace_bytes"] == _ws_ex(*shape, dtype, algorithm=algorithm)
    if pl["schedule"] == "grid":
        assert pl["nchunks"] == 1 and pl["workspace_bytes"] == 0 and pl["kernel_launches"] == 1
    if pl["schedule"] == "chunked":
        assert pl["nchunks"] > 1 and pl["kernel_launches"] == 3 and pl["workspace_bytes"] > 0
        assert pl["chunk_len"] % 64 == 0 and (shape[3] + pl["chunk_len"] - 1) // pl["chunk_len"] == pl["nchunks"]


def test_kernel_path_choice():
    assert ssm.describe_scan(4, 512, 16, 4096, dtype=BF16)["path"] == "fast"
    assert ssm.describe_scan(4, 512, 16, 4096, dtype=F32)["path"] == "general"          # float32 io
    assert ssm.describe_scan(4, 512, 16, 4096, dtype=BF16, discretization="zoh")["path"] == "fast"
    assert ssm.describe_scan(4, 512, 16, 4096, dtype=F32, discretization="zoh")["path"] == "general"
    assert ssm.describe_scan(4, 512, 16, 4100, dtype=BF16, discretization="zoh")["path"] == "general"
    assert ssm.describe_scan(4, 512, 16, 4100, dtype=BF16)["path"] == "general"          # L not a multiple of 8
    assert ssm.describe_scan(4, 512, 16, 32, dtype=BF16)["path"] == "general"            # shorter than a tile


def test_explicit_schedules():
    pl = ssm.describe_scan(4, 512, 16, 4096, dtype=BF16, algorithm="chunked", chunk_len=512)
    assert (pl["schedule"], pl["nchunks"], pl["chunk_len"], pl["kernel_launches"]) == ("chunked", 8, 512, 3)
    assert pl["ctas"] == 4 * (512 // 128) * 8
    pl = ssm.describe_scan(4, 5120, 16, 4096, dtype=BF16, algorithm="single_pass")
    assert (pl["schedule"], pl["nchunks"], pl["workspace_bytes"], pl["ctas"]) == ("grid", 1, 0, 4 * 5120 // 128)
    assert ssm.describe_scan(2, 256, 16, 0, dtype=BF16)["kernel_launches"] == 0


def test_bad_plans_are_refused():
    with pytest.raises(ssm.SSMError):
        ssm.describe_scan(4, 512, 16, 4096, dtype=BF16, algorithm="chunked", chunk_len=100)   # not a multiple of 64
    with pytest.raises(ssm.SSMError):
        ssm.describe_scan(4, 512, 17, 4096, dtype=BF16)                                       # dstate above 16
    lib = ssm.load_library()
    pl = ssm.ScanPlan()
    pl.struct_size = 3                                                                        # wrong struct size
    assert lib.ssm_scan_fwd_describe(4, 512, 16, 4096, 1, None, ctypes.byref(pl)) == ssm.SSM_ERR_INVALID_ARG


@pytest.mark.gpu
def test_full_size_workloads_run_the_balanced_and_chunked_schedules():
    """With the device's resident-CTA count known: the 2.8B layer (160 groups of 128 channels, at
    least one per SM) runs the balanced persistent schedule in one launch, one CTA per SM; the 130M
    layer (96 groups) runs one pass per group, which the wave count makes faster than time chunks;
    the 2^20-step sequence (12 groups) splits time into chunks."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    big = ssm.describe_scan(4, 5120, 16, 4096, dtype=BF16)
    assert (big["path"], big["schedule"], big["kernel_launches"]) == ("fast", "balanced", 1)
    assert big["ctas"] == sms and big["workspace_bytes"] > 0
    small = ssm.describe_scan(8, 1536, 16, 2048, dtype=BF16)
    assert (small["path"], small["schedule"], small["ctas"]) == ("fast", "grid", 96)
    long = ssm.describe_scan(1, 1536, 16, 1 << 20, dtype=BF16)
    assert (long["path"], long["schedule"]) == ("fast", "chunked") and long["nchunks"] > 1
