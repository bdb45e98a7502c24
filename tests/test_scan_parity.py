"""GPU parity of the prefill scan (C ABI through the binding) against the fp64 oracle.

Tolerances: max relative error (with a floor of 1e-3 of the largest reference value) of 2e-5 for
float32 io and 1e-2 for bfloat16 io with float32 state.  Small shapes are compared element by
element over every output; the full-size workloads are compared over every output too (the oracle runs
on all host cores, in channel blocks for the 2^20-step sequence), in the launch configuration the
benchmark times (algorithm "auto").
"""
import numpy as np
import pytest
import torch

from selective_state_space_139_b300 import ssm
from selective_state_space_139_b300 import workloads as W
from tests._helpers import max_rel_err, oracle_channels, sample_channels, to64

import oracle

pytestmark = pytest.mark.gpu

TOL = {torch.float32: 2e-5, torch.bfloat16: 1e-2}


def _dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


def _run(inp, **kw):
    y, hL = ssm.selective_scan_fwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], D=inp.get("D"),
                                   z=inp.get("z"), delta_bias=inp.get("delta_bias"), **kw)
    torch.cuda.synchronize()
    return y, hL


def _full_oracle(inp, softplus=True, h0=None, discretization="delta_b"):
    return oracle.selective_scan(to64(inp["u"]), to64(inp["delta"]), to64(inp["A"]), to64(inp["B"]), to64(inp["C"]),
                                 D=to64(inp.get("D")), z=to64(inp.get("z")), delta_bias=to64(inp.get("delta_bias")),
                                 delta_softplus=softplus, h0=to64(h0), discretization=discretization)


def _check_full(inp, y, hL, tol, **okw):
    ry, rh = _full_oracle(inp, **okw)
    ey = max_rel_err(to64(y), ry)
    eh = max_rel_err(to64(hL), rh)
    assert ey <= tol and eh <= tol, (ey, eh)
    return ey, eh


def test_tiny_f32_workload_full():
    dev = _dev()
    inp = W.make_scan_inputs(W.WORKLOADS["tiny-f32"], device=dev)
    y, hL = _run(inp)
    _check_full(inp, y, hL, TOL[torch.float32])


@pytest.mark.parametrize("algorithm", ["auto", "single_pass"])
def test_mamba130m_layer_full(algorithm):
    dev = _dev()
    inp = W.make_scan_inputs(W.WORKLOADS["mamba130m-layer"], device=dev)
    y, hL = _run(inp, algorithm=algorithm)
    _check_full(inp, y, hL, TOL[torch.bfloat16])


_ORACLE_CACHE = {}


def _rel_err_on_device(y, ref):
    """The parity metric computed on the GPU (float64), for outputs too large to hold twice on the host."""
    y = y.double()
    ref = ref.double()
    scale = max(float(ref.abs().max()), 1e-30)
    return float(((y - ref).abs() / torch.clamp(ref.abs(), min=1e-3 * scale)).max())


def _blockwise_errors(inp, y, hL, batch, dim, block):
    """The parity metric over every channel: the oracle runs on blocks of channels (host memory stays
    bounded for long sequences) and its results are gathered on the device, rounded to float32 for y
    (a 6e-8 relative change, far below the 1e-2 bound) and kept in float64 for the final state."""
    dev = y.device
    ref_y = torch.empty(y.shape, dtype=torch.float32, device=dev)
    ref_h = torch.empty(hL.shape, dtype=torch.float64, device=dev)
    chans = [(b, d) for b in range(batch) for d in range(dim)]
    for i in range(0, len(chans), block):
        part = chans[i:i + block]
        ry, rh = oracle_channels(inp, part)
        bi = torch.tensor([c[0] for c in part])
        di = torch.tensor([c[1] for c in part])
        ref_y[bi, di] = torch.from_numpy(ry).to(dev, torch.float32)
        ref_h[bi, di] = torch.from_numpy(rh).to(dev)
    return _rel_err_on_device(y, ref_y), _rel_err_on_device(hL, ref_h)


@pytest.mark.parametrize("algorithm", ["auto", "chunked"])
def test_mamba28b_layer_full(algorithm):
    """Every output of the Mamba-2.8B layer (batch 4, d_inner 5120, L 4096) against the oracle."""
    dev = _dev()
    w = W.WORKLOADS["mamba2.8b-layer"]
    inp = W.make_scan_inputs(w, device=dev)
    y, hL = _run(inp, algorithm=algorithm)
    assert torch.isfinite(y).all()
    if w.name not in _ORACLE_CACHE:
        _ORACLE_CACHE[w.name] = _full_oracle(inp)
    ry, rh = _ORACLE_CACHE[w.name]
    assert max_rel_err(to64(y), ry) <= 1e-2
    assert max_rel_err(to64(hL), rh) <= 1e-2


def test_long_dna_full():
    """Every output of the long-sequence workload (batch 1, d_inner 1536, L 2^20), oracle on blocks of
    channels."""
    dev = _dev()
    w = W.WORKLOADS["long-dna"]
    inp = W.make_scan_inputs(w, device=dev)
    y, hL = _run(inp)
    assert torch.isfinite(y).all()
    ey, eh = _blockwise_errors(inp, y, hL, w.batch, w.dim, block=96)
    assert ey <= 1e-2 and eh <= 1e-2, (ey, eh)


def test_long_sequence_beyond_2_31_elements():
    """The long-sequence workload with two batch rows: 3.2e9 elements per io tensor, so the offsets of
    the second row exceed 2^31.  Sampled channels of both rows (the last channel of the last row
    included) against the oracle, every output finite, status clean."""
    import dataclasses
    dev = _dev()
    w = dataclasses.replace(W.WORKLOADS["long-dna"], name="long-dna-x2", batch=2, seed=1013)
    assert w.batch * w.dim * w.seqlen > 2 ** 31
    inp = W.make_scan_inputs(w, device=dev)
    y, hL = _run(inp)
    assert torch.isfinite(y).all() and torch.isfinite(hL).all()
    assert ssm.device_status() == ssm.SSM_OK
    chans = sorted(set(sample_channels(w.batch, w.dim, 24, seed=3) + [(1, w.dim - 1), (1, 0), (0, w.dim - 1)]))
    ry, rh = oracle_channels(inp, chans)
    bi = torch.tensor([c[0] for c in chans])
    di = torch.tensor([c[1] for c in chans])
    assert max_rel_err(to64(y[bi, di]), ry) <= 1e-2
    assert max_rel_err(to64(hL[bi, di]), rh) <= 1e-2


SHAPES = [  # batch, dim, dstate, L
    (1, 64, 16, 1), (1, 64, 16, 7), (2, 130, 16, 33), (1, 200, 5, 257), (3, 129, 16, 100),
    (2, 256, 16, 64), (1, 128, 16, 512), (2, 300, 1, 130),
]


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("shape", SHAPES)
def test_ragged_shapes(shape, dtype):
    dev = _dev()
    b, d, n, L = shape
    inp = W.random_scan_inputs(b, d, n, L, "f32" if dtype == torch.float32 else "bf16", seed=11 + L, device=dev)
    y, hL = _run(inp)
    _check_full(inp, y, hL, TOL[dtype])


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_optional_operands_and_softplus_off(dtype):
    dev = _dev()
    inp = W.random_scan_inputs(2, 160, 16, 200, "f32" if dtype == torch.float32 else "bf16", seed=5, device=dev)
    # no gate, no D, no bias
    bare = dict(inp, z=None, D=None, delta_bias=None)
    y, hL = _run(bare)
    _check_full(bare, y, hL, TOL[dtype])
    # softplus off: Δ = Δ_raw must then be non-negative for a decaying recurrence: use 0.1|Δ_raw|
    # and no bias (the generated biases are negative, softplus^-1 of values below 0.1)
    pos = dict(inp, delta=(inp["delta"].float().abs() * 0.1).to(inp["delta"].dtype), delta_bias=None)
    y, hL = _run(pos, delta_softplus=False)
    _check_full(pos, y, hL, TOL[dtype], softplus=False)


@pytest.mark.parametrize("discretization", ["delta_b", "zoh"])
@pytest.mark.parametrize("use_z", [True, False])
@pytest.mark.parametrize("softplus", [True, False])
def test_fast_kernel_flag_instances(discretization, use_z, softplus):
    """Every compiled instance of the bf16 fast kernel (gate or none, softplus on or off, Δ·B or
    exact ZOH), in the grid schedule and in the chunked schedule (its aggregate pass included)."""
    dev = _dev()
    b, d, n, L = 2, 136, 16, 256
    assert ssm.describe_scan(b, d, n, L, dtype=torch.bfloat16, discretization=discretization)["path"] == "fast"
    inp = W.random_scan_inputs(b, d, n, L, "bf16", seed=3 + 2 * use_z + softplus, device=dev)
    if not use_z:
        inp = dict(inp, z=None)
    if not softplus:
        # Δ = Δ_raw must be non-negative without softplus: 0.1|Δ_raw|, no bias
        inp = dict(inp, delta=(inp["delta"].float().abs() * 0.1).to(inp["delta"].dtype), delta_bias=None)
    h0 = torch.randn((b, d, n), device=dev)
    for algo, chunk in (("single_pass", 0), ("chunked", 64)):
        y, hL = _run(inp, delta_softplus=softplus, discretization=discretization, h0=h0, algorithm=algo,
                     chunk_len=chunk)
        _check_full(inp, y, hL, TOL[torch.bfloat16], softplus=softplus, discretization=discretization, h0=h0)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("chunk", [64, 128, 192])
def test_chunked_with_initial_state(chunk, dtype):
    dev = _dev()
    inp = W.random_scan_inputs(2, 140, 16, 501, "f32" if dtype == torch.float32 else "bf16", seed=chunk, device=dev)
    h0 = torch.randn((2, 140, 16), device=dev, dtype=torch.float32)
    y, hL = _run(inp, algorithm="chunked", chunk_len=chunk, h0=h0)
    _check_full(inp, y, hL, TOL[dtype], h0=h0)
    y1, h1 = _run(inp, algorithm="single_pass", h0=h0)
    _check_full(inp, y1, h1, TOL[dtype], h0=h0)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_general_A(dtype):
    dev = _dev()
    inp = W.random_scan_inputs(2, 136, 16, 300, "f32" if dtype == torch.float32 else "bf16", seed=9, device=dev)
    g = torch.Generator(device=dev)
    g.manual_seed(4)
    inp["A"] = -torch.exp(torch.randn((136, 16), generator=g, device=dev))   # no (n+1) structure
    y, hL = _run(inp)
    _check_full(inp, y, hL, TOL[dtype])
    # a mix: half the channels structured, half not (the shortcut is decided per warp)
    inp["A"][:64] = -torch.arange(1, 17, device=dev, dtype=torch.float32)
    y, hL = _run(inp)
    _check_full(inp, y, hL, TOL[dtype])


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_zoh_discretization(dtype):
    dev = _dev()
    inp = W.random_scan_inputs(1, 130, 16, 150, "f32" if dtype == torch.float32 else "bf16", seed=21, device=dev)
    inp["A"][0, 3] = 0.0   # the a -> 0 limit
    y, hL = _run(inp, discretization="zoh")
    _check_full(inp, y, hL, TOL[dtype], discretization="zoh")


ZOH_FAST_SHAPES = [  # batch, dim, dstate, L: bf16 shapes the fast kernel takes (L a multiple of 8, >= 64)
    (2, 256, 16, 512), (1, 128, 16, 64), (3, 129, 16, 136), (2, 300, 5, 200), (1, 200, 1, 72),
]


@pytest.mark.parametrize("shape", ZOH_FAST_SHAPES)
def test_zoh_fast_path(shape):
    """The exact-ZOH input term on the bf16 fast kernel (structured A: the rescaled k = h/(-u/A[d,0])
    form), every output, with an initial state."""
    dev = _dev()
    b, d, n, L = shape
    assert ssm.describe_scan(b, d, n, L, dtype=torch.bfloat16, discretization="zoh")["path"] == "fast"
    inp = W.random_scan_inputs(b, d, n, L, "bf16", seed=31 + L, a_scale=(0.5, 2.0), device=dev)
    h0 = torch.randn((b, d, n), device=dev)
    y, hL = _run(inp, discretization="zoh", h0=h0)
    _check_full(inp, y, hL, TOL[torch.bfloat16], discretization="zoh", h0=h0)


def test_zoh_fast_path_general_A_and_zero_rows():
    """Exact ZOH on the fast kernel's per-state path: A without the (n+1) structure, single zero
    entries (the A -> 0 limit Δ·B) and whole zero rows (structured but A[d,0] = 0), next to
    structured warps."""
    dev = _dev()
    inp = W.random_scan_inputs(2, 256, 16, 320, "bf16", seed=41, device=dev)
    g = torch.Generator(device=dev)
    g.manual_seed(6)
    A = -torch.exp(torch.randn((256, 16), generator=g, device=dev))
    A[:64] = -0.5 * torch.arange(1, 17, device=dev, dtype=torch.float32)   # structured warps
    A[70, 3] = 0.0
    A[100, 0] = 0.0
    A[160:192] = 0.0                                                        # zero rows, one whole warp
    A[200, :] = 0.0                                                         # a zero row in a mixed warp
    A[230, 5] = -1e-6                                                       # |Δ A| far below 1/32
    inp["A"] = A
    h0 = torch.randn((2, 256, 16), device=dev)
    y, hL = _run(inp, discretization="zoh", h0=h0)
    _check_full(inp, y, hL, TOL[torch.bfloat16], discretization="zoh", h0=h0)


@pytest.mark.parametrize("L", [256, 150])
def test_zoh_tiny_and_denormal_A(L):
    """Exact ZOH where 1/A would overflow: zero, tiny (1e-30) and denormal (1e-40) entries of A, and a
    structured row whose A[d,0] is denormal.  Both kernels (L = 256: the fast kernel; L = 150: the
    general one) must give the A -> 0 limit Δ·B for those states, finite everywhere."""
    dev = _dev()
    inp = W.random_scan_inputs(2, 136, 16, L, "bf16", seed=53 + L, device=dev)
    A = inp["A"].clone()
    A[3, 2] = 0.0
    A[10, 5] = -1e-30
    A[20, 7] = -1e-40
    A[21, 0] = 1e-40
    A[40, :] = 1e-39 * torch.arange(1, 17, device=dev, dtype=torch.float32)   # structured, denormal A[d,0]
    inp["A"] = A
    y, hL = _run(inp, discretization="zoh")
    assert torch.isfinite(y).all() and torch.isfinite(hL).all()
    _check_full(inp, y, hL, TOL[torch.bfloat16], discretization="zoh")


@pytest.mark.parametrize("chunk", [64, 192])
def test_zoh_fast_path_chunked(chunk):
    """Exact ZOH through the chunked schedule: aggregate pass, carry pass, main pass."""
    dev = _dev()
    inp = W.random_scan_inputs(2, 140, 16, 512, "bf16", seed=chunk + 3, device=dev)
    h0 = torch.randn((2, 140, 16), device=dev)
    y, hL = _run(inp, algorithm="chunked", chunk_len=chunk, discretization="zoh", h0=h0)
    _check_full(inp, y, hL, TOL[torch.bfloat16], discretization="zoh", h0=h0)


def test_zoh_fast_path_balanced_sampled():
    """Exact ZOH through the balanced persistent schedule (CTA-to-CTA carries), sampled channels."""
    dev = _dev()
    b, d, n, L = 8, 2400, 16, 200
    inp = W.random_scan_inputs(b, d, n, L, "bf16", seed=77, a_scale=(0.5, 2.0), device=dev)
    assert ssm.describe_scan(b, d, n, L, dtype=torch.bfloat16, discretization="zoh")["schedule"] == "balanced"
    h0 = torch.randn((b, d, n), device=dev)
    y, hL = _run(inp, discretization="zoh", h0=h0)
    chans = sorted(set(sample_channels(b, d, 160, seed=5) + [(bb, dd) for bb in (0, b - 1) for dd in (127, 128, d - 1)]))
    ry, rh = oracle_channels(inp, chans, h0=h0, discretization="zoh")
    bi = torch.tensor([c[0] for c in chans])
    di = torch.tensor([c[1] for c in chans])
    assert max_rel_err(to64(y[bi, di]), ry) <= 1e-2
    assert max_rel_err(to64(hL[bi, di]), rh) <= 1e-2
    assert torch.isfinite(y).all() and torch.isfinite(hL).all()
    assert ssm.device_status() == ssm.SSM_OK


@pytest.mark.parametrize("discretization", ["delta_b", "zoh"])
def test_general_A_mamba28b_layer_full(discretization):
    """Every output of the Mamba-2.8B layer with A = -exp(3 U[0,1)) per (d, n) (no (n+1) structure: the
    fast kernel's per-state path), both input terms, in the benchmark's launch configuration."""
    dev = _dev()
    w = W.WORKLOADS["mamba2.8b-layer"]
    inp = W.make_scan_inputs(w, device=dev)
    g = torch.Generator(device=dev).manual_seed(w.seed + 17)
    inp["A"] = -torch.exp(3.0 * torch.rand(inp["A"].shape, generator=g, device=dev))
    y, hL = _run(inp, discretization=discretization)
    assert torch.isfinite(y).all()
    ry, rh = _full_oracle(inp, discretization=discretization)
    assert max_rel_err(to64(y), ry) <= 1e-2
    assert max_rel_err(to64(hL), rh) <= 1e-2


def test_zoh_mamba28b_layer_full():
    """Every output of the exact-ZOH prefill of the Mamba-2.8B layer (batch 4, d_inner 5120, L 4096) in
    the benchmark's launch configuration against the oracle."""
    dev = _dev()
    w = W.WORKLOADS["mamba2.8b-layer"]
    inp = W.make_scan_inputs(w, device=dev)
    y, hL = _run(inp, discretization="zoh")
    assert torch.isfinite(y).all()
    ry, rh = _full_oracle(inp, discretization="zoh")
    assert max_rel_err(to64(y), ry) <= 1e-2
    assert max_rel_err(to64(hL), rh) <= 1e-2


def test_outputs_fully_overwritten_and_status_clean():
    dev = _dev()
    inp = W.random_scan_inputs(2, 200, 16, 333, "bf16", seed=3, device=dev)
    y = torch.full_like(inp["u"], float("nan"))
    hL = torch.full((2, 200, 16), float("nan"), device=dev)
    for algo in ("single_pass", "chunked"):
        y.fill_(float("nan"))
        hL.fill_(float("nan"))
        ssm.selective_scan_fwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], D=inp["D"], z=inp["z"],
                               delta_bias=inp["delta_bias"], out=y, last_state=hL, algorithm=algo,
                               chunk_len=128 if algo == "chunked" else 0)
        torch.cuda.synchronize()
        assert torch.isfinite(y).all() and torch.isfinite(hL).all()
    assert ssm.device_status() == ssm.SSM_OK


def test_unaligned_buffers_take_the_general_kernel():
    dev = _dev()
    inp = W.random_scan_inputs(2, 256, 16, 512, "bf16", seed=8, device=dev)
    y_tma, h_tma = _run(inp)
    # same values at a base address that is only 2-byte aligned: TMA cannot describe it
    shifted = {}
    for k in ("u", "delta", "z", "B", "C"):
        t = inp[k]
        buf = torch.empty(t.numel() + 1, dtype=t.dtype, device=dev)
        v = buf[1:].view(t.shape)
        v.copy_(t)
        shifted[k] = v
    shifted.update({k: inp[k] for k in ("A", "D", "delta_bias")})
    y_pl, h_pl = _run(shifted)
    # two different kernels (the bf16 fast path and the general kernel): both must meet the bound
    _check_full(inp, y_tma, h_tma, 1e-2)
    _check_full(inp, y_pl, h_pl, 1e-2)


def test_seqlen_zero_returns_initial_state():
    dev = _dev()
    inp = W.random_scan_inputs(2, 64, 16, 0, "bf16", seed=1, device=dev)
    h0 = torch.randn((2, 64, 16), device=dev)
    _, hL = _run(inp, h0=h0)
    assert torch.equal(hL, h0)
    _, hL = _run(inp)
    assert torch.count_nonzero(hL) == 0


def test_binding_rejects_cpu_tensors():
    inp = W.random_scan_inputs(1, 8, 16, 16, "bf16", seed=1)
    with pytest.raises(ValueError):
        ssm.selective_scan_fwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"])


BALANCED_SHAPES = [  # at least one 128-channel group per resident CTA: balanced persistent schedule
    (8, 2400, 16, 200),     # 152 groups, 4 tiles per group, a ragged last tile of one 8-step chunk
    (64, 512, 16, 256),     # 256 groups
    (5, 4100, 16, 136),     # ragged dim (4100 = 32 * 128 + 4), last tile of one 8-step chunk
    (8, 2400, 7, 128),      # dstate 7
]


@pytest.mark.parametrize("shape", BALANCED_SHAPES)
def test_balanced_schedule_sampled(shape):
    dev = _dev()
    b, d, n, L = shape
    inp = W.random_scan_inputs(b, d, n, L, "bf16", seed=d + L, a_scale=(0.5, 2.0), device=dev)
    h0 = torch.randn((b, d, n), device=dev)
    y, hL = _run(inp, h0=h0)
    chans = sample_channels(b, d, 160, seed=L)
    # channels at group boundaries and in the last group of each batch row
    chans += [(bb, dd) for bb in (0, b - 1) for dd in (63, 64, 127, 128, d - 1)]
    chans = sorted(set(chans))
    ry, rh = oracle_channels(inp, chans, h0=h0)
    bi = torch.tensor([c[0] for c in chans])
    di = torch.tensor([c[1] for c in chans])
    assert max_rel_err(to64(y[bi, di]), ry) <= 1e-2
    assert max_rel_err(to64(hL[bi, di]), rh) <= 1e-2
    assert torch.isfinite(y).all() and torch.isfinite(hL).all()
    assert ssm.device_status() == ssm.SSM_OK


def test_balanced_schedule_is_deterministic():
    dev = _dev()
    inp = W.random_scan_inputs(8, 2400, 16, 512, "bf16", seed=1, device=dev)
    y1, h1 = _run(inp)
    y2, h2 = _run(inp)
    assert torch.equal(y1, y2) and torch.equal(h1, h2)
