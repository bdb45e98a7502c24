"""GPU parity of the scan backward (C ABI through the binding) against the fp64 oracle's reverse-mode
gradients.

Tolerances as for the forward: max relative error (floor 1e-3 of the largest reference value) of
2e-5 for float32 io and 1e-2 for bfloat16 io.  Small and ragged shapes compare every output; the
Mamba-130M layer compares every output at full size, the cross-channel sums dB and dC included; the
Mamba-2.8B layer compares the per-channel gradients (du, ddelta, dz) and the per-dim sums (dA, dD,
ddelta_bias) of sampled dims over all batch rows, in the configuration the benchmark times.
"""
import numpy as np
import pytest
import torch

from selective_state_space_139_b300 import ssm
from selective_state_space_139_b300 import workloads as W
from tests._helpers import max_rel_err, to64

import oracle

pytestmark = pytest.mark.gpu

TOL = {torch.float32: 2e-5, torch.bfloat16: 1e-2}
KEYS = ("du", "ddelta", "dz", "dA", "dB", "dC", "dD", "ddelta_bias")


def _dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


def _inputs(batch, dim, dstate, seqlen, io, seed, dev, a_scale=None):
    inp = W.random_scan_inputs(batch, dim, dstate, seqlen, io, seed=seed, a_scale=a_scale, device=dev)
    inp["dy"] = W.make_cotangent(batch, dim, seqlen, inp["u"].dtype, seed, device=dev)
    return inp


def _gpu(inp, use_z=True, use_D=True, use_bias=True, softplus=True):
    g = ssm.selective_scan_bwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["dy"],
                               D=inp["D"] if use_D else None, z=inp["z"] if use_z else None,
                               delta_bias=inp["delta_bias"] if use_bias else None, delta_softplus=softplus)
    torch.cuda.synchronize()
    return g


def _oracle(inp, use_z=True, use_D=True, use_bias=True, softplus=True):
    return oracle.scan_backward(to64(inp["u"]), to64(inp["delta"]), to64(inp["A"]), to64(inp["B"]), to64(inp["C"]),
                                to64(inp["dy"]), D=to64(inp["D"]) if use_D else None,
                                z=to64(inp["z"]) if use_z else None,
                                delta_bias=to64(inp["delta_bias"]) if use_bias else None, delta_softplus=softplus)


def _compare(g, r, tol, keys=KEYS):
    errs = {}
    for k in keys:
        if r.get(k) is None or g.get(k) is None:
            assert g.get(k) is None or k in ("dD", "ddelta_bias"), k
            continue
        errs[k] = max_rel_err(to64(g[k]), r[k])
    bad = {k: e for k, e in errs.items() if not e <= tol}
    assert not bad, (bad, errs)
    return errs


@pytest.mark.parametrize("shape,io", [((1, 64, 16, 256), "f32"), ((2, 200, 13, 333), "f32"),
                                      ((3, 130, 16, 77), "bf16"), ((2, 256, 16, 512), "bf16"),
                                      ((1, 5, 1, 9), "f32"), ((2, 129, 16, 1), "bf16")])
def test_backward_small_and_ragged(shape, io):
    dev = _dev()
    inp = _inputs(*shape, io, seed=sum(shape), dev=dev)
    g = _gpu(inp)
    _compare(g, _oracle(inp), TOL[inp["u"].dtype])


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("opts", [dict(use_z=False), dict(use_D=False), dict(use_bias=False),
                                  dict(use_z=False, use_D=False, use_bias=False, softplus=False)])
def test_backward_optional_operands(io, opts):
    dev = _dev()
    inp = _inputs(2, 96, 16, 200, io, seed=7, dev=dev)
    if not opts.get("softplus", True):
        inp["delta"] = (inp["delta"].float().abs() * 0.05).to(inp["delta"].dtype)   # positive steps without softplus
    g = _gpu(inp, **opts)
    r = _oracle(inp, **opts)
    if not opts.get("use_z", True):
        assert g["dz"] is None
    if not opts.get("use_D", True):
        assert g["dD"] is None
    if not opts.get("use_bias", True):
        assert g["ddelta_bias"] is None
    _compare(g, r, TOL[inp["u"].dtype])


@pytest.mark.parametrize("use_z", [True, False])
@pytest.mark.parametrize("softplus", [True, False])
@pytest.mark.parametrize("L", [200, 203])
def test_backward_flag_instances(use_z, softplus, L):
    """Every compiled instance of the bf16 two-lane backward kernels: gate or none, softplus on or
    off, every 8-step segment full (L = 200) or a ragged last segment (L = 203)."""
    dev = _dev()
    inp = _inputs(2, 96, 16, L, "bf16", seed=L + 2 * use_z + softplus, dev=dev)
    if not softplus:
        # Δ = Δ_raw without softplus: positive steps 0.05|Δ_raw| and no bias (the generated biases are
        # negative, softplus^-1 of steps below 0.1)
        inp["delta"] = (inp["delta"].float().abs() * 0.05).to(inp["delta"].dtype)
    g = _gpu(inp, use_z=use_z, use_bias=softplus, softplus=softplus)
    _compare(g, _oracle(inp, use_z=use_z, use_bias=softplus, softplus=softplus), TOL[inp["u"].dtype])


def test_backward_mamba130m_layer_full():
    dev = _dev()
    w = W.WORKLOADS["mamba130m-layer"]
    inp = W.make_scan_inputs(w, device=dev)
    inp["dy"] = W.make_cotangent(w.batch, w.dim, w.seqlen, inp["u"].dtype, w.seed, device=dev)
    g = _gpu(inp)
    _compare(g, _oracle(inp), TOL[torch.bfloat16])


def test_backward_mamba2p8b_layer_full():
    """Every output of the 2.8B-layer backward against the oracle, in the launch configuration the
    benchmark times: du, dΔ, dz of every channel and step, the batch-summed dA, dD, dbias, and the
    channel-summed dB, dC of every (batch row, state, step)."""
    dev = _dev()
    w = W.WORKLOADS["mamba2.8b-layer"]
    inp = W.make_scan_inputs(w, device=dev)
    inp["dy"] = W.make_cotangent(w.batch, w.dim, w.seqlen, inp["u"].dtype, w.seed, device=dev)
    g = _gpu(inp)
    r = _oracle(inp)
    tol = TOL[torch.bfloat16]
    errs = {}
    for k in KEYS:
        if r.get(k) is None:
            continue
        errs[k] = max_rel_err(to64(g[k]), r[k])
        r[k] = None   # bounded host memory: one full-size pair at a time
    bad = {k: e for k, e in errs.items() if not e <= tol}
    assert not bad, (bad, errs)


def test_backward_seqlen_zero_gives_zero_parameter_gradients():
    dev = _dev()
    inp = _inputs(2, 64, 16, 8, "f32", seed=3, dev=dev)
    for k in ("u", "delta", "z", "dy"):
        inp[k] = inp[k][:, :, :0].contiguous()
    for k in ("B", "C"):
        inp[k] = inp[k][:, :, :0].contiguous()
    g = _gpu(inp)
    assert g["du"].numel() == 0 and g["dB"].numel() == 0
    for k in ("dA", "dD", "ddelta_bias"):
        assert torch.count_nonzero(g[k]).item() == 0, k


def test_backward_rejects_cpu_tensors():
    _dev()
    inp = _inputs(1, 8, 4, 16, "f32", seed=1, dev="cpu")
    with pytest.raises(ValueError):
        ssm.selective_scan_bwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["dy"])
