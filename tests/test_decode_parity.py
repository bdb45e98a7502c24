"""GPU parity of the one-token decode step against the fp64 oracle.

The full-size workload (batch 256, d_inner 5120, dstate 16, 1000 tokens) runs 1000 steps on the
GPU and must match, over every channel and step, one 1000-token prefill of the same inputs by the
oracle (causal conv + SiLU, then the selective scan); the final SSM state and conv state must match
too.
Small shapes (ragged dim, dstate < 16, float32 io) are compared over every channel.
"""
import numpy as np
import pytest
import torch

from selective_state_space_139_b300 import ssm
from selective_state_space_139_b300 import workloads as W
from tests._helpers import max_rel_err, to64

import oracle

pytestmark = pytest.mark.gpu


def _dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


def _decode_all(inp, steps, batch, dim, N, dev):
    state = torch.zeros((batch, dim, N), device=dev)
    conv_state = torch.zeros((batch, dim, 3), device=dev)
    ys = torch.empty_like(inp["x"][:steps])
    for t in range(steps):
        ssm.selective_state_update(inp["x"][t], inp["delta"][t], inp["A"], inp["B"][t], inp["C"][t], inp["D"],
                                   inp["z"][t], state, conv_state, inp["conv_w"], delta_bias=inp["delta_bias"],
                                   out=ys[t])
    torch.cuda.synchronize()
    return ys, state, conv_state


def _oracle_prefill(inp, chans, steps):
    """Oracle: conv + SiLU over the token stream, then the scan, for the listed channels."""
    bs = np.array([c[0] for c in chans], dtype=np.int64)
    ds = np.array([c[1] for c in chans], dtype=np.int64)
    bi, di = torch.as_tensor(bs), torch.as_tensor(ds)
    x = to64(inp["x"][:steps, bi, di].T)              # (n, steps)
    w = to64(inp["conv_w"][di])
    u, conv_tail = oracle.causal_conv1d(x, w, silu=True)
    B = to64(inp["B"][:steps].permute(1, 2, 0))        # (batch, N, steps)
    C = to64(inp["C"][:steps].permute(1, 2, 0))
    y, hL = oracle.selective_scan_channels(u, to64(inp["delta"][:steps, bi, di].T), to64(inp["A"][di]), B, C, bs,
                                           D=to64(inp["D"][di]), z=to64(inp["z"][:steps, bi, di].T),
                                           delta_bias=to64(inp["delta_bias"][di]))
    return y, hL, conv_tail, bi, di


def _rel_err_on_device(y, ref):
    """The parity metric computed on the GPU (float64), for outputs too large to hold twice on the host."""
    y = y.double()
    ref = ref.double()
    scale = max(float(ref.abs().max()), 1e-30)
    return float(((y - ref).abs() / torch.clamp(ref.abs(), min=1e-3 * scale)).max())


def test_decode_2p8b_1000_tokens_matches_prefill():
    """Every output of 1000 decode steps (batch 256, d_inner 5120) against one 1000-token oracle
    prefill: the oracle runs on blocks of channels and its results are gathered on the device (y
    rounded to float32, a 6e-8 relative change; state in float64; conv state exact)."""
    dev = _dev()
    w = W.WORKLOADS["decode-2.8b"]
    inp = W.make_decode_inputs(w, device=dev)
    ys, state, conv_state = _decode_all(inp, w.steps, w.batch, w.dim, w.dstate, dev)
    assert torch.isfinite(ys).all() and torch.isfinite(state).all()
    ref_y = torch.empty(ys.shape, dtype=torch.float32, device=dev)           # (steps, batch, dim)
    ref_h = torch.empty(state.shape, dtype=torch.float64, device=dev)
    chans = [(b, d) for b in range(w.batch) for d in range(w.dim)]
    block = 32768
    for i in range(0, len(chans), block):
        part = chans[i:i + block]
        ry, rh, rc, bi, di = _oracle_prefill(inp, part, w.steps)
        ref_y[:, bi, di] = torch.from_numpy(ry.T.copy()).to(dev, torch.float32)
        ref_h[bi, di] = torch.from_numpy(rh).to(dev)
        np.testing.assert_array_equal(to64(conv_state[bi, di]), rc)   # raw inputs, kept exactly
    assert _rel_err_on_device(ys, ref_y) <= 1e-2
    assert _rel_err_on_device(state, ref_h) <= 1e-2


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("shape", [(3, 37, 16), (2, 20, 5), (1, 64, 16), (5, 130, 1)])
def test_decode_small_shapes_every_channel(shape, io):
    dev = _dev()
    batch, dim, N = shape
    wk = W.DecodeWorkload("t", batch, dim, N, 4, 40, io, seed=dim + N)
    inp = W.make_decode_inputs(wk, device=dev)
    ys, state, conv_state = _decode_all(inp, wk.steps, batch, dim, N, dev)
    chans = [(b, d) for b in range(batch) for d in range(dim)]
    ry, rh, rc, bi, di = _oracle_prefill(inp, chans, wk.steps)
    tol = 2e-5 if io == "f32" else 1e-2
    assert max_rel_err(to64(ys[:, bi, di].T), ry) <= tol
    assert max_rel_err(to64(state[bi, di]), rh) <= tol
    np.testing.assert_array_equal(to64(conv_state[bi, di]), rc)


@pytest.mark.parametrize("use_z", [True, False])
@pytest.mark.parametrize("softplus", [True, False])
def test_decode_flag_instances(use_z, softplus):
    """Every compiled instance of the bf16 decode kernel (gate or none, softplus on or off) against the
    oracle's decode step, token by token, over every channel."""
    dev = _dev()
    batch, dim, N, steps = 3, 64, 16, 20
    wk = W.DecodeWorkload("t", batch, dim, N, 4, steps, "bf16", seed=5 + 2 * use_z + softplus)
    inp = W.make_decode_inputs(wk, device=dev)
    bias = inp["delta_bias"]
    if not softplus:
        # Δ = Δ_raw without softplus: positive steps 0.05|Δ_raw| and no bias
        inp["delta"] = (inp["delta"].float().abs() * 0.05).to(inp["delta"].dtype)
        bias = None
    state = torch.zeros((batch, dim, N), device=dev)
    conv_state = torch.zeros((batch, dim, 3), device=dev)
    bidx = np.repeat(np.arange(batch, dtype=np.int64), dim)
    didx = np.tile(np.arange(dim, dtype=np.int64), batch)
    di = torch.as_tensor(didx)
    st_o = np.zeros((batch * dim, N))
    cs_o = np.zeros((batch * dim, 3))
    for t in range(steps):
        z_t = inp["z"][t] if use_z else None
        y = ssm.selective_state_update(inp["x"][t], inp["delta"][t], inp["A"], inp["B"][t], inp["C"][t], inp["D"], z_t,
                                       state, conv_state, inp["conv_w"], delta_bias=bias, delta_softplus=softplus)
        ry, st_o, cs_o = oracle.state_update(to64(inp["x"][t]).reshape(-1), to64(inp["delta"][t]).reshape(-1),
                                             to64(inp["A"])[didx], to64(inp["B"][t]), to64(inp["C"][t]), bidx, st_o, cs_o,
                                             to64(inp["conv_w"])[didx], D=to64(inp["D"])[didx],
                                             z_t=None if z_t is None else to64(z_t).reshape(-1),
                                             delta_bias=None if bias is None else to64(bias)[didx],
                                             delta_softplus=softplus)
        torch.cuda.synchronize()
        assert max_rel_err(to64(y).reshape(-1), ry) <= 1e-2, t
    assert max_rel_err(to64(state).reshape(batch * dim, N), st_o) <= 1e-2
    np.testing.assert_array_equal(to64(conv_state).reshape(batch * dim, 3), cs_o)
