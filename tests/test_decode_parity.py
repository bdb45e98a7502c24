"""GPU parity of the one-token decode step against the fp64 oracle.

The full-size workload (batch 256, d_inner 5120, dstate 16, 1000 tokens) runs 1000 steps on the
GPU and must match, on sampled channels, one 1000-token prefill of the same inputs by the oracle
(causal conv + SiLU, then the selective scan); the final SSM state and conv state must match too.
Small shapes (ragged dim, dstate < 16, float32 io) are compared over every channel.
"""
import numpy as np
import pytest
import torch

from selective_state_space_139_b300 import ssm
from selective_state_space_139_b300 import workloads as W
from tests._helpers import max_rel_err, sample_channels, to64

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


def test_decode_2p8b_1000_tokens_matches_prefill():
    dev = _dev()
    w = W.WORKLOADS["decode-2.8b"]
    inp = W.make_decode_inputs(w, device=dev)
    ys, state, conv_state = _decode_all(inp, w.steps, w.batch, w.dim, w.dstate, dev)
    chans = sample_channels(w.batch, w.dim, 48, seed=4)
    ry, rh, rc, bi, di = _oracle_prefill(inp, chans, w.steps)
    assert max_rel_err(to64(ys[:, bi, di].T), ry) <= 1e-2
    assert max_rel_err(to64(state[bi, di]), rh) <= 1e-2
    np.testing.assert_array_equal(to64(conv_state[bi, di]), rc)   # raw inputs, kept exactly
    assert torch.isfinite(ys).all() and torch.isfinite(state).all()


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
