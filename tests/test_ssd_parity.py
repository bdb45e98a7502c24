"""GPU parity of the Mamba-2 SSD forward (C ABI through the binding) against the fp64 oracle.

bf16 io with float32 accumulation and state: max relative error (floor 1e-3 of the largest
reference value) of 1e-2, the bound used for every bf16-io path.  Small and ragged shapes compare
every output; so do the full Mamba-2 layer and the full decode workload, in the configurations the
benchmark times.  The balanced schedule (sequences split between CTAs, the state carried through the
workspace) is compared with one CTA per sequence bit for bit and with the oracle.
"""
import numpy as np
import pytest
import torch

from selective_state_space_139_b300 import ssm
from selective_state_space_139_b300 import workloads as W
from tests._helpers import max_rel_err, to64

import oracle

pytestmark = pytest.mark.gpu

TOL = 1e-2


def _dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


def _oracle(inp, use_D=True, use_bias=True, softplus=True, h0=None):
    return oracle.ssd_scan(to64(inp["x"]), to64(inp["dt"]), to64(inp["A"]), to64(inp["B"]), to64(inp["C"]),
                           D=to64(inp["D"]) if use_D else None, dt_bias=to64(inp["dt_bias"]) if use_bias else None,
                           dt_softplus=softplus, h0=None if h0 is None else to64(h0))


def _run(inp, use_D=True, use_bias=True, softplus=True, h0=None):
    y, hT = ssm.ssd_fwd(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], D=inp["D"] if use_D else None,
                        dt_bias=inp["dt_bias"] if use_bias else None, dt_softplus=softplus, h0=h0)
    torch.cuda.synchronize()
    return y, hT


def _check(y, hT, ry, rh):
    ey, eh = max_rel_err(to64(y), ry), max_rel_err(to64(hT), rh)
    assert ey <= TOL and eh <= TOL, (ey, eh)
    return ey, eh


def test_ssd_small_full():
    dev = _dev()
    inp = W.make_ssd_inputs(W.WORKLOADS["ssd-small"], device=dev)
    y, hT = _run(inp)
    _check(y, hT, *_oracle(inp))


@pytest.mark.parametrize("L", [1, 63, 64, 65, 200])
def test_ssd_ragged_lengths(L):
    dev = _dev()
    w = W.SsdWorkload("adhoc", 2, L, 3, 64, 128, 1, 2000 + L)
    inp = W.make_ssd_inputs(w, device=dev)
    y, hT = _run(inp)
    _check(y, hT, *_oracle(inp))


def test_ssd_groups_h0_and_options():
    dev = _dev()
    w = W.SsdWorkload("adhoc", 2, 150, 6, 64, 128, 3, 2101)
    inp = W.make_ssd_inputs(w, device=dev)
    g = torch.Generator(device=dev)
    g.manual_seed(7)
    h0 = torch.randn((2, 6, 64, 128), generator=g, device=dev)
    y, hT = _run(inp, h0=h0)
    _check(y, hT, *_oracle(inp, h0=h0))
    y, hT = _run(inp, use_D=False, use_bias=False)
    _check(y, hT, *_oracle(inp, use_D=False, use_bias=False))
    inp["dt"] = (inp["dt"].float().abs() * 0.05).to(torch.bfloat16)      # positive steps without softplus
    y, hT = _run(inp, softplus=False, use_bias=False)     # (the bias is negative: it would make Δ < 0)
    _check(y, hT, *_oracle(inp, softplus=False, use_bias=False))


def test_ssd_mamba2_layer_full():
    """Every output of the Mamba-2 SSD layer (batch 4, L 4096, 128 heads x 64, d_state 128)."""
    dev = _dev()
    w = W.WORKLOADS["mamba2-ssd-layer"]
    inp = W.make_ssd_inputs(w, device=dev)
    y, hT = _run(inp)
    assert torch.isfinite(y).all()
    _check(y, hT, *_oracle(inp))


def _run_sched(inp, balanced, ctas=0, h0=None):
    y, hT = ssm.ssd_fwd(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], D=inp["D"], dt_bias=inp["dt_bias"],
                        h0=h0, balanced=balanced, ctas=ctas)
    torch.cuda.synchronize()
    assert ssm.device_status() == ssm.SSM_OK
    return y, hT


@pytest.mark.parametrize("ctas", [1, 2, 3, 5, 7])
def test_ssd_balanced_ranges_match_one_cta_per_sequence(ctas, L=293):
    """The balanced schedule on 8 sequences (batch 2 x 4 heads, 2 groups) of 5 chunks, the last one
    ragged (L 293), cut into at most `ctas` ranges: with 3, 5 or 7 ranges the cuts fall inside
    sequences, so heads are published, tails continue from the carried state and whole sequences
    run in between; one range runs every sequence in one CTA.  The per-chunk arithmetic is the same
    and the carried state is exact float32, so y and the final state equal those of one CTA per
    sequence bit for bit, and both match the oracle, with h0 given and without."""
    dev = _dev()
    w = W.SsdWorkload("adhoc", 2, L, 4, 64, 128, 2, 2400 + L)
    inp = W.make_ssd_inputs(w, device=dev)
    assert ssm.ssd_workspace_size(2, L, 4, ctas) > 0
    g = torch.Generator(device=dev)
    g.manual_seed(11)
    for h0 in (None, torch.randn((2, 4, 64, 128), generator=g, device=dev)):
        yg, hg = _run_sched(inp, balanced=False, h0=h0)
        yb, hb = _run_sched(inp, balanced=True, ctas=ctas, h0=h0)
        assert torch.equal(yb, yg) and torch.equal(hb, hg)
        _check(yb, hb, *_oracle(inp, h0=h0))


@pytest.mark.parametrize("L,ctas", [(1, 3), (64, 3), (65, 7), (640, 3)])
def test_ssd_balanced_lengths(L, ctas):
    """The balanced schedule at one chunk (every range whole sequences), exactly one chunk, one step
    into a second chunk, and ten chunks per sequence."""
    test_ssd_balanced_ranges_match_one_cta_per_sequence(ctas, L)


def test_ssd_workspace_size_and_one_wave_shapes():
    """No workspace when the sequences fit in one wave of resident CTAs (or in `ctas`), a carry per
    range otherwise; the workload's 512 sequences take the balanced schedule on a B300."""
    _dev()
    assert ssm.ssd_workspace_size(2, 293, 4, 8) == 0           # 8 sequences on up to 8 ranges
    assert ssm.ssd_workspace_size(2, 293, 4, 0) == 0           # fewer sequences than resident CTAs
    ws = ssm.ssd_workspace_size(2, 293, 4, 3)
    assert ws >= 3 * 64 * 128 * 4 + 4 * 4 and ws % 256 == 0   # carries, flags, range counter
    w = W.WORKLOADS["mamba2-ssd-layer"]
    assert ssm.ssd_workspace_size(w.batch, w.seqlen, w.nheads) > 0
    lib = ssm.load_library()
    assert lib.ssm_ssd_fwd_workspace_size(0, 293, 4, 0) == 0 and lib.ssm_ssd_fwd_workspace_size(2, 293, 4, -1) == 0


def test_ssd_balanced_rejects_a_small_workspace():
    dev = _dev()
    w = W.SsdWorkload("adhoc", 2, 293, 4, 64, 128, 2, 2401)
    inp = W.make_ssd_inputs(w, device=dev)
    need = ssm.ssd_workspace_size(2, 293, 4, 3)
    small = torch.empty(need - 256, dtype=torch.uint8, device=dev)
    y = torch.empty_like(inp["x"])
    lib = ssm.load_library()
    st = lib.ssm_ssd_fwd_ex(inp["x"].data_ptr(), inp["dt"].data_ptr(), inp["A"].data_ptr(), inp["B"].data_ptr(),
                            inp["C"].data_ptr(), None, None, 1, None, y.data_ptr(), None, 2, 293, 4, 64, 128, 2,
                            ssm.SSM_BF16, small.data_ptr(), need - 256, 3, None)
    assert st == ssm.SSM_ERR_INVALID_ARG


def test_ssd_seqlen_zero_passes_the_state_through():
    dev = _dev()
    w = W.SsdWorkload("adhoc", 1, 0, 2, 64, 128, 1, 2200)
    inp = W.make_ssd_inputs(w, device=dev)
    h0 = torch.randn((1, 2, 64, 128), device=dev)
    y, hT = _run(inp, h0=h0)
    assert y.numel() == 0 and torch.equal(hT, h0)


def test_ssd_rejects_cpu_tensors_and_other_sizes():
    dev = _dev()
    w = W.SsdWorkload("adhoc", 1, 16, 2, 64, 128, 1, 2300)
    cpu = W.make_ssd_inputs(w)
    with pytest.raises(ValueError):
        ssm.ssd_fwd(cpu["x"], cpu["dt"], cpu["A"], cpu["B"], cpu["C"])
    inp = W.make_ssd_inputs(W.SsdWorkload("adhoc", 1, 16, 2, 32, 128, 1, 2301), device=dev)
    with pytest.raises(ssm.SSMError):
        ssm.ssd_fwd(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"])


# ---------------------------------------------------------------- the Mamba-2 decode step

def _decode_steps(d, state, first, count, use_D=True, use_bias=True):
    ys = []
    for t in range(first, first + count):
        ys.append(ssm.ssd_state_update(d["x"][t], d["dt"][t], d["A"], d["B"][t], d["C"][t], state,
                                       D=d["D"] if use_D else None, dt_bias=d["dt_bias"] if use_bias else None))
    torch.cuda.synchronize()
    return torch.stack(ys, dim=1)   # (batch, steps, nheads, headdim)


@pytest.mark.parametrize("groups", [1, 2])
def test_ssd_decode_steps_match_the_recurrence(groups):
    dev = _dev()
    w = W.SsdWorkload("adhoc", 3, 20, 6, 64, 128, groups, 2400 + groups)
    d = W.make_ssd_decode_inputs(w, device=dev)
    g = torch.Generator(device=dev)
    g.manual_seed(9)
    h0 = torch.randn((3, 6, 64, 128), generator=g, device=dev)
    state = h0.clone()
    y = _decode_steps(d, state, 0, w.seqlen)
    full = {k: d[k].transpose(0, 1) for k in ("x", "dt", "B", "C")}
    ry, rh = oracle.ssd_scan(to64(full["x"]), to64(full["dt"]), to64(d["A"]), to64(full["B"]), to64(full["C"]),
                             D=to64(d["D"]), dt_bias=to64(d["dt_bias"]), h0=to64(h0))
    _check(y, state, ry, rh)


def test_ssd_prefill_then_decode_equals_longer_prefill():
    """ssm_ssd_fwd over 150 tokens, then 30 decode steps from its final state, against the oracle
    recurrence over all 180 tokens."""
    dev = _dev()
    w = W.SsdWorkload("adhoc", 2, 180, 4, 64, 128, 1, 2500)
    inp = W.make_ssd_inputs(w, device=dev)
    L1 = 150
    pre = {k: inp[k][:, :L1].contiguous() for k in ("x", "dt", "B", "C")}
    y1, state = ssm.ssd_fwd(pre["x"], pre["dt"], inp["A"], pre["B"], pre["C"], D=inp["D"], dt_bias=inp["dt_bias"])
    dec = {k: inp[k][:, L1:].transpose(0, 1).contiguous() for k in ("x", "dt", "B", "C")}
    dec.update({k: inp[k] for k in ("A", "D", "dt_bias")})
    y2 = _decode_steps(dec, state, 0, w.seqlen - L1)
    ry, rh = oracle.ssd_scan(to64(inp["x"]), to64(inp["dt"]), to64(inp["A"]), to64(inp["B"]), to64(inp["C"]),
                             D=to64(inp["D"]), dt_bias=to64(inp["dt_bias"]))
    _check(torch.cat([y1, y2], dim=1), state, ry, rh)


def test_ssd_decode_workload_full():
    """Every output of the Mamba-2 decode workload (64 sequences x 128 heads, 200 token steps) against
    one oracle prefill of the same token stream."""
    dev = _dev()
    w = W.WORKLOADS["mamba2-decode"]
    d = W.make_ssd_decode_inputs(w, device=dev)
    state = torch.zeros((w.batch, w.nheads, w.headdim, w.dstate), device=dev)
    y = _decode_steps(d, state, 0, w.seqlen)
    full = {k: d[k].transpose(0, 1) for k in ("x", "dt", "B", "C")}
    ry, rh = oracle.ssd_scan(to64(full["x"]), to64(full["dt"]), to64(d["A"]), to64(full["B"]), to64(full["C"]),
                             D=to64(d["D"]), dt_bias=to64(d["dt_bias"]))
    _check(y, state, ry, rh)
