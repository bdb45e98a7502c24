"""Host-side checks of the seeded input generator (no GPU)."""
import math

import torch

from selective_state_space_139_b300 import workloads as W


def test_named_workloads_sizes_and_bytes():
    w = W.WORKLOADS["mamba2.8b-layer"]
    assert (w.batch, w.dim, w.dstate, w.seqlen, w.io_dtype) == (4, 5120, 16, 4096, "bf16")
    # 4 bf16 (B, D, L) tensors + 2 bf16 (B, N, L) + fp32 final state + A, D, bias
    assert abs(w.algorithmic_bytes() / 1e6 - 673.8) < 0.1
    d = W.WORKLOADS["decode-2.8b"]
    assert abs(d.bytes_per_step() / 1e6 - 210.2) < 0.3
    assert W.WORKLOADS["long-dna"].seqlen == 1 << 20


def test_generator_is_deterministic_and_shaped():
    w = W.ScanWorkload("t", 2, 8, 16, 37, "bf16", 5, a_scale=(0.5, 2.0))
    a, b = W.make_scan_inputs(w), W.make_scan_inputs(w)
    for k in ("u", "delta", "z", "B", "C", "A", "D", "delta_bias"):
        assert torch.equal(a[k], b[k]), k
    assert a["u"].shape == (2, 8, 37) and a["u"].dtype == torch.bfloat16
    assert a["B"].shape == (2, 16, 37) and a["A"].shape == (8, 16) and a["A"].dtype == torch.float32
    # A[d, n] = -(n+1) * scale_d, scale in [0.5, 2]
    ratio = a["A"] / a["A"][:, :1]
    assert torch.allclose(ratio, torch.arange(1, 17, dtype=torch.float32).expand(8, 16), rtol=1e-6)
    assert bool((-a["A"][:, 0] >= 0.5).all() and (-a["A"][:, 0] <= 2.0).all())
    # softplus(bias) log-uniform in [1e-3, 1e-1]
    s = torch.nn.functional.softplus(a["delta_bias"].double())
    assert bool((s > 0.999e-3).all() and (s < 0.1001).all())


def test_symbol_stream_uses_four_embeddings():
    w = W.ScanWorkload("s", 1, 6, 16, 300, "bf16", 9, symbol_alphabet=4)
    x = W.make_scan_inputs(w)
    cols = {tuple(x["u"][0, :, t].float().tolist()) for t in range(300)}
    assert len(cols) == 4
    assert torch.equal(x["u"][0, :, 7], x["embedding"][x["symbols"][0, 7]])


def test_decode_inputs_shapes():
    d = W.DecodeWorkload("d", 3, 10, 16, 4, 5, "bf16", 3)
    x = W.make_decode_inputs(d)
    assert x["x"].shape == (5, 3, 10) and x["B"].shape == (5, 3, 16) and x["conv_w"].shape == (10, 4)
    assert abs(float(x["conv_w"].std()) - 0.5) < 0.25


def test_ssd_generators_shapes_ranges_and_determinism():
    w = W.WORKLOADS["ssd-small"]
    a = W.make_ssd_inputs(w)
    b = W.make_ssd_inputs(w)
    assert a["x"].shape == (w.batch, w.seqlen, w.nheads, w.headdim) and a["x"].dtype == torch.bfloat16
    assert a["dt"].shape == (w.batch, w.seqlen, w.nheads)
    assert a["B"].shape == a["C"].shape == (w.batch, w.seqlen, w.ngroups, w.dstate)
    for k in ("A", "D", "dt_bias"):
        assert a[k].shape == (w.nheads,) and a[k].dtype == torch.float32
    for k in a:
        assert torch.equal(a[k], b[k])                        # same seed, same tensors
    assert (a["A"] < 0).all() and (a["A"] >= -16).all() and (a["A"] <= -1).all()
    s = torch.nn.functional.softplus(a["dt_bias"].double())   # softplus(dt_bias) is the drawn step size
    assert (s >= 1e-3 * (1 - 1e-5)).all() and (s <= 0.1 * (1 + 1e-5)).all()
    assert not torch.equal(W.make_ssd_inputs(w, seed=w.seed + 1)["x"], a["x"])


def test_ssd_decode_inputs_are_the_prefill_stream_step_major():
    w = W.WORKLOADS["ssd-small"]
    full = W.make_ssd_inputs(w)
    d = W.make_ssd_decode_inputs(w)
    assert d["x"].shape == (w.seqlen, w.batch, w.nheads, w.headdim)
    for k in ("x", "dt", "B", "C"):
        assert torch.equal(d[k].transpose(0, 1), full[k])
    bh = w.batch * w.nheads
    expect = 2 * bh * 64 * 128 * 4 + (2 * bh * 64 + bh + 2 * w.batch * w.ngroups * 128) * 2 + 3 * w.nheads * 4
    assert W.ssd_decode_bytes_per_step(w) == expect
