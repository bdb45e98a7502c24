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
