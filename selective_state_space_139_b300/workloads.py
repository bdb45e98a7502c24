"""Seeded synthetic inputs for the selective scan and the decode step.

This module only draws random numbers and lays them out; it holds none of the method's
arithmetic, so both the CUDA path and the CPU oracle can be fed from it.  Every workload is
identified by name and sizes; the seed is fixed per workload.

Shapes (all contiguous):
    u, delta (Δ_raw), z : (batch, dim, L)      io dtype (float32 or bfloat16)
    B, C                : (batch, dstate, L)   io dtype
    A                   : (dim, dstate)        float32
    D, delta_bias       : (dim,)               float32
Decode step inputs are the same per token with L dropped; conv_w is (dim, 4) float32.

Distributions follow the layer shapes named on the pages (Mamba-130M: d_inner 1536; Mamba-2.8B:
d_inner 5120; d_state 16; d_conv 4):
    u, Δ_raw, z, B, C, D ~ N(0, 1)
    delta_bias = log(expm1(s)), s log-uniform in [1e-3, 1e-1]   (so that softplus(bias) = s)
    A[d, n] = -(n + 1) * scale_d, scale_d = 1 or log-uniform in [0.5, 2]
    long-sequence u[:, :, t] = E[sym_t], sym_t iid uniform over a 4-letter alphabet,
        E (4, dim) ~ N(0, 1)  (a stand-in for DNA-like symbol streams)
    conv_w ~ N(0, 1/4)
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Dict, Optional, Tuple

import torch


@dataclass(frozen=True)
class ScanWorkload:
    name: str
    batch: int
    dim: int
    dstate: int
    seqlen: int
    io_dtype: str                      # "f32" or "bf16"
    seed: int
    a_scale: Optional[Tuple[float, float]] = None   # log-uniform per-channel scale of A, or None (=1)
    symbol_alphabet: int = 0           # >0: u drawn from an alphabet mapped to fixed embeddings

    @property
    def tokens(self) -> int:
        return self.batch * self.seqlen

    @property
    def torch_dtype(self):
        return torch.float32 if self.io_dtype == "f32" else torch.bfloat16

    def algorithmic_bytes(self) -> int:
        """Reads of u, Δ, z, B, C and writes of y and the final state (fp32), plus A, D, bias."""
        e = 4 if self.io_dtype == "f32" else 2
        bdl = self.batch * self.dim * self.seqlen
        bnl = self.batch * self.dstate * self.seqlen
        return (4 * bdl + 2 * bnl) * e + self.batch * self.dim * self.dstate * 4 + \
            self.dim * self.dstate * 4 + 2 * self.dim * 4


@dataclass(frozen=True)
class DecodeWorkload:
    name: str
    batch: int
    dim: int
    dstate: int
    dconv: int
    steps: int
    io_dtype: str
    seed: int
    a_scale: Optional[Tuple[float, float]] = None

    @property
    def tokens_per_step(self) -> int:
        return self.batch

    def bytes_per_step(self) -> int:
        """State read+write (fp32), conv_state read+write (fp32), per-token io, conv weights, params."""
        e = 4 if self.io_dtype == "f32" else 2
        bd = self.batch * self.dim
        return (2 * bd * self.dstate * 4 + 2 * bd * (self.dconv - 1) * 4 + 4 * bd * e +
                2 * self.batch * self.dstate * e + self.dim * self.dconv * 4 +
                self.dim * self.dstate * 4 + 2 * self.dim * 4)


@dataclass(frozen=True)
class SsdWorkload:
    """Mamba-2 SSD layer: x (batch, L, nheads, headdim), B/C (batch, L, ngroups, dstate)."""
    name: str
    batch: int
    seqlen: int
    nheads: int
    headdim: int
    dstate: int
    ngroups: int
    seed: int
    a_range: Tuple[float, float] = (1.0, 16.0)   # -A log-uniform in this range

    @property
    def tokens(self) -> int:
        return self.batch * self.seqlen

    def algorithmic_bytes(self) -> int:
        """Reads of x, dt, B, C (bf16) and writes of y (bf16) and the final state (fp32), plus A, D, bias."""
        bl = self.batch * self.seqlen
        return (2 * bl * self.nheads * self.headdim + bl * self.nheads + 2 * bl * self.ngroups * self.dstate) * 2 + \
            self.batch * self.nheads * self.headdim * self.dstate * 4 + 3 * self.nheads * 4

    def flops(self) -> int:
        """Multiply-adds x 2 of the chunked form with 64-step chunks: C B^T (causal half), the masked
        product with x (causal half), C H^T and the state update, per (batch, head, chunk)."""
        q, p_, n = 64, self.headdim, self.dstate
        nch = (self.seqlen + q - 1) // q
        per_chunk = q * q * n // 2 + q * q * p_ // 2 + q * n * p_ + q * p_ * n
        return 2 * per_chunk * nch * self.batch * self.nheads


WORKLOADS: Dict[str, object] = {
    "tiny-f32": ScanWorkload("tiny-f32", 1, 64, 16, 256, "f32", 1000),
    "mamba130m-layer": ScanWorkload("mamba130m-layer", 8, 1536, 16, 2048, "bf16", 1001),
    "mamba2.8b-layer": ScanWorkload("mamba2.8b-layer", 4, 5120, 16, 4096, "bf16", 1002, a_scale=(0.5, 2.0)),
    "long-dna": ScanWorkload("long-dna", 1, 1536, 16, 1 << 20, "bf16", 1003, symbol_alphabet=4),
    # Mamba-2 geometry of "Модуль 8", §10: 8192 SSM channels in one B/C group, d_state 128
    # (headdim 64, so 128 heads); batch and length as the 2.8B Mamba-1 layer
    "mamba2-ssd-layer": SsdWorkload("mamba2-ssd-layer", 4, 4096, 128, 64, 128, 1, 1005),
    "ssd-small": SsdWorkload("ssd-small", 2, 300, 6, 64, 128, 1, 1006),
    # Mamba-2 decode: the SSD layer's heads, 64 sequences, 200 token steps (state 268 MB > L2)
    "mamba2-decode": SsdWorkload("mamba2-decode", 64, 200, 128, 64, 128, 1, 1007),
    "decode-2.8b": DecodeWorkload("decode-2.8b", 256, 5120, 16, 4, 1000, "bf16", 1004, a_scale=(0.5, 2.0)),
}


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _loguniform(n: int, lo: float, hi: float, g: torch.Generator, device) -> torch.Tensor:
    r = torch.rand(n, generator=g, device=device, dtype=torch.float64)
    return torch.exp(math.log(lo) + r * (math.log(hi) - math.log(lo)))


def make_params(dim: int, dstate: int, seed: int, a_scale=None, device="cpu") -> Dict[str, torch.Tensor]:
    """A (dim, dstate), D (dim), delta_bias (dim), all float32."""
    g = _gen(seed * 7919 + 17, device)
    n1 = torch.arange(1, dstate + 1, device=device, dtype=torch.float32)
    if a_scale is None:
        scale = torch.ones(dim, device=device, dtype=torch.float32)
    else:
        scale = _loguniform(dim, a_scale[0], a_scale[1], g, device).to(torch.float32)
    A = -(scale[:, None] * n1[None, :])                      # float32 products
    D = torch.randn(dim, generator=g, device=device, dtype=torch.float32)
    s = _loguniform(dim, 1e-3, 1e-1, g, device)
    delta_bias = torch.log(torch.expm1(s)).to(torch.float32)  # inverse of softplus: softplus(bias) = s
    return {"A": A.contiguous(), "D": D, "delta_bias": delta_bias}


def make_scan_inputs(w: ScanWorkload, device="cpu", seed: Optional[int] = None) -> Dict[str, torch.Tensor]:
    """All inputs of one prefill call, generated on ``device``."""
    seed = w.seed if seed is None else seed
    g = _gen(seed, device)
    dt = w.torch_dtype
    shp = (w.batch, w.dim, w.seqlen)
    out = make_params(w.dim, w.dstate, seed, w.a_scale, device)
    if w.symbol_alphabet:
        E = torch.randn(w.symbol_alphabet, w.dim, generator=g, device=device, dtype=torch.float32).to(dt)
        sym = torch.randint(0, w.symbol_alphabet, (w.batch, w.seqlen), generator=g, device=device)
        u = torch.empty(shp, device=device, dtype=dt)
        for b in range(w.batch):
            u[b] = E[sym[b]].transpose(0, 1)
        out["symbols"] = sym
        out["embedding"] = E
    else:
        u = torch.randn(shp, generator=g, device=device, dtype=torch.float32).to(dt)
    out["u"] = u.contiguous()
    out["delta"] = torch.randn(shp, generator=g, device=device, dtype=torch.float32).to(dt)
    out["z"] = torch.randn(shp, generator=g, device=device, dtype=torch.float32).to(dt)
    out["B"] = torch.randn((w.batch, w.dstate, w.seqlen), generator=g, device=device, dtype=torch.float32).to(dt)
    out["C"] = torch.randn((w.batch, w.dstate, w.seqlen), generator=g, device=device, dtype=torch.float32).to(dt)
    return out


def make_cotangent(batch: int, dim: int, seqlen: int, dtype: torch.dtype, seed: int, device="cpu") -> torch.Tensor:
    """dy (batch, dim, seqlen) ~ N(0, 1) in the io dtype: the incoming gradient of a backward call."""
    g = _gen(seed * 104729 + 3, device)
    return torch.randn((batch, dim, seqlen), generator=g, device=device, dtype=torch.float32).to(dtype).contiguous()


def make_decode_inputs(w: DecodeWorkload, steps: Optional[int] = None, device="cpu",
                       seed: Optional[int] = None) -> Dict[str, torch.Tensor]:
    """Per-token inputs for ``steps`` tokens, stacked along a leading time axis:
    x, delta, z (steps, batch, dim); B, C (steps, batch, dstate); plus A, D, delta_bias, conv_w."""
    seed = w.seed if seed is None else seed
    steps = w.steps if steps is None else steps
    g = _gen(seed, device)
    dt = torch.float32 if w.io_dtype == "f32" else torch.bfloat16
    out = make_params(w.dim, w.dstate, seed, w.a_scale, device)
    out["conv_w"] = (0.5 * torch.randn((w.dim, w.dconv), generator=g, device=device, dtype=torch.float32)).contiguous()
    shp = (steps, w.batch, w.dim)
    out["x"] = torch.randn(shp, generator=g, device=device, dtype=torch.float32).to(dt)
    out["delta"] = torch.randn(shp, generator=g, device=device, dtype=torch.float32).to(dt)
    out["z"] = torch.randn(shp, generator=g, device=device, dtype=torch.float32).to(dt)
    out["B"] = torch.randn((steps, w.batch, w.dstate), generator=g, device=device, dtype=torch.float32).to(dt)
    out["C"] = torch.randn((steps, w.batch, w.dstate), generator=g, device=device, dtype=torch.float32).to(dt)
    return out


def random_scan_inputs(batch: int, dim: int, dstate: int, seqlen: int, io_dtype: str = "f32", seed: int = 0,
                       a_scale=None, device="cpu") -> Dict[str, torch.Tensor]:
    """Ad-hoc sizes with the same distributions (parity tests on ragged shapes)."""
    w = ScanWorkload(f"adhoc-{batch}x{dim}x{dstate}x{seqlen}", batch, dim, dstate, seqlen, io_dtype, seed,
                     a_scale=a_scale)
    return make_scan_inputs(w, device=device)


def make_ssd_inputs(w: SsdWorkload, device="cpu", seed: Optional[int] = None) -> Dict[str, torch.Tensor]:
    """x, dt, B, C ~ N(0, 1) in bf16; A = -s with s log-uniform in ``a_range`` per head; D ~ N(0, 1);
    dt_bias = log(expm1(s')) with s' log-uniform in [1e-3, 0.1] (softplus(dt_bias) = s'), all float32."""
    seed = w.seed if seed is None else seed
    g = _gen(seed, device)
    bf = torch.bfloat16
    out = {
        "x": torch.randn((w.batch, w.seqlen, w.nheads, w.headdim), generator=g, device=device).to(bf),
        "dt": torch.randn((w.batch, w.seqlen, w.nheads), generator=g, device=device).to(bf),
        "B": torch.randn((w.batch, w.seqlen, w.ngroups, w.dstate), generator=g, device=device).to(bf),
        "C": torch.randn((w.batch, w.seqlen, w.ngroups, w.dstate), generator=g, device=device).to(bf),
    }
    out["A"] = -_loguniform(w.nheads, w.a_range[0], w.a_range[1], g, device).to(torch.float32)
    out["D"] = torch.randn(w.nheads, generator=g, device=device, dtype=torch.float32)
    s = _loguniform(w.nheads, 1e-3, 1e-1, g, device)
    out["dt_bias"] = torch.log(torch.expm1(s)).to(torch.float32)
    return out


def make_ssd_decode_inputs(w: SsdWorkload, device="cpu", seed: Optional[int] = None) -> Dict[str, torch.Tensor]:
    """Per-token inputs of ``w.seqlen`` Mamba-2 decode steps, stacked along a leading step axis:
    x (steps, batch, nheads, headdim), dt (steps, batch, nheads), B, C (steps, batch, ngroups, dstate),
    drawn as ``make_ssd_inputs`` draws them; A, D, dt_bias as there."""
    full = make_ssd_inputs(w, device=device, seed=seed)
    out = {k: full[k].transpose(0, 1).contiguous() for k in ("x", "dt", "B", "C")}
    out.update({k: full[k] for k in ("A", "D", "dt_bias")})
    return out


def ssd_decode_bytes_per_step(w: SsdWorkload) -> int:
    """State read + write (fp32), per-token x, dt, B, C and y (bf16), A, D, dt_bias."""
    bh = w.batch * w.nheads
    return 2 * bh * w.headdim * w.dstate * 4 + (2 * bh * w.headdim + bh + 2 * w.batch * w.ngroups * w.dstate) * 2 + \
        3 * w.nheads * 4
