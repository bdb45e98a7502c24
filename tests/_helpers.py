"""Shared test helpers: the parity metric and oracle calls on sampled channels."""
import numpy as np
import torch

import oracle


def max_rel_err(y, ref, floor_frac=1e-3):
    """max_i |y_i - r_i| / max(|r_i|, floor_frac * max_j |r_j|)  (the parity metric)."""
    y = np.asarray(y, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if ref.size == 0:
        return 0.0
    scale = max(float(np.max(np.abs(ref))), 1e-30)
    den = np.maximum(np.abs(ref), floor_frac * scale)
    return float(np.max(np.abs(y - ref) / den))


def to64(t):
    return None if t is None else t.detach().to("cpu").double().numpy()


def oracle_channels(inp, chans, delta_softplus=True, use_z=True, use_D=True, use_bias=True, h0=None,
                    discretization="delta_b", threads=0):
    """Oracle y rows and final states for the listed (b, d) channels of a prefill input dict."""
    chans = list(chans)
    bs = np.array([c[0] for c in chans], dtype=np.int64)
    ds = np.array([c[1] for c in chans], dtype=np.int64)
    bi = torch.as_tensor(bs)
    di = torch.as_tensor(ds)
    u = to64(inp["u"][bi, di])
    dl = to64(inp["delta"][bi, di])
    z = to64(inp["z"][bi, di]) if use_z and inp.get("z") is not None else None
    A = to64(inp["A"][di])
    D = to64(inp["D"][di]) if use_D and inp.get("D") is not None else None
    bias = to64(inp["delta_bias"][di]) if use_bias and inp.get("delta_bias") is not None else None
    B = to64(inp["B"])
    C = to64(inp["C"])
    h0c = None if h0 is None else to64(h0[bi, di])
    return oracle.selective_scan_channels(u, dl, A, B, C, bs, D=D, z=z, delta_bias=bias, delta_softplus=delta_softplus,
                                          h0=h0c, discretization=discretization, threads=threads)


def sample_channels(batch, dim, n, seed=0):
    rng = np.random.default_rng(seed)
    picks = {(0, 0), (batch - 1, dim - 1), (0, dim - 1), (batch - 1, 0)}
    while len(picks) < min(n, batch * dim):
        picks.add((int(rng.integers(batch)), int(rng.integers(dim))))
    return sorted(picks)
