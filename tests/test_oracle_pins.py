"""Pins for the fp64 oracle: each check ties it to something other than itself.

* the pages' worked examples (``tests/golden/``): the affine composition (2,1)∘(3,4) and the
  ZOH-vs-ΔB gap of 10% at Δ ≈ 0.193747558 ("Модуль 8. Альтернативы Transformer", §7 and §5);
* closed forms: A = 0 turns the scan into Δ-weighted prefix sums (numpy cumsum); the page's
  closed-form prefix h_t = Σ_j (Π_{i>j} Ā_i) B̄_j x_j as an O(L²) brute force with general
  diagonal A ("State Space Models: Mamba и альтернатива Transformer", "SSM Scan Algorithm";
  the semi-separable matrix of "Модуль 8", §7);
* special cases that reduce to a library routine: constant Δ, B, C give the LTI convolution
  y = K*u with K_k = Σ_n C_n Ā_n^k Δ B_n ("State Space Models…", "S4: Structured State Space"),
  evaluated with numpy.convolve; the causal conv against numpy.convolve;
* invariants: zero input gives zero output and state; z = 0 gives y = 0; softplus(v) - softplus(-v) = v
  and SiLU(z) - SiLU(-z) = z; Δ = 0 keeps h; Δ|A| ≫ 1 resets h to ΔBu;
* the chunked (aggregate/carry/re-run) form equals the sequential one for every chunk length;
* a prefill followed by decode steps equals one longer prefill ("Модуль 8", §6/§14 caches);
* the backward (reverse-mode) oracle against central finite differences of sum(dy * y) for every
  input, with and without softplus, gate and skip, and against the exact gradient of the A = 0,
  no-gate case (y is then linear in u);
* the Mamba-2 SSD oracle (recurrence and chunked block form) against the semi-separable matrix
  M_ij = C_i·B_j Π_{r=j+1..i} a_r Δ_j written out as an O(L²) brute force ("Модуль 8", §7), against
  the already pinned Mamba-1 oracle (each (head, p) row is a Mamba-1 channel whose A row repeats the
  head's scalar), and against numpy prefix sums when A = 0.

Each mistake a plausible bug would make (a dropped D term, a sign error in the exponent, reading
before updating, swapping B and C, the gate before the D skip, the conv tap order) fails at
least one of these; ``test_planted_mistakes_are_caught`` checks that on mutated copies of the C
source.
"""
import math
import os
import shutil
import subprocess
import tempfile

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


def _rand_problem(rng, batch=2, dim=3, N=4, L=20, general_A=False):
    u = rng.standard_normal((batch, dim, L))
    delta = rng.standard_normal((batch, dim, L))
    if general_A:
        A = -np.exp(rng.standard_normal((dim, N)))
    else:
        A = -np.tile(np.arange(1, N + 1, dtype=np.float64), (dim, 1)) * rng.uniform(0.5, 2, (dim, 1))
    B = rng.standard_normal((batch, N, L))
    C = rng.standard_normal((batch, N, L))
    D = rng.standard_normal(dim)
    z = rng.standard_normal((batch, dim, L))
    bias = np.log(np.expm1(rng.uniform(1e-3, 1e-1, dim)))
    return dict(u=u, delta=delta, A=A, B=B, C=C, D=D, z=z, delta_bias=bias)


def _load_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append([float(x) for x in line.split()])
    return rows


# ---------------------------------------------------------------- the pages' worked examples

def test_compose_worked_example():
    for la, lb, ea, eb, ra, rb in _load_golden("affine_compose.txt"):
        assert oracle.compose_affine((la, lb), (ea, eb)) == (ra, rb)


def test_zoh_epsilon_worked_example():
    (a, b, dlt, eps, tol), = _load_golden("zoh_epsilon.txt")
    # one step from h = 0 with x = 1, C = 1, no D, no gate, Δ given directly (softplus off)
    kw = dict(u=np.ones((1, 1, 1)), delta=np.full((1, 1, 1), dlt), A=np.full((1, 1), a),
              B=np.full((1, 1, 1), b), C=np.ones((1, 1, 1)), delta_softplus=False)
    y_db, _ = oracle.selective_scan(**kw)
    y_zoh, _ = oracle.selective_scan(**kw, discretization="zoh")
    with np.errstate(divide="ignore", invalid="ignore"):   # a planted mistake can make y_zoh zero
        ratio = y_db[0, 0, 0] / y_zoh[0, 0, 0]
    assert abs(ratio - 1 - eps) < tol
    # and ε grows with Δ (the page's table direction): smaller step, smaller gap
    kw["delta"] = np.full((1, 1, 1), dlt / 4)
    y_db2, _ = oracle.selective_scan(**kw)
    y_zoh2, _ = oracle.selective_scan(**kw, discretization="zoh")
    assert 0 < y_db2[0, 0, 0] / y_zoh2[0, 0, 0] - 1 < eps


def test_zoh_a_to_zero_limit():
    # (e^{Δa} - 1)/a -> Δ as a -> 0, and a = 0 exactly must not produce a NaN (§4).
    for a in (0.0, 1e-300, -1e-12):
        kw = dict(u=np.ones((1, 1, 1)), delta=np.full((1, 1, 1), 0.7), A=np.full((1, 1), a),
                  B=np.full((1, 1, 1), 2.0), C=np.ones((1, 1, 1)), delta_softplus=False)
        y, _ = oracle.selective_scan(**kw, discretization="zoh")
        assert np.isfinite(y).all()
        assert abs(y[0, 0, 0] - 0.7 * 2.0) < 1e-10


# ---------------------------------------------------------------- closed forms

def test_a_zero_is_delta_weighted_prefix_sum():
    rng = _rng(1)
    p = _rand_problem(rng, L=33)
    p["A"] = np.zeros_like(p["A"])
    y, hL = oracle.selective_scan(**p)
    v = p["delta"] + p["delta_bias"][None, :, None]
    dlt = np.logaddexp(0.0, v)                                   # log(1 + e^v)
    w = dlt * p["u"]                                             # (b, d, L)
    h = np.cumsum(w[:, :, None, :] * p["B"][:, None, :, :], axis=-1)   # (b, d, N, L)
    s = np.einsum("bnl,bdnl->bdl", p["C"], h) + p["D"][None, :, None] * p["u"]
    ref = s * p["z"] / (1 + np.exp(-p["z"]))
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(hL, h[..., -1], rtol=1e-12, atol=1e-12)


def test_semiseparable_bruteforce_general_A():
    rng = _rng(2)
    p = _rand_problem(rng, batch=2, dim=3, N=5, L=40, general_A=True)
    y, hL = oracle.selective_scan(**p)
    dlt = np.logaddexp(0.0, p["delta"] + p["delta_bias"][None, :, None])
    bsz, dim, L = p["u"].shape
    ref = np.zeros_like(y)
    for b in range(bsz):
        for d in range(dim):
            S = np.concatenate([[0.0], np.cumsum(dlt[b, d])])   # S[i+1] = Σ_{r<=i} Δ_r
            for i in range(L):
                acc = 0.0
                for j in range(i + 1):
                    decay = np.exp(p["A"][d] * (S[i + 1] - S[j + 1]))   # Π_{r=j+1..i} exp(Δ_r A)
                    acc += np.sum(p["C"][b, :, i] * decay * dlt[b, d, j] * p["B"][b, :, j]) * p["u"][b, d, j]
                acc += p["D"][d] * p["u"][b, d, i]
                zz = p["z"][b, d, i]
                ref[b, d, i] = acc * zz / (1 + np.exp(-zz))
    np.testing.assert_allclose(y, ref, rtol=1e-10, atol=1e-12)


def test_lti_reduces_to_convolution():
    rng = _rng(3)
    N, L = 4, 50
    A = -rng.uniform(0.2, 2.0, (1, N))
    dlt = 0.3
    Bn = rng.standard_normal(N)
    Cn = rng.standard_normal(N)
    Dd = 0.7
    u = rng.standard_normal((1, 1, L))
    y, _ = oracle.selective_scan(u=u, delta=np.full((1, 1, L), dlt), A=A,
                                 B=np.repeat(Bn[None, :, None], L, axis=2),
                                 C=np.repeat(Cn[None, :, None], L, axis=2), D=np.array([Dd]),
                                 delta_softplus=False)
    Abar = np.exp(dlt * A[0])
    K = np.array([np.sum(Cn * Abar ** k * dlt * Bn) for k in range(L)])
    ref = np.convolve(u[0, 0], K)[:L] + Dd * u[0, 0]
    np.testing.assert_allclose(y[0, 0], ref, rtol=1e-11, atol=1e-12)


# ---------------------------------------------------------------- invariants

def test_zero_input_and_zero_gate():
    rng = _rng(4)
    p = _rand_problem(rng)
    p0 = dict(p, u=np.zeros_like(p["u"]))
    y, hL = oracle.selective_scan(**p0)
    assert np.all(y == 0) and np.all(hL == 0)
    pz = dict(p, z=np.zeros_like(p["z"]))
    y, hL = oracle.selective_scan(**pz)
    assert np.all(y == 0) and np.any(hL != 0)


def test_softplus_and_silu_identities():
    # single step, A = 0, B = C = u = 1, D = 0, no gate: y = softplus(v)
    vs = np.array([-40.0, -3.0, -0.5, 0.0, 0.5, 3.0, 40.0])
    n = len(vs)

    def one_step(v, z=None):
        y, _ = oracle.selective_scan_channels(u=np.ones((n, 1)), delta=v[:, None], A=np.zeros((n, 1)),
                                              B=np.ones((1, 1, 1)), C=np.ones((1, 1, 1)),
                                              bidx=np.zeros(n, np.int64), z=z)
        return y[:, 0]

    sp, spm = one_step(vs), one_step(-vs)
    np.testing.assert_allclose(sp - spm, vs, rtol=0, atol=1e-14)      # softplus(v) - softplus(-v) = v
    assert abs(sp[3] - math.log(2.0)) < 1e-15                           # softplus(0) = ln 2
    assert abs(sp[0] / math.exp(-40.0) - 1) < 1e-15                     # softplus(v) ~ e^v as v -> -inf
    assert np.all(sp > 0)
    zs = np.linspace(-6, 6, n)
    g_plus = one_step(np.zeros(n), z=zs[:, None]) / math.log(2.0)
    g_minus = one_step(np.zeros(n), z=-zs[:, None]) / math.log(2.0)
    np.testing.assert_allclose(g_plus - g_minus, zs, atol=1e-14)       # SiLU(z) - SiLU(-z) = z
    assert abs(one_step(np.zeros(1)[:1].repeat(n), z=np.zeros((n, 1)))[0]) == 0.0


def test_zero_step_keeps_state_and_large_step_resets_it():
    rng = _rng(5)
    N = 3
    h0 = rng.standard_normal((1, 1, N))
    A = -np.array([[1.0, 2.0, 3.0]])
    B = rng.standard_normal((1, N, 1))
    C = rng.standard_normal((1, N, 1))
    kw = dict(u=np.full((1, 1, 1), 0.8), A=A, B=B, C=C, delta_softplus=False, h0=h0)
    _, h = oracle.selective_scan(delta=np.zeros((1, 1, 1)), **kw)
    np.testing.assert_array_equal(h, h0)                               # Δ = 0: h unchanged
    big = 800.0
    _, h = oracle.selective_scan(delta=np.full((1, 1, 1), big), **kw)
    np.testing.assert_allclose(h[0, 0], big * B[0, :, 0] * 0.8, rtol=1e-15)   # forget all, write ΔBu


def test_update_before_read_and_gate_after_skip():
    # one step from h0 = 0: y_0 = (C·(Δ B u) + D u) * SiLU(z) -- catches read-before-update and gate placement
    N = 2
    B = np.array([[[0.5], [-1.5]]])
    C = np.array([[[2.0], [0.25]]])
    u, dl, D, z = 1.3, 0.4, -0.6, 0.9
    y, _ = oracle.selective_scan(u=np.full((1, 1, 1), u), delta=np.full((1, 1, 1), dl), A=-np.ones((1, N)),
                                 B=B, C=C, D=np.array([D]), z=np.full((1, 1, 1), z), delta_softplus=False)
    s = (2.0 * 0.5 + 0.25 * -1.5) * dl * u + D * u
    assert abs(y[0, 0, 0] - s * z / (1 + math.exp(-z))) < 1e-15


def test_batch_index_selects_b_and_c():
    rng = _rng(6)
    p = _rand_problem(rng, batch=3, dim=2)
    y, hL = oracle.selective_scan(**p)
    for b in range(3):
        q = {k: (v[b:b + 1] if k in ("u", "delta", "z", "B", "C") else v) for k, v in p.items()}
        yb, hb = oracle.selective_scan(**q)
        np.testing.assert_array_equal(yb[0], y[b])
        np.testing.assert_array_equal(hb[0], hL[b])


# ---------------------------------------------------------------- chunked form

@pytest.mark.parametrize("chunk", [1, 2, 3, 7, 32, 61, 1000])
def test_chunked_equals_sequential(chunk):
    rng = _rng(7)
    p = _rand_problem(rng, batch=2, dim=3, N=6, L=61)
    p["h0"] = rng.standard_normal((2, 3, 6))
    y, hL = oracle.selective_scan(**p)
    yc, hc = oracle.chunked_scan(chunk=chunk, **p)
    np.testing.assert_allclose(yc, y, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(hc, hL, rtol=1e-12, atol=1e-13)


def test_h0_continues_a_split_sequence():
    rng = _rng(8)
    p = _rand_problem(rng, L=40)
    y, hL = oracle.selective_scan(**p)
    cut = 17
    first = {k: (v[..., :cut] if k in ("u", "delta", "z", "B", "C") else v) for k, v in p.items()}
    second = {k: (v[..., cut:] if k in ("u", "delta", "z", "B", "C") else v) for k, v in p.items()}
    y1, h1 = oracle.selective_scan(**first)
    y2, h2 = oracle.selective_scan(h0=h1, **second)
    np.testing.assert_allclose(np.concatenate([y1, y2], -1), y, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(h2, hL, rtol=1e-13, atol=1e-14)


# ---------------------------------------------------------------- conv and decode

def test_causal_conv_matches_numpy_convolve():
    rng = _rng(9)
    n, L, K = 3, 25, 4
    x = rng.standard_normal((n, L))
    w = rng.standard_normal((n, K))
    out, st = oracle.causal_conv1d(x, w, silu=False)
    for c in range(n):
        ref = np.convolve(x[c], w[c][::-1])[:L]      # cross-correlation with K-1 zeros in front
        np.testing.assert_allclose(out[c], ref, rtol=1e-13, atol=1e-14)
    np.testing.assert_array_equal(st, x[:, -(K - 1):])
    out2, _ = oracle.causal_conv1d(x, w, silu=True)
    np.testing.assert_allclose(out2 - oracle.causal_conv1d(-x, w, silu=True)[0], out, atol=1e-13)


def test_decode_window_orientation():
    # conv_state holds the last K-1 inputs oldest first and w[K-1] multiplies the newest input
    cs = np.array([[10.0, 20.0, 30.0]])
    for k, expect in enumerate([10.0, 20.0, 30.0, 40.0]):
        w = np.zeros((1, 4))
        w[0, k] = 1.0
        y, st, cs2 = oracle.state_update(x_t=np.array([40.0]), delta_t=np.array([0.0]), A=np.zeros((1, 1)),
                                         B_t=np.ones((1, 1)), C_t=np.ones((1, 1)), bidx=np.zeros(1, np.int64),
                                         state=np.zeros((1, 1)), conv_state=cs, conv_w=w, delta_softplus=False)
        assert st[0, 0] == 0.0 and y[0] == 0.0          # Δ = 0: nothing written
        np.testing.assert_array_equal(cs2, [[20.0, 30.0, 40.0]])
        y, st, _ = oracle.state_update(x_t=np.array([40.0]), delta_t=np.array([1.0]), A=np.zeros((1, 1)),
                                       B_t=np.ones((1, 1)), C_t=np.ones((1, 1)), bidx=np.zeros(1, np.int64),
                                       state=np.zeros((1, 1)), conv_state=cs, conv_w=w, delta_softplus=False)
        assert abs(st[0, 0] - expect / (1 + math.exp(-expect))) < 1e-12


def test_prefill_then_decode_equals_longer_prefill():
    rng = _rng(10)
    batch, dim, N, K, L1, L2 = 2, 3, 5, 4, 13, 9
    L = L1 + L2
    x = rng.standard_normal((batch, dim, L))
    w = 0.5 * rng.standard_normal((dim, K))
    p = _rand_problem(rng, batch=batch, dim=dim, N=N, L=L)
    wfull = np.tile(w, (batch, 1))
    # one prefill over L tokens: conv + SiLU, then the scan
    u, _ = oracle.causal_conv1d(x.reshape(-1, L), wfull)
    y_ref, h_ref = oracle.selective_scan(**dict(p, u=u.reshape(batch, dim, L)))
    # prefill L1 tokens, then L2 decode steps from (last_state, conv tail)
    u1, cs = oracle.causal_conv1d(x[..., :L1].reshape(-1, L1), wfull)
    first = {k: (v[..., :L1] if k in ("delta", "z", "B", "C") else v) for k, v in p.items()}
    first["u"] = u1.reshape(batch, dim, L1)
    y1, h = oracle.selective_scan(**first)
    h = h.reshape(-1, N)
    bidx = np.repeat(np.arange(batch), dim)
    A_c = np.tile(p["A"], (batch, 1))
    D_c = np.tile(p["D"], batch)
    b_c = np.tile(p["delta_bias"], batch)
    ys = []
    for t in range(L1, L):
        yt, h, cs = oracle.state_update(x_t=x[..., t].reshape(-1), delta_t=p["delta"][..., t].reshape(-1), A=A_c,
                                        B_t=p["B"][..., t], C_t=p["C"][..., t], bidx=bidx, state=h,
                                        conv_state=cs, conv_w=wfull, D=D_c, z_t=p["z"][..., t].reshape(-1),
                                        delta_bias=b_c)
        ys.append(yt.reshape(batch, dim))
    y = np.concatenate([y1, np.stack(ys, -1)], -1)
    np.testing.assert_allclose(y, y_ref, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(h.reshape(batch, dim, N), h_ref, rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------- backward: finite differences

@pytest.mark.parametrize("softplus,gate,skip", [(True, True, True), (False, False, False), (True, False, True)])
def test_backward_matches_central_differences(softplus, gate, skip):
    rng = _rng(11)
    b, d, N, L = 2, 3, 5, 12
    u = rng.standard_normal((b, d, L))
    dl = rng.standard_normal((b, d, L)) if softplus else rng.uniform(0.05, 0.5, (b, d, L))
    A = -np.exp(rng.standard_normal((d, N)))
    B = rng.standard_normal((b, N, L))
    C = rng.standard_normal((b, N, L))
    D = rng.standard_normal(d) if skip else None
    z = rng.standard_normal((b, d, L)) if gate else None
    bias = 0.3 * rng.standard_normal(d) if softplus else None
    dy = rng.standard_normal((b, d, L))
    g = oracle.scan_backward(u, dl, A, B, C, dy, D=D, z=z, delta_bias=bias, delta_softplus=softplus)
    base = dict(u=u, delta=dl, A=A, B=B, C=C, D=D, z=z, delta_bias=bias, delta_softplus=softplus)

    def loss(**kw):
        y, _ = oracle.selective_scan(**dict(base, **kw))
        return float((y * dy).sum())

    eps = 1e-6
    checks = [("u", "du"), ("delta", "ddelta"), ("A", "dA"), ("B", "dB"), ("C", "dC")]
    if gate:
        checks.append(("z", "dz"))
    if skip:
        checks.append(("D", "dD"))
    if softplus:
        checks.append(("delta_bias", "ddelta_bias"))
    for name, key in checks:
        arr = base[name]
        for _ in range(6):
            idx = tuple(int(rng.integers(n)) for n in arr.shape)
            hi, lo = arr.copy(), arr.copy()
            hi[idx] += eps
            lo[idx] -= eps
            fd = (loss(**{name: hi}) - loss(**{name: lo})) / (2 * eps)
            assert abs(fd - g[key][idx]) <= 1e-7 * max(1.0, abs(fd)), (name, idx, fd, g[key][idx])


def test_backward_of_a_linear_input_is_exact():
    # y is linear in u when Δ does not depend on u: with A = 0, no gate and no D,
    # dL/du_t = Σ_{s >= t} dy_s Δ_t C_s·B_t exactly (the prefix-sum closed form read backwards)
    rng = _rng(12)
    L, N = 10, 3
    u = rng.standard_normal((1, 1, L))
    dl = rng.uniform(0.1, 1.0, (1, 1, L))
    B = rng.standard_normal((1, N, L))
    C = rng.standard_normal((1, N, L))
    dy = rng.standard_normal((1, 1, L))
    g = oracle.scan_backward(u, dl, np.zeros((1, N)), B, C, dy, delta_softplus=False)
    ref = np.array([sum(dy[0, 0, s] * dl[0, 0, t] * float(C[0, :, s] @ B[0, :, t]) for s in range(t, L))
                    for t in range(L)])
    np.testing.assert_allclose(g["du"][0, 0], ref, rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------- Mamba-2 SSD ("Модуль 8", §7)

def _ssd_inputs(seed, batch=2, L=29, nheads=4, headdim=3, dstate=5, ngroups=2, a_zero=False):
    r = _rng(seed)
    x = r.standard_normal((batch, L, nheads, headdim))
    dt = r.standard_normal((batch, L, nheads))
    A = np.zeros(nheads) if a_zero else -r.uniform(0.5, 2.0, nheads)
    B = r.standard_normal((batch, L, ngroups, dstate))
    C = r.standard_normal((batch, L, ngroups, dstate))
    D = r.standard_normal(nheads)
    bias = r.standard_normal(nheads) - 1.0
    h0 = r.standard_normal((batch, nheads, headdim, dstate))
    return x, dt, A, B, C, D, bias, h0


def _ssd_bruteforce(x, dt, A, B, C, D, bias, h0):
    """y = M x with M_ij = (C_i·B_j) Π_{r=j+1..i} a_r Δ_j for i ≥ j, plus the initial state read through
    (Π_{r≤i} a_r) C_i, plus D x: the semi-separable matrix written out, O(L²) per head."""
    batch, L, nheads, P = x.shape
    G = B.shape[2]
    y = np.zeros_like(x)
    for b in range(batch):
        for h in range(nheads):
            g = h // (nheads // G)
            dl = np.logaddexp(0.0, dt[b, :, h] + bias[h])
            a = np.exp(dl * A[h])
            for i in range(L):
                for j in range(i + 1):
                    m = float(C[b, i, g] @ B[b, j, g]) * float(np.prod(a[j + 1:i + 1])) * dl[j]
                    y[b, i, h] += m * x[b, j, h]
                y[b, i, h] += float(np.prod(a[:i + 1])) * (h0[b, h] @ C[b, i, g]) + D[h] * x[b, i, h]
    return y


def test_ssd_matches_semiseparable_bruteforce():
    args = _ssd_inputs(31)
    ref = _ssd_bruteforce(*args)
    x, dt, A, B, C, D, bias, h0 = args
    for chunk in (None, 4):
        y, _ = oracle.ssd_scan(x, dt, A, B, C, D=D, dt_bias=bias, h0=h0, chunk=chunk)
        assert np.max(np.abs(y - ref)) <= 1e-10 * max(1.0, np.max(np.abs(ref))), chunk


def test_ssd_reduces_to_mamba1_channels():
    """Each (head, p) row of the SSD is a Mamba-1 channel whose A row is the head's scalar repeated
    over the states, with the head's Δ and the group's B and C."""
    x, dt, A, B, C, D, bias, h0 = _ssd_inputs(32)
    batch, L, nheads, P = x.shape
    G, N = B.shape[2], B.shape[3]
    y, hT = oracle.ssd_scan(x, dt, A, B, C, D=D, dt_bias=bias, h0=h0)
    rows = [(b, h, q) for b in range(batch) for h in range(nheads) for q in range(P)]
    u = np.array([x[b, :, h, q] for b, h, q in rows])
    dl = np.array([dt[b, :, h] for b, h, q in rows])
    Ar = np.array([np.full(N, A[h]) for b, h, q in rows])
    Bm = np.stack([B[b, :, g].T for b in range(batch) for g in range(G)])     # (batch*G, N, L)
    bidx = np.array([b * G + h // (nheads // G) for b, h, q in rows])
    y1, h1 = oracle.selective_scan_channels(u, dl, Ar, Bm, np.stack([C[b, :, g].T for b in range(batch)
                                                                     for g in range(G)]), bidx,
                                            D=np.array([D[h] for b, h, q in rows]),
                                            delta_bias=np.array([bias[h] for b, h, q in rows]),
                                            h0=np.array([h0[b, h, q] for b, h, q in rows]))
    got = np.array([y[b, :, h, q] for b, h, q in rows])
    assert np.max(np.abs(got - y1)) <= 1e-12 * max(1.0, np.max(np.abs(y1)))
    assert np.max(np.abs(np.array([hT[b, h, q] for b, h, q in rows]) - h1)) <= 1e-12 * max(1.0, np.max(np.abs(h1)))


def test_ssd_a_zero_is_prefix_sum():
    """A = 0: H_t = Σ_{s≤t} Δ_s x_s B_s^T (numpy cumsum), y_t = H_t C_t + D x_t."""
    x, dt, A, B, C, D, bias, _ = _ssd_inputs(33, a_zero=True)
    batch, L, nheads, P = x.shape
    G = B.shape[2]
    y, hT = oracle.ssd_scan(x, dt, A, B, C, D=D, dt_bias=bias)
    for b in range(batch):
        for h in range(nheads):
            g = h // (nheads // G)
            dl = np.logaddexp(0.0, dt[b, :, h] + bias[h])
            terms = dl[:, None, None] * x[b, :, h][:, :, None] * B[b, :, g][:, None, :]    # (L, P, N)
            Hs = np.cumsum(terms, axis=0)
            ref = np.einsum("tpn,tn->tp", Hs, C[b, :, g]) + D[h] * x[b, :, h]
            assert np.max(np.abs(y[b, :, h] - ref)) <= 1e-11 * max(1.0, np.max(np.abs(ref)))
            assert np.max(np.abs(hT[b, h] - Hs[-1])) <= 1e-11 * max(1.0, np.max(np.abs(Hs[-1])))


@pytest.mark.parametrize("chunk", [1, 3, 16, 29, 64])
def test_ssd_chunked_equals_sequential(chunk):
    x, dt, A, B, C, D, bias, h0 = _ssd_inputs(34)
    y1, h1 = oracle.ssd_scan(x, dt, A, B, C, D=D, dt_bias=bias, h0=h0)
    y2, h2 = oracle.ssd_scan(x, dt, A, B, C, D=D, dt_bias=bias, h0=h0, chunk=chunk)
    assert np.max(np.abs(y1 - y2)) <= 1e-11 * max(1.0, np.max(np.abs(y1)))
    assert np.max(np.abs(h1 - h2)) <= 1e-11 * max(1.0, np.max(np.abs(h1)))


# ---------------------------------------------------------------- the pins catch planted mistakes

_MUTATIONS = {
    "drop_D": ("if (p->D) y += p->D[c] * x;", ""),
    "exp_sign": ("*abar = exp(delta * a);", "*abar = exp(-delta * a);"),
    "read_before_update": ("    step(p, c, t, h);\n    p->y[c * p->L + t] = readout(p, c, t, h);",
                           "    p->y[c * p->L + t] = readout(p, c, t, h);\n    step(p, c, t, h);"),
    "B_for_C": ("const double* Cb = p->C + p->bidx[c]", "const double* Cb = p->B + p->bidx[c]"),
    "gate_before_skip": ("  if (p->D) y += p->D[c] * x;\n  if (p->z) y *= silu(p->z[c * p->L + t]);",
                         "  if (p->z) y *= silu(p->z[c * p->L + t]);\n  if (p->D) y += p->D[c] * x;"),
    "softplus_sign": ("return v > 0.0 ? v + log1p(exp(-v)) : log1p(exp(v));",
                      "return v > 0.0 ? v + log1p(exp(v)) : log1p(exp(v));"),
    "conv_tap_order": ("s += w[c * K + k] * xpad[t + k];", "s += w[c * K + (K - 1 - k)] * xpad[t + k];"),
    "compose_order": ("*b_out = a2 * b1 + b2;", "*b_out = a1 * b2 + b1;"),
    "ssd_decay_index": ("if (j < i) decay *= a[j + 1];", "if (j < i) decay *= a[j];"),
    "ssd_group_index": ("const int g = h / (p->nheads / p->ngroups);", "const int g = h % p->ngroups;"),
    "ssd_drop_D": ("y[i] = s + (p->D ? p->D[h] * x[i] : 0.0);", "y[i] = s;"),
    "ssd_state_decay": ("H[i * N + n] = a * H[i * N + n] + dl * x[i] * Bt[n];",
                        "H[i * N + n] = H[i * N + n] + dl * x[i] * Bt[n];"),
}

_PIN_TESTS = [test_compose_worked_example, test_zoh_epsilon_worked_example, test_a_zero_is_delta_weighted_prefix_sum,
              test_semiseparable_bruteforce_general_A, test_lti_reduces_to_convolution, test_zero_input_and_zero_gate,
              test_softplus_and_silu_identities, test_update_before_read_and_gate_after_skip,
              test_causal_conv_matches_numpy_convolve, test_decode_window_orientation,
              test_prefill_then_decode_equals_longer_prefill, test_ssd_matches_semiseparable_bruteforce,
              test_ssd_reduces_to_mamba1_channels, test_ssd_a_zero_is_prefix_sum]


@pytest.mark.parametrize("name", sorted(_MUTATIONS))
def test_planted_mistakes_are_caught(name, monkeypatch):
    old, new = _MUTATIONS[name]
    src = open(oracle._SRC).read()
    assert old in src, f"mutation anchor for {name} not found"
    tmp = tempfile.mkdtemp()
    try:
        mutated = os.path.join(tmp, "ssm_oracle.c")
        open(mutated, "w").write(src.replace(old, new))
        so = os.path.join(tmp, "libssm_oracle.so")
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-D_POSIX_C_SOURCE=200809L", "-fPIC", "-shared", "-pthread",
                               "-o", so, mutated, "-lm"])
        monkeypatch.setattr(oracle, "_SRC", mutated)
        monkeypatch.setattr(oracle, "_LIB_PATH", so)
        monkeypatch.setattr(oracle, "_lib", None)
        caught = 0
        for t in _PIN_TESTS:
            try:
                t()
            except AssertionError:
                caught += 1
        assert caught > 0, f"no pin caught the planted mistake {name}"
    finally:
        monkeypatch.setattr(oracle, "_lib", None)
        shutil.rmtree(tmp, ignore_errors=True)
