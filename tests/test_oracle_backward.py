"""Pins of the backward oracle (gradients of the forward recurrence) against
results fixed independently of its code: central finite differences of the
forward oracle for every input coordinate, the adjoint identity of the linear
map x -> y, and the reverse-cumulative-sum form of the step and rate
gradients (the form the GPU path uses)."""

import numpy as np
import pytest

import oracle
from complex_valued_state_gb300 import workloads as wl


@pytest.fixture(scope="module")
def orc():
    oracle.build()
    return oracle


def case(seed, Bz=1, T=7, H=2, N=3, P=2, a_scale=1.0):
    d = wl.random_case(seed, Bz, T, H, N, P, a_scale=a_scale)
    d = {k: (v.astype(np.complex128) if np.iscomplexobj(v) else v.astype(np.float64)) for k, v in d.items()}
    rng = np.random.default_rng(seed + 100)
    dy = rng.standard_normal((Bz, T, H, P)) + 1j * rng.standard_normal((Bz, T, H, P))
    return d, dy


def loss(orc, d, dy):
    y, _ = orc.cssd_naive(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"])
    return float(np.real(np.sum(np.conj(dy) * y)))


def fd_grad(orc, d, dy, name, eps=1e-6):
    """dL/dRe w + i dL/dIm w (complex w) or dL/dw (real w), central differences."""
    w = d[name]
    g = np.zeros_like(w)
    for idx in np.ndindex(w.shape):
        parts = (1.0, 1j) if np.iscomplexobj(w) else (1.0,)
        for unit in parts:
            hi = {**d, name: w.copy()}
            lo = {**d, name: w.copy()}
            hi[name][idx] += eps * unit
            lo[name][idx] -= eps * unit
            g[idx] += unit * (loss(orc, hi, dy) - loss(orc, lo, dy)) / (2 * eps)
    return g


@pytest.mark.parametrize("shape", [(1, 7, 2, 3, 2), (2, 5, 1, 2, 4)])
@pytest.mark.parametrize("name,key", [("x", "gx"), ("dt", "gdt"), ("A", "gA"), ("B", "gB"), ("C", "gC"), ("D", "gD")])
def test_gradients_match_finite_differences(orc, shape, name, key):
    Bz, T, H, N, P = shape
    d, dy = case(sum(shape), Bz, T, H, N, P)
    g = orc.cssd_backward(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], dy)
    fd = fd_grad(orc, d, dy, name)
    assert np.max(np.abs(g[key] - fd)) <= 1e-7 * max(1.0, np.max(np.abs(fd)))


def test_adjoint_identity(orc):
    """y is linear in x, and gx applies its adjoint to dy:
    sum conj(dy) y = sum x conj(gx) (complex, exact up to rounding), per (batch, head)."""
    d, dy = case(11, Bz=2, T=40, H=3, N=4, P=3)
    y, _ = orc.cssd_naive(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"])
    g = orc.cssd_backward(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], dy)
    lhs = np.sum(np.conj(dy) * y, axis=(1, 3))
    rhs = np.sum(d["x"] * np.conj(g["gx"]), axis=(1, 3))
    assert np.max(np.abs(lhs - rhs)) <= 1e-10 * np.max(np.abs(lhs))


def test_step_and_rate_gradients_as_reverse_cumulative_sums(orc):
    """With r_t = sum_p (conj(dy_t) y_t - x_t conj(gx_t)) and R_t = sum_{u >= t} r_u,
    the gradient with respect to z_t = softplus(dt_t) A is conj(R_t), so
    gdt_t = Re(R_t A) sigmoid(dt_t) and gA = sum_{b,t} softplus(dt_t) conj(R_t)."""
    d, dy = case(12, Bz=2, T=33, H=3, N=4, P=5)
    y, _ = orc.cssd_naive(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"])
    g = orc.cssd_backward(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], dy)
    r = np.sum(np.conj(dy) * y - d["x"] * np.conj(g["gx"]), axis=3)  # [Bz, T, H]
    R = np.cumsum(r[:, ::-1], axis=1)[:, ::-1]
    dt = d["dt"]
    sp = np.maximum(dt, 0) + np.log1p(np.exp(-np.abs(dt)))
    sig = 1.0 / (1.0 + np.exp(-dt))
    assert np.max(np.abs(g["gdt"] - np.real(R * d["A"][None, None, :]) * sig)) <= 1e-9 * np.max(np.abs(g["gdt"]))
    gA = np.sum(sp * np.conj(R), axis=(0, 1))
    assert np.max(np.abs(g["gA"] - gA)) <= 1e-9 * np.max(np.abs(gA))
    assert np.max(np.abs(R[:, 0])) <= 1e-9 * np.max(np.abs(R))  # the whole sum is zero


def test_zero_rate_has_no_step_gradient(orc):
    """A = 0: the per-step factor is 1 whatever dt is, so gdt = 0."""
    d, dy = case(13, a_scale=0.0)
    g = orc.cssd_backward(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], dy)
    assert np.max(np.abs(g["gdt"])) < 1e-12
