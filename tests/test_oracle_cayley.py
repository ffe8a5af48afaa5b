"""Pins of the oracle for the per-coordinate Cayley-phase recurrence
("Complex Phase-State Dynamics Reduce the Optimization Steps of Sequence
Models", sections 5.2-5.5, Appendix A Algorithms 1-2) against results fixed
independently of the oracle's code: the identities the paper states for the
Cayley phase, brute-force unrolled sums, and closed forms of the clamped scan.
"""

import math

import numpy as np
import pytest

from complex_valued_state_gb300 import workloads as wl


@pytest.fixture(scope="module")
def orc():
    import oracle

    oracle.build()
    return oracle


def small(seed=0, Bz=2, T=150, H=2, N=3, gate_mean=0.0):
    w = wl.HMAMBA_SCAN.with_(batch=Bz, seqlen=T, nheads=H, dstate=N, headdim=N)
    return wl.make_cayley_inputs(w, seed=seed, gate_mean=gate_mean)


def test_algorithm1_identities(orc):
    """|lambda| = 1 and arg lambda = 2 arctan phi; |a| = sigmoid(u) at values
    with exact sigmoids; special phases lambda(0) = 1, lambda(1) = i,
    lambda(-1) = -i."""
    theta = np.linspace(-3.1, 3.1, 41)
    phi = np.tan(theta / 2)  # so that 2 arctan(phi) = theta
    a = orc.cayley_coefficients(phi, np.full_like(phi, 60.0))  # gate = 1 to double precision
    assert np.allclose(np.abs(a), 1.0, atol=1e-15, rtol=0)
    assert np.allclose(np.angle(a), theta, atol=1e-13, rtol=0)
    # sigmoid(0) = 1/2, sigmoid(ln 3) = 3/4, sigmoid(-ln 3) = 1/4
    u = np.array([0.0, math.log(3.0), -math.log(3.0)])
    a = orc.cayley_coefficients(np.zeros(3), u)
    assert np.allclose(a, [0.5, 0.75, 0.25], atol=1e-15, rtol=0)
    a = orc.cayley_coefficients(np.array([0.0, 1.0, -1.0]), np.full(3, 60.0))
    assert np.allclose(a, [1.0, 1j, -1j], atol=1e-15, rtol=0)


def test_recurrence_against_unrolled_sum(orc):
    """psi_t = (prod_{r<=t} a_r) psi0 + sum_{s<=t} (prod_{s<r<=t} a_r) b_s, read
    out as conj(C_t) psi_t, written out term by term on a tiny case."""
    d = small(seed=3, Bz=1, T=6, H=1, N=2)
    a = orc.cayley_coefficients(d["phi"], d["u"])[0, :, 0, :]  # [T, N]
    b = d["b"][0, :, 0, :].astype(np.complex128)
    C = d["C"][0, :, 0, :].astype(np.complex128)
    p0 = d["psi0"][0, 0].astype(np.complex128)
    y, pf = orc.cayley_recurrence(d["phi"], d["u"], d["b"], d["C"], psi0=d["psi0"])
    for t in range(6):
        psi = np.prod(a[: t + 1], axis=0) * p0
        for s in range(t + 1):
            psi = psi + np.prod(a[s + 1 : t + 1], axis=0) * b[s]
        assert np.allclose(y[0, t, 0], np.conj(C[t]) * psi, rtol=1e-13, atol=1e-14)
    assert np.allclose(pf[0, 0], psi, rtol=1e-13, atol=1e-14)


def test_readout_conjugates_C(orc):
    d = small(seed=4, Bz=1, T=9, H=1, N=4)
    C = np.full_like(d["C"], 1j)
    y, pf = orc.cayley_recurrence(d["phi"], d["u"], d["b"], C, psi0=d["psi0"])
    assert np.allclose(y[0, -1, 0], -1j * pf[0, 0], rtol=1e-14, atol=0)  # conj(i) psi


@pytest.mark.parametrize("chunk", [1, 3, 64])
def test_unclamped_scan_equals_recurrence(orc, chunk):
    """Algorithm 2 without the clamp is exact (up to rounding) for any chunk,
    including a ragged last chunk and strongly decaying gates."""
    d = small(seed=5, T=150, gate_mean=0.0)
    yr, pr = orc.cayley_recurrence(d["phi"], d["u"], d["b"], d["C"], psi0=d["psi0"])
    yc, pc = orc.cayley_chunked(d["phi"], d["u"], d["b"], d["C"], chunk, -math.inf, psi0=d["psi0"])
    scale = np.max(np.abs(yr))
    assert np.max(np.abs(yc - yr)) < 1e-12 * scale
    assert np.max(np.abs(pc - pr)) < 1e-12 * np.max(np.abs(pr))


def test_clamped_scan_is_exact_while_the_clamp_is_inactive(orc):
    d = small(seed=6, T=200, gate_mean=4.0)  # gates near 0.98: a chunk's log-gate sum stays far above -30
    yr, pr = orc.cayley_recurrence(d["phi"], d["u"], d["b"], d["C"], psi0=d["psi0"])
    yc, pc = orc.cayley_chunked(d["phi"], d["u"], d["b"], d["C"], 64, -30.0, psi0=d["psi0"])
    assert np.max(np.abs(yc - yr)) < 1e-12 * np.max(np.abs(yr))


def test_clamp_closed_form(orc):
    """Constant gate e^-1, no phase, b = 1, chunk 64, clamp -30: within a chunk
    the cumulative log-gate is -m, clamped at -30 from m = 30 on, so
        m <= 30: psi_m = e^-m x0 + (1 - e^-m) / (1 - e^-1)
        m >  30: psi_m = e^-30 x0 + (e - e^-29) / (e - 1) + (m - 30),
    x0 being the previous chunk's last state.  The exact recurrence instead
    tends to 1 / (1 - e^-1): the clamp changes the result once it is active."""
    T, ch = 128, 64
    g = math.exp(-1.0)
    u = np.full((1, T, 1, 1), math.log(g / (1.0 - g)))
    phi = np.zeros((1, T, 1, 1))
    one = np.ones((1, T, 1, 1), np.complex128)
    y, pf = orc.cayley_chunked(phi, u, one, one, ch, -30.0)
    e = math.e
    want, x0 = [], 0.0
    for c in range(T // ch):
        for m in range(1, ch + 1):
            if m <= 30:
                v = math.exp(-m) * x0 + (1 - math.exp(-m)) / (1 - math.exp(-1))
            else:
                v = math.exp(-30) * x0 + (e - math.exp(-29)) / (e - 1) + (m - 30)
            want.append(v)
        x0 = want[-1]
    assert np.allclose(y[0, :, 0, 0], want, rtol=1e-12, atol=0)
    assert abs(pf[0, 0, 0] - want[-1]) < 1e-12 * want[-1]
    exact, _ = orc.cayley_recurrence(phi, u, one, one)
    assert abs(exact[0, 63, 0, 0] - 1 / (1 - g)) < 1e-12
    assert y[0, 63, 0, 0].real > 30  # clamped: 34 undecayed inputs on top


def test_phase_transport(orc):
    """Impulse at t = 0 with unit gates: the modulus is carried exactly and the
    argument advances by sum_t 2 arctan(phi_t) (the paper's Lemma 6.2 for this
    recurrence); with gates alpha_t the modulus is |b_0| prod alpha_t."""
    rng = np.random.default_rng(11)
    T = 300
    phi = rng.normal(0.0, 0.7, size=(1, T, 1, 1))
    b = np.zeros((1, T, 1, 1), np.complex128)
    b[0, 0, 0, 0] = 0.6 - 0.8j
    one = np.ones_like(b)
    for lo in (-math.inf, -30.0):
        _, pf = orc.cayley_chunked(phi, np.full(phi.shape, 60.0), b, one, 64, lo)
        assert abs(abs(pf[0, 0, 0]) - 1.0) < 1e-12
        # the impulse enters at t = 0 after that token's update; later tokens rotate it
        turn = np.angle(0.6 - 0.8j) + np.sum(2 * np.arctan(phi[0, 1:, 0, 0]))
        assert abs(np.angle(pf[0, 0, 0] * np.exp(-1j * turn))) < 1e-10
    u = rng.normal(3.0, 0.5, size=(1, T, 1, 1))
    _, pf = orc.cayley_recurrence(phi, u, b, one)
    assert abs(abs(pf[0, 0, 0]) - np.prod(1 / (1 + np.exp(-u[0, 1:, 0, 0])))) < 1e-12
