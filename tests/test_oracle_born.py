"""Pins of the causal Born attention oracle (Algorithm 3 of the phase-state
paper), each against something fixed independently of the oracle's code:
the recurrent feature-map form, closed forms, invariances the definition
implies, and the two-state interference example the pages print."""

import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "born_two_state.txt")


def cgauss(rng, shape):
    return (rng.standard_normal(shape) + 1j * rng.standard_normal(shape)) / math.sqrt(2.0)


def case(seed, Bz=2, T=23, H=3, D=4):
    rng = np.random.default_rng(seed)
    q, k, v = cgauss(rng, (Bz, T, H, D)), cgauss(rng, (Bz, T, H, D)), cgauss(rng, (Bz, T, H, D))
    tau = rng.uniform(0.5, 2.0, (Bz, T, H))
    return q, k, v, tau


def rel(a, b):
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


@pytest.fixture(scope="module")
def orc():
    oracle.build()
    return oracle


@pytest.mark.parametrize("D,T", [(1, 9), (3, 31), (4, 23), (8, 40)])
def test_direct_form_equals_feature_map_form(orc, D, T):
    """|<q|k>|^2 = q^H (k k^H) q: the per-position D x D recurrence gives the
    same psi as the quadratic sum over earlier positions."""
    q, k, v, tau = case(D * 100 + T, T=T, D=D)
    assert rel(orc.born_attention(q, k, v, tau), orc.born_attention_feature_map(q, k, v)) < 1e-12


def test_feature_map_form_catches_a_missing_conjugate(orc):
    """The score without the bra's conjugate, sum_a q_a k_a, is a different
    quantity; the feature-map form tells the two apart."""
    q, k, v, tau = case(7, Bz=1, T=12, H=1, D=3)
    g = np.einsum("tha,sha->hts", q[0], k[0])  # no conjugate: the planted mistake
    s = np.abs(g) ** 2 * np.tril(np.ones((12, 12)))[None]
    wrong = np.einsum("hts,shm->thm", s, v[0]) / s.sum(-1).T[..., None]
    ref = orc.born_attention_feature_map(q, k, v)[0]
    assert rel(wrong, ref) > 1e-3
    assert rel(orc.born_attention(q, k, v, tau)[0], ref) < 1e-12


def test_temperature_and_width_cancel(orc):
    """s_ij carries 1/(D tau_i) in numerator and denominator alike."""
    q, k, v, tau = case(3)
    tau2 = np.random.default_rng(4).uniform(0.01, 100.0, tau.shape)
    assert rel(orc.born_attention(q, k, v, tau), orc.born_attention(q, k, v, tau2)) < 1e-13


def test_first_position_returns_its_value(orc):
    q, k, v, tau = case(5)
    psi = orc.born_attention(q, k, v, tau)
    assert np.max(np.abs(psi[:, 0] - v[:, 0])) < 1e-13


def test_equal_keys_give_the_running_mean(orc):
    """Every key equal: each row's scores are constant, so psi_i is the mean
    of v_0 .. v_i."""
    q, k, v, tau = case(6, T=17)
    k[:] = k[:, :1]
    psi = orc.born_attention(q, k, v, tau)
    mean = np.cumsum(v, axis=1) / np.arange(1, 18)[None, :, None, None]
    assert rel(psi, mean) < 1e-12


def test_causality(orc):
    q, k, v, tau = case(8, T=30)
    psi = orc.born_attention(q, k, v, tau)
    k2, v2 = k.copy(), v.copy()
    k2[:, 19:] += 1.0 + 2.0j
    v2[:, 19:] -= 3.0
    psi2 = orc.born_attention(q, k2, v2, tau)
    assert np.array_equal(psi[:, :19], psi2[:, :19])
    assert not np.allclose(psi[:, 19:], psi2[:, 19:])


def test_phase_invariance(orc):
    """A unit phase on a query or on a key leaves every squared modulus, and so
    psi, unchanged."""
    q, k, v, tau = case(9)
    rng = np.random.default_rng(10)
    a = np.exp(1j * rng.uniform(-math.pi, math.pi, q.shape[:3]))[..., None]
    b = np.exp(1j * rng.uniform(-math.pi, math.pi, k.shape[:3]))[..., None]
    assert rel(orc.born_attention(q * a, k * b, v, tau), orc.born_attention(q, k, v, tau)) < 1e-12


def test_orthogonal_query_gives_zero(orc):
    """A query orthogonal to every key so far has all-zero scores; the reading
    returns psi = 0 there."""
    D, T = 2, 3
    q = np.zeros((1, T, 1, D), complex)
    k = np.zeros((1, T, 1, D), complex)
    v = np.ones((1, T, 1, D), complex)
    k[0, :, 0, 0] = 1.0  # every key along |phi1>
    q[0, :, 0, 1] = 1.0  # every query along |phi2>
    psi = orc.born_attention(q, k, v, np.ones((1, T, 1)))
    assert np.array_equal(psi, np.zeros_like(psi))


def test_two_state_interference_as_printed(orc):
    """The pages' two-state computation as an attention: position 0 holds the
    key |psi(theta)> with value (1, 0), position 1 the key |e> with value
    (0, 1) and the query |e>.  Then psi_1 = (p, 1) / (p + 1), so
    p = psi_1[0] / psi_1[1] must equal (1 + cos theta) / 2, and the printed
    endpoints 1 (theta = 0) and 0 (theta = pi)."""
    rows = [l.split() for l in open(GOLDEN) if l.strip() and not l.startswith("#")]
    checks = [(float(r[0]), float(r[1])) for r in rows] + [(t, None) for t in (0.3, 1.1, 2.0, 2.9, -1.7)]
    for theta, printed in checks:
        s = 1.0 / math.sqrt(2.0)
        q = np.array([[[0, 0]], [[s, s]]], complex)[None]
        k = np.array([[[s, s * np.exp(1j * theta)]], [[s, s]]], complex)[None]
        v = np.array([[[1, 0]], [[0, 1]]], complex)[None]
        psi = orc.born_attention(q, k, v, np.ones((1, 2, 1)))
        p = (psi[0, 1, 0, 0] / psi[0, 1, 0, 1]).real
        assert abs(p - 0.5 * (1.0 + math.cos(theta))) < 1e-12
        if printed is not None:
            assert abs(p - printed) < 1e-12
