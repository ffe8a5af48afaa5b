"""Pins for the CPU oracle: each check ties it to something other than itself.

* closed-form unrolled sum (brute force over all source tokens), on tiny inputs;
* the chunkwise identity, with time-varying dt and ragged lengths;
* A = 0 reduces the recurrence to a prefix sum;
* the decay gains the pages print (0.99^1024, 0.999^1024);
* discretisation order: softplus(0) = ln 2, so a = 2^A exactly;
* Lemma 6.2 of the phase-state paper: phases add, magnitudes multiply;
* the constant-input geometric series over 4096 steps;
* the phase-associative-memory sum (its eq. 7) and its lossless retrieval with
  orthogonal keys;
* state hand-off: T tokens then k single steps equals T + k tokens.
"""

import math
import os

import numpy as np
import pytest

from complex_valued_state_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rel_err(a, b):
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


def _softplus(v):
    v = np.asarray(v, dtype=np.float64)
    return np.maximum(v, 0) + np.log1p(np.exp(-np.abs(v)))


def brute_force(x, dt, A, B, C, D):
    """y_t = sum_{s<=t} C_t^T (prod_{u=s+1..t} a_u) B_s x_s^T + D x_t, zero start.

    The product of per-step factors is formed by explicit multiplication, not
    by an exponential of a sum.
    """
    x, B, C = (np.asarray(v, np.complex128) for v in (x, B, C))
    Bz, T, H, P = x.shape
    a = np.exp(_softplus(dt) * np.asarray(A, np.complex128)[None, None, :])  # [Bz,T,H]
    y = np.zeros((Bz, T, H, P), np.complex128)
    for b in range(Bz):
        for h in range(H):
            for t in range(T):
                acc = np.zeros(P, np.complex128)
                for s in range(t + 1):
                    prod = 1.0 + 0j
                    for u in range(s + 1, t + 1):
                        prod *= a[b, u, h]
                    acc += prod * (C[b, t, h] @ B[b, s, h]) * x[b, s, h]
                y[b, t, h] = acc + D[h] * x[b, t, h]
    return y


@pytest.mark.parametrize("shape", [(1, 1, 1, 2, 3), (2, 5, 2, 3, 2), (1, 12, 3, 4, 4)])
def test_naive_equals_unrolled_sum(oracle_lib, shape):
    Bz, T, H, N, P = shape
    d = wl.random_case(100 + T, Bz, T, H, N, P, dt_std=1.0)
    y, _ = oracle_lib.cssd_naive(**d)
    ref = brute_force(**d)
    assert rel_err(y, ref) < 1e-12


def test_bruteforce_detects_conjugation_and_order(oracle_lib):
    # The pin must be able to fail: a conjugated B or a readout before the
    # update each move the result far outside the tolerance.
    d = wl.random_case(7, 1, 6, 2, 3, 2, dt_std=1.0)
    ref = brute_force(**d)
    conj = dict(d, B=np.conj(d["B"]))
    assert rel_err(oracle_lib.cssd_naive(**conj)[0], ref) > 1e-2
    # readout before the update == the result shifted by one token
    y, _ = oracle_lib.cssd_naive(**d)
    assert rel_err(y[:, 1:] - d["D"][None, None, :, None] * d["x"][:, 1:], ref[:, 1:]) > 1e-2


CHUNK_CASES = [(c, t) for c in (1, 3, 4, 64) for t in sorted({1, max(c - 1, 1), c, c + 1, 19, 70})]


@pytest.mark.parametrize("chunk,T", CHUNK_CASES)
def test_chunked_equals_naive(oracle_lib, chunk, T):
    d = wl.random_case(1000 + 7 * chunk + T, 2, T, 2, 3, 4, dt_std=1.0)
    y, hf = oracle_lib.cssd_naive(**d)
    yc, hc = oracle_lib.cssd_chunked(**d, chunk=chunk)
    assert yc.shape == y.shape
    assert rel_err(yc, y) < 1e-12
    assert rel_err(hc, hf) < 1e-12


def _chunked_numpy(x, dt, A, B, C, D, chunk, misaligned=False):
    """Compact chunkwise form used only to show the test inputs discriminate.

    With misaligned=True the carry-in decay uses exp(CD[z] - CD[c]) against the
    list shifted by one chunk, the propagation that the chunkwise page's
    Pitfalls section reports as wrong whenever chunk totals differ.
    """
    x, B, C = (np.asarray(v, np.complex128) for v in (x, B, C))
    Bz, T, H, P = x.shape
    N = B.shape[-1]
    pad = (chunk - T % chunk) % chunk
    nc = (T + pad) // chunk
    alog = _softplus(dt) * np.asarray(A, np.complex128)[None, None, :]
    padT = lambda v: np.concatenate([v, np.zeros((Bz, pad) + v.shape[2:], v.dtype)], axis=1)
    X, Bp, Cp, Al = padT(x), padT(B), padT(C), padT(alog)
    X = X.reshape(Bz, nc, chunk, H, P)
    Bp = Bp.reshape(Bz, nc, chunk, H, N)
    Cp = Cp.reshape(Bz, nc, chunk, H, N)
    Acs = np.cumsum(Al.reshape(Bz, nc, chunk, H), axis=2)
    seg = Acs[:, :, :, None, :] - Acs[:, :, None, :, :]  # b c l s h
    mask = np.tril(np.ones((chunk, chunk), bool))[None, None, :, :, None]
    L = np.where(mask, np.exp(np.where(mask, seg, 0)), 0)
    ydiag = np.einsum("bclhn,bcshn,bclsh,bcshp->bclhp", Cp, Bp, L, X)
    ds = np.exp(Acs[:, :, -1:, :] - Acs)
    S = np.einsum("bclhn,bclh,bclhp->bchnp", Bp, ds, X)
    ct = Acs[:, :, -1, :]  # b c h
    CD = np.cumsum(ct, axis=1)
    Hin = np.zeros((Bz, nc, H, N, P), np.complex128)
    for z in range(nc):
        for c in range(nc):
            if misaligned:
                # decay exp(CD[z] - CD[c]) applied to the shifted list [0, S_0, S_1, ...]
                if c <= z and c >= 1:
                    Hin[:, z] += np.exp(CD[:, z] - CD[:, c])[..., None, None] * S[:, c - 1]
            elif c < z:
                Hin[:, z] += np.exp(CD[:, z - 1] - CD[:, c])[..., None, None] * S[:, c]
    yoff = np.einsum("bclhn,bchnp,bclh->bclhp", Cp, Hin, np.exp(Acs))
    y = (ydiag + yoff).reshape(Bz, nc * chunk, H, P)[:, :T]
    return y + np.asarray(D)[None, None, :, None] * x


def test_chunk_inputs_discriminate_misaligned_propagation(oracle_lib):
    d = wl.random_case(4242, 1, 16, 2, 4, 4, dt_std=1.0)
    y, _ = oracle_lib.cssd_naive(**d)
    assert rel_err(_chunked_numpy(**d, chunk=4), y) < 1e-12
    assert rel_err(_chunked_numpy(**d, chunk=4, misaligned=True), y) > 1e-2
    # the same misalignment is invisible when every chunk total is equal (dt constant)
    d0 = dict(d, dt=np.zeros_like(d["dt"]))
    y0, _ = oracle_lib.cssd_naive(**d0)
    assert rel_err(_chunked_numpy(**d0, chunk=4, misaligned=True), y0) < 1e-12


def test_zero_rate_is_prefix_sum(oracle_lib):
    d = wl.random_case(5, 2, 33, 3, 5, 4, a_scale=0.0)
    y, hf = oracle_lib.cssd_naive(**d)
    outer = np.einsum("bthn,bthp->bthnp", d["B"].astype(np.complex128), d["x"].astype(np.complex128))
    hs = np.cumsum(outer, axis=1)
    ref = np.einsum("bthn,bthnp->bthp", d["C"].astype(np.complex128), hs) + d["D"][None, None, :, None] * d["x"].astype(np.complex128)
    assert rel_err(y, ref) < 1e-12
    assert rel_err(hf, hs[:, -1]) < 1e-12


def _impulse(T, A, dt_value, H=1):
    """Unit impulse at t = 0 with constant readout; N = P = 1."""
    x = np.zeros((1, T, H, 1), np.complex128)
    x[:, 0] = 1.0
    B = np.ones((1, T, H, 1), np.complex128)
    C = np.ones((1, T, H, 1), np.complex128)
    dt = np.full((1, T, H), dt_value, np.float64)
    return dict(x=x, dt=dt, A=np.asarray(A, np.complex128), B=B, C=C, D=np.zeros(H))


def test_printed_decay_gains(oracle_lib):
    rows = [l.split(maxsplit=4) for l in open(os.path.join(GOLDEN, "decay_facts.txt")) if not l.startswith("#")]
    assert len(rows) == 2
    dt_unit = math.log(math.e - 1.0)  # softplus(dt_unit) = 1
    for rho, T, gain, tol, _cite in rows:
        rho, T, gain, tol = float(rho), int(T), float(gain), float(tol)
        y, _ = oracle_lib.cssd_naive(**_impulse(T + 1, [math.log(rho)], dt_unit))
        ratio = abs(y[0, T, 0, 0]) / abs(y[0, 0, 0, 0])
        assert abs(ratio - gain) <= tol, (rho, ratio, gain)


def test_discretisation_order(oracle_lib):
    # dt = 0: softplus(0) = ln 2, so the per-step factor is 2^A (not exp(softplus(0 * A)) = 2).
    A = np.array([-1.0 + 0.5j])
    y, _ = oracle_lib.cssd_naive(**_impulse(3, A, 0.0))
    expect = 2.0 ** A[0]
    assert abs(y[0, 1, 0, 0] / y[0, 0, 0, 0] - expect) < 1e-14
    assert abs(y[0, 2, 0, 0] / y[0, 0, 0, 0] - expect**2) < 1e-14


def test_phase_transport_lemma(oracle_lib):
    # Two heads j, k from an impulse: arg(y_j conj y_k) advances by the summed phase
    # differences and |y_j conj y_k| shrinks by the product of both magnitudes.
    T = 200
    rng = np.random.default_rng(11)
    A = np.array([-0.02 + 1.3j, -0.05 - 0.4j])
    d = _impulse(T, A, 0.0, H=2)
    d["dt"] = rng.normal(-1.0, 0.8, size=(1, T, 2))
    d["B"][:, 0, :, 0] = np.array([0.7 + 0.2j, -0.3 + 0.9j])
    y, _ = oracle_lib.cssd_naive(**d)
    rho = y[0, :, 0, 0] * np.conj(y[0, :, 1, 0])
    sp = _softplus(d["dt"][0])  # [T, 2]
    dphase = np.sum(sp[1:, 0] * A[0].imag - sp[1:, 1] * A[1].imag)
    want_arg = np.angle(rho[0]) + dphase
    got_arg = np.angle(rho[-1])
    assert abs(np.angle(np.exp(1j * (got_arg - want_arg)))) < 1e-10
    want_mag = abs(rho[0]) * np.exp(np.sum(sp[1:, 0] * A[0].real + sp[1:, 1] * A[1].real))
    assert abs(abs(rho[-1]) / want_mag - 1) < 1e-10


def test_geometric_series_4096_steps(oracle_lib):
    Bz, H, N, P, n = 2, 3, 4, 3, 4096
    d = wl.random_case(77, Bz, 1, H, N, P)
    rng = np.random.default_rng(78)
    h0 = (rng.standard_normal((Bz, H, N, P)) + 1j * rng.standard_normal((Bz, H, N, P))) / math.sqrt(2)
    tok = {k: d[k][:, 0] for k in ("x", "B", "C", "dt")}
    rep = {k: np.repeat(d[k], n, axis=1) for k in ("x", "B", "C", "dt")}
    y, hf = oracle_lib.cssd_naive(rep["x"], rep["dt"], d["A"], rep["B"], rep["C"], d["D"], h0=h0)
    hn, yn, yinf = oracle_lib.geom_closed_form(h0, tok["x"], tok["dt"], d["A"], tok["B"], tok["C"], d["D"], n)
    assert rel_err(hn, hf) < 1e-10
    assert rel_err(yn, y[:, -1]) < 1e-10
    # decaying heads converge to the fixed point, whatever the start
    assert rel_err(yinf, yn) < 1e-8
    # n = 1 is one ordinary step
    h1, y1 = oracle_lib.cssd_step(h0, tok["x"], tok["dt"], d["A"], tok["B"], tok["C"], d["D"])
    hn1, yn1, _ = oracle_lib.geom_closed_form(h0, tok["x"], tok["dt"], d["A"], tok["B"], tok["C"], d["D"], 1)
    assert rel_err(hn1, h1) < 1e-13 and rel_err(yn1, y1) < 1e-13


def test_pam_sum_equals_mapped_recurrence(oracle_lib):
    w = wl.PAM.with_(batch=1, seqlen=24, nheads=2, dstate=4, headdim=4)
    d = wl.make_inputs(w)
    y, _ = oracle_lib.cssd_naive(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"])
    Q, K, V = (d[k].astype(np.complex128) for k in ("Q", "K", "V"))
    gamma, dd = d["gamma"], w.dstate
    T, H = w.seqlen, w.nheads
    ref = np.zeros_like(y)
    for h in range(H):
        for t in range(T):
            for i in range(t + 1):
                decay = gamma[h] ** (t - i)
                ref[0, t, h] += decay * np.sum(np.conj(K[0, i, h]) * Q[0, t, h] / math.sqrt(dd)) * V[0, i, h]
    # float32 storage of ln(gamma) and dt = ln(e - 1) perturbs the decay by ~1e-7 per step
    assert rel_err(y, ref) < 1e-4
    assert rel_err(y.real, ref.real) < 1e-4


def test_pam_orthogonal_keys_retrieve_exactly(oracle_lib):
    d = 8
    n = np.arange(d)
    K = np.exp(2j * np.pi * np.outer(n, n) / d)  # rows: mutually orthogonal unit-modulus keys
    rng = np.random.default_rng(3)
    V = np.exp(1j * rng.uniform(-np.pi, np.pi, size=(d, d)))
    for j in (0, 3, 7):
        T = d + 1
        x = np.zeros((1, T, 1, d), np.complex128)
        B = np.zeros((1, T, 1, d), np.complex128)
        C = np.zeros((1, T, 1, d), np.complex128)
        x[0, :d, 0] = V
        B[0, :d, 0] = np.conj(K)
        C[0, d, 0] = K[j] / d  # K_j^* . Q~ = 1, K_i^* . Q~ = 0 for i != j
        y, _ = oracle_lib.cssd_naive(x, np.zeros((1, T, 1)), np.zeros(1, np.complex128), B, C, np.zeros(1))
        assert np.max(np.abs(y[0, d, 0] - V[j])) < 1e-12


def test_state_handoff_equals_longer_sequence(oracle_lib):
    Bz, T, k, H, N, P = 2, 9, 4, 2, 3, 2
    d = wl.random_case(31, Bz, T + k, H, N, P)
    y_all, h_all = oracle_lib.cssd_naive(**d)
    head = {kk: (v[:, :T] if kk in ("x", "dt", "B", "C") else v) for kk, v in d.items()}
    _, h = oracle_lib.cssd_naive(**head)
    for t in range(T, T + k):
        h, yt = oracle_lib.cssd_step(h, d["x"][:, t], d["dt"][:, t], d["A"], d["B"][:, t], d["C"][:, t], d["D"])
        assert rel_err(yt, y_all[:, t]) < 1e-12
    assert rel_err(h, h_all) < 1e-12
    # and the initial-state argument of the sequential form continues the same way
    tail = {kk: (v[:, T:] if kk in ("x", "dt", "B", "C") else v) for kk, v in d.items()}
    _, h_tail = oracle_lib.cssd_naive(**head)
    y2, h2 = oracle_lib.cssd_naive(**tail, h0=h_tail)
    assert rel_err(y2, y_all[:, T:]) < 1e-12 and rel_err(h2, h_all) < 1e-12


@pytest.mark.parametrize("T,C", [(1, 64), (63, 64), (64, 64), (65, 64), (2048, 64), (65536, 128), (20, 4), (5, 128)])
def test_chunk_bookkeeping(T, C):
    pad = (C - T % C) % C
    nc = (T + pad) // C
    assert nc == -(-T // C) and 0 <= pad < C and nc * C == T + pad
