"""The seeded input generators: shapes, dtypes, determinism and recipes."""

import math

import numpy as np

from complex_valued_state_gb300 import workloads as wl


def test_shapes_dtypes_and_determinism():
    w = wl.TINY
    a, b = wl.make_inputs(w), wl.make_inputs(w)
    assert a["x"].shape == (1, 256, 1, 16) and a["x"].dtype == np.complex64
    assert a["B"].shape == a["C"].shape == (1, 256, 1, 16) and a["B"].dtype == np.complex64
    assert a["dt"].shape == (1, 256, 1) and a["dt"].dtype == np.float32
    assert a["A"].shape == (1,) and a["A"].dtype == np.complex64
    assert a["D"].shape == (1,) and a["D"].dtype == np.float32
    for k in a:
        assert np.array_equal(a[k], b[k])
    c = wl.make_inputs(w, seed=123)
    assert not np.array_equal(a["x"], c["x"])


def test_distribution_moments():
    d = wl.make_inputs(wl.MAMBA2_LAYER.with_(seqlen=256))
    N = wl.MAMBA2_LAYER.dstate
    assert abs(np.mean(np.abs(d["x"]) ** 2) - 1.0) < 0.02
    assert abs(np.mean(np.abs(d["B"]) ** 2) * N - 1.0) < 0.02
    assert abs(np.mean(d["dt"]) + 1.0) < 0.01 and abs(np.std(d["dt"]) - 0.5) < 0.01
    assert np.all(d["A"].real <= -0.5 + 1e-6) and np.all(d["A"].real >= -4.0 - 1e-6)
    assert np.all(np.abs(d["A"].imag) <= math.pi + 1e-6)


def test_slow_decay_rates():
    w = wl.LONG_SEQ.with_(seqlen=512)
    d = wl.make_inputs(w)
    rho_mean_dt = np.exp(math.log1p(math.exp(-1.0)) * d["A"].real.astype(np.float64))
    assert np.all(rho_mean_dt >= 0.9 - 1e-6) and np.all(rho_mean_dt <= 0.9999 + 1e-6)


def test_pam_mapping():
    w = wl.PAM.with_(seqlen=16, batch=2)
    d = wl.make_inputs(w)
    assert np.allclose(np.abs(d["Q"]), 1, atol=1e-6) and np.allclose(np.abs(d["K"]), 1, atol=1e-6)
    assert np.array_equal(d["B"], np.conj(d["K"]).astype(np.complex64))
    assert np.allclose(d["C"], d["Q"] / math.sqrt(w.dstate), atol=1e-7)
    assert np.array_equal(d["x"], d["V"]) and np.all(d["D"] == 0)
    sp = np.log1p(np.exp(d["dt"].astype(np.float64)))
    assert np.allclose(sp, 1.0, atol=1e-6)
    assert np.allclose(np.exp(d["A"].real.astype(np.float64)), d["gamma"], rtol=1e-6)


def test_decode_tokens_are_independent_per_step():
    w = wl.DECODE.with_(batch=4, nheads=2)
    t3a, t3b, t4 = wl.decode_token(w, 3), wl.decode_token(w, 3), wl.decode_token(w, 4)
    assert np.array_equal(t3a["x"], t3b["x"]) and not np.array_equal(t3a["x"], t4["x"])
    f = wl.decode_fixed(w)
    assert f["h"].shape == (4, 2, 128, 64) and f["h"].dtype == np.complex64
