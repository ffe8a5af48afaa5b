"""GPU parity of the constant-input shortcuts (cssd_step_n, cssd_step_infinite)
against the oracle: its closed form, which the CPU tests pin to the
step-by-step loop, and the step-by-step loop itself where the closed form is
singular (a = 1).  Bar as for every output: max |got - ref| <= 2e-3 max |ref|.
"""

import numpy as np
import pytest
import torch

from complex_valued_state_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

TOL = 2e-3
TOK = ("x", "dt", "B", "C")


@pytest.fixture(scope="module")
def cs():
    from complex_valued_state_gb300 import build as cbuild
    from complex_valued_state_gb300 import cssd

    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for gpu tests")
    cbuild.build()
    cssd.load()
    return cssd


def rel_err(got, ref):
    return float(np.max(np.abs(np.asarray(got, np.complex128) - ref)) / max(np.max(np.abs(ref)), 1e-30))


def to_dev(d, keys):
    return {k: torch.from_numpy(np.ascontiguousarray(d[k])).cuda() for k in keys}


def case(N, P, batch=3, nheads=5):
    w = wl.DECODE.with_(batch=batch, nheads=nheads, dstate=N, headdim=P)
    return w, wl.decode_fixed(w), wl.decode_token(w, 0)


@pytest.mark.parametrize("N", [16, 32, 64, 128])
@pytest.mark.parametrize("P", [16, 32, 64])
@pytest.mark.parametrize("n", [0, 1, 7, 4096, 1_000_000])
def test_step_n_matches_closed_form(cs, oracle_lib, N, P, n):
    w, fx, tok = case(N, P)
    h = torch.from_numpy(fx["h"]).cuda()
    A, D = torch.from_numpy(fx["A"]).cuda(), torch.from_numpy(fx["D"]).cuda()
    t = to_dev(tok, TOK)
    y = cs.step_n(h, t["x"], t["dt"], A, t["B"], t["C"], D, n)
    torch.cuda.synchronize()
    hn, yn, _ = oracle_lib.geom_closed_form(fx["h"], tok["x"], tok["dt"], fx["A"], tok["B"], tok["C"], fx["D"], n)
    assert rel_err(y.cpu().numpy(), yn) < TOL
    assert rel_err(h.cpu().numpy(), hn) < TOL


def test_step_n_equals_the_step_loop(cs, oracle_lib):
    """37 calls of cssd_step, the oracle's 37-step loop and one cssd_step_n(37) agree."""
    w, fx, tok = case(64, 64, batch=4, nheads=6)
    A, D = torch.from_numpy(fx["A"]).cuda(), torch.from_numpy(fx["D"]).cuda()
    t = to_dev(tok, TOK)
    h_loop = torch.from_numpy(fx["h"]).cuda()
    for _ in range(37):
        y_loop = cs.step(h_loop, t["x"], t["dt"], A, t["B"], t["C"], D)
    h_once = torch.from_numpy(fx["h"]).cuda()
    y_once = cs.step_n(h_once, t["x"], t["dt"], A, t["B"], t["C"], D, 37)
    torch.cuda.synchronize()
    h_ref = fx["h"].astype(np.complex128)
    for _ in range(37):
        h_ref, y_ref = oracle_lib.cssd_step(h_ref, tok["x"], tok["dt"], fx["A"], tok["B"], tok["C"], fx["D"])
    assert rel_err(y_once.cpu().numpy(), y_ref) < TOL and rel_err(h_once.cpu().numpy(), h_ref) < TOL
    assert rel_err(y_loop.cpu().numpy(), y_ref) < TOL and rel_err(h_loop.cpu().numpy(), h_ref) < TOL


def test_step_n_zero_rate_adds_the_input_n_times(cs, oracle_lib):
    """A = 0 gives a = 1: the closed form's ratio is 0/0 and the kernel must
    take its limit, g_n = n.  The oracle's step loop is the reference."""
    w, fx, tok = case(32, 16, batch=2, nheads=3)
    A0 = np.zeros_like(fx["A"])
    h = torch.from_numpy(fx["h"]).cuda()
    t = to_dev(tok, TOK)
    y = cs.step_n(h, t["x"], t["dt"], torch.from_numpy(A0).cuda(), t["B"], t["C"],
                  torch.from_numpy(fx["D"]).cuda(), 50)
    torch.cuda.synchronize()
    h_ref = fx["h"].astype(np.complex128)
    for _ in range(50):
        h_ref, y_ref = oracle_lib.cssd_step(h_ref, tok["x"], tok["dt"], A0, tok["B"], tok["C"], fx["D"])
    assert rel_err(y.cpu().numpy(), y_ref) < TOL
    assert rel_err(h.cpu().numpy(), h_ref) < TOL


def test_decode_constant_input_run_in_one_call_sampled_heads(cs, oracle_lib):
    """The decode workload's 4096-step constant-input run, as one call, at full size."""
    w = wl.DECODE
    fx = wl.decode_fixed(w)
    tok = wl.decode_token(w, 0)
    h = torch.from_numpy(fx["h"]).cuda()
    A, D = torch.from_numpy(fx["A"]).cuda(), torch.from_numpy(fx["D"]).cuda()
    t = to_dev(tok, TOK)
    y = cs.step_n(h, t["x"], t["dt"], A, t["B"], t["C"], D, 4096)
    torch.cuda.synchronize()
    bs, hs = np.array([0, 77, 255]), np.array([1, 17, 31])
    sub = {k: tok[k][bs][:, hs] for k in tok}
    hn, yn, _ = oracle_lib.geom_closed_form(fx["h"][bs][:, hs], sub["x"], sub["dt"], fx["A"][hs], sub["B"],
                                            sub["C"], fx["D"][hs], 4096)
    assert rel_err(y.cpu().numpy()[bs][:, hs], yn) < TOL
    assert rel_err(h.cpu().numpy()[bs][:, hs], hn) < TOL


def test_step_infinite_matches_limit_full_size(cs, oracle_lib):
    w = wl.DECODE
    fx = wl.decode_fixed(w)
    tok = wl.decode_token(w, 0)
    t = to_dev(tok, TOK)
    A, D = torch.from_numpy(fx["A"]).cuda(), torch.from_numpy(fx["D"]).cuda()
    y = cs.step_infinite(t["x"], t["dt"], A, t["B"], t["C"], D)
    torch.cuda.synchronize()
    bs = np.array([0, 1, 128, 255])
    sub = {k: tok[k][bs] for k in tok}
    _, _, yinf = oracle_lib.geom_closed_form(fx["h"][bs], sub["x"], sub["dt"], fx["A"], sub["B"], sub["C"],
                                             fx["D"], 1)
    assert rel_err(y.cpu().numpy()[bs], yinf) < TOL


@pytest.mark.parametrize("N", [16, 128])
def test_long_constant_run_approaches_the_limit(cs, N):
    """For decaying heads (|a| < 1) the n-step output converges to y_inf."""
    w, fx, tok = case(N, 32, batch=2, nheads=4)
    A, D = torch.from_numpy(fx["A"]).cuda(), torch.from_numpy(fx["D"]).cuda()
    t = to_dev(tok, TOK)
    h = torch.from_numpy(fx["h"]).cuda()
    y_n = cs.step_n(h, t["x"], t["dt"], A, t["B"], t["C"], D, 10**7)
    y_inf = cs.step_infinite(t["x"], t["dt"], A, t["B"], t["C"], D)
    torch.cuda.synchronize()
    assert rel_err(y_n.cpu().numpy(), y_inf.cpu().numpy().astype(np.complex128)) < TOL
