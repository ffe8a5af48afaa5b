"""The forward over inputs whose magnitudes lie far from 1, or differ widely
inside one tile or between chunks.  The dstate-64 forward rounds its GEMM
operands to IEEE half after a power-of-two scale per tile and operand; these
cases check that the scales keep every operand inside the half range and that
the epilogues take them out exactly, against the oracle (fp64).  The dstate-128
forward (TF32 operands) runs the same cases.

Bar: max |got - ref| <= 2e-3 * max |ref| (complex modulus), per output tensor.
"""

import numpy as np
import pytest
import torch

from complex_valued_state_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

TOL = 2e-3
KEYS = ("x", "dt", "A", "B", "C", "D")


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
    return float(np.max(np.abs(np.asarray(got, np.complex128) - ref)) / max(np.max(np.abs(ref)), 1e-300))


def run(cs, oracle_lib, d, chunk=64):
    g = {k: torch.from_numpy(np.ascontiguousarray(d[k])).cuda() for k in KEYS}
    y, h = cs.chunked_forward(**g, chunk=chunk)
    torch.cuda.synchronize()
    y_ref, h_ref = oracle_lib.cssd_naive(**d)
    assert np.all(np.isfinite(y.cpu().numpy())) and np.all(np.isfinite(h.cpu().numpy()))
    return rel_err(y.cpu().numpy(), y_ref), rel_err(h.cpu().numpy(), h_ref)


@pytest.mark.parametrize("N", [64, 128])
@pytest.mark.parametrize("sx,sb,sc", [(1e12, 1e-9, 1e3), (1e-8, 1e-6, 1e-4), (3e5, 2e4, 1e-3), (1.0, 1e8, 1e-8)])
def test_scaled_inputs(cs, oracle_lib, N, sx, sb, sc):
    """x, B and C multiplied by factors from 1e-8 to 1e12: each lies outside
    the half range (6e-5 to 65504) at one end or the other, unscaled."""
    d = wl.random_case(9600 + N, 2, 200, 3, N, 64)
    d["x"] = (d["x"] * sx).astype(np.complex64)
    d["B"] = (d["B"] * sb).astype(np.complex64)
    d["C"] = (d["C"] * sc).astype(np.complex64)
    d["D"][:] = 0  # y is then the state-space part alone
    ey, eh = run(cs, oracle_lib, d)
    assert ey < TOL and eh < TOL, (ey, eh)


@pytest.mark.parametrize("N", [64, 128])
def test_magnitudes_differ_inside_a_tile(cs, oracle_lib, N):
    """One token per tile carries x and B a thousand times larger than the
    rest, and every fifth token's C is a thousand times smaller."""
    d = wl.random_case(9610 + N, 2, 256, 2, N, 64)
    big = np.arange(256) % 64 == 17
    d["x"][:, big] *= 1e3
    d["B"][:, big] *= 1e3
    d["C"][:, np.arange(256) % 5 == 0] *= 1e-3
    ey, eh = run(cs, oracle_lib, d)
    assert ey < TOL and eh < TOL, (ey, eh)


@pytest.mark.parametrize("N", [64, 128])
def test_chunks_of_different_scale(cs, oracle_lib, N):
    """The first two chunks have x a million times smaller than the rest, so
    tile scales differ by 2^20 along the sequence while the carried state
    mixes them."""
    d = wl.random_case(9620 + N, 1, 320, 2, N, 64, dt_mean=-3.0)
    d["x"][:, :128] *= 1e-6
    ey, eh = run(cs, oracle_lib, d)
    assert ey < TOL and eh < TOL, (ey, eh)


@pytest.mark.parametrize("N", [64, 128])
def test_zero_tiles(cs, oracle_lib, N):
    """All-zero x in the first and third chunks (a tile whose largest x
    component is 0), zero B in the last, partial chunk."""
    d = wl.random_case(9630 + N, 2, 230, 2, N, 64)
    d["x"][:, :64] = 0
    d["x"][:, 128:192] = 0
    d["B"][:, 192:] = 0
    ey, eh = run(cs, oracle_lib, d)
    assert ey < TOL and eh < TOL, (ey, eh)


@pytest.mark.parametrize("N", [64, 128])
def test_growing_state(cs, oracle_lib, N):
    """A = 0 (no decay, no rotation) over 1024 tokens with x of one sign
    pattern: the state grows like T (to about 2e4, near the largest half
    value unscaled), so the carried-in state's scale moves from tile to tile."""
    d = wl.random_case(9640 + N, 1, 1024, 2, N, 64, a_scale=0.0)
    d["x"] = (100 * (np.abs(d["x"].real) + 1j * np.abs(d["x"].imag))).astype(np.complex64)
    d["B"][:] = d["B"][:, :1]  # one B for every token
    ey, eh = run(cs, oracle_lib, d)
    assert ey < TOL and eh < TOL, (ey, eh)
