"""GPU parity at the largest sizes the boundary accepts along the grid's
batch dimension (65535, the CUDA limit of a grid's y and z extent that the
CUDA-core kernels put the batch on), for the CUDA-core and tensor-core forwards
and the decode step.  Sampled batch rows are compared with the oracle, which
computes each (batch, head) independently.

Bar: max |got - ref| <= 2e-3 * max |ref| (complex modulus), per output tensor.
"""

import numpy as np
import pytest
import torch

from complex_valued_state_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

TOL = 2e-3
BMAX = 65535
ROWS = [0, 1, 32767, BMAX - 1]
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
    return float(np.max(np.abs(np.asarray(got, np.complex128) - ref)) / max(np.max(np.abs(ref)), 1e-30))


def rows_of(d, rows):
    return {k: (v if k in ("A", "D") else v[rows]) for k, v in d.items()}


# (128, 16): the CUDA-core kernels (dstate 128 with a smaller headdim);
# (16, 16): the half-operand kernel padded to 64; (64, 64): the same kernel unpadded
@pytest.mark.parametrize("N,P,T", [(128, 16, 3), (16, 16, 3), (64, 64, 2)])
def test_forward_at_batch_limit(cs, oracle_lib, N, P, T):
    d = wl.random_case(9100 + N, BMAX, T, 1, N, P)
    g = {k: torch.from_numpy(np.ascontiguousarray(d[k])).cuda() for k in KEYS}
    y, hf = cs.chunked_forward(**g, chunk=64)
    torch.cuda.synchronize()
    y_ref, h_ref = oracle_lib.cssd_naive(**rows_of(d, ROWS))
    assert rel_err(y.cpu().numpy()[ROWS], y_ref) < TOL
    assert rel_err(hf.cpu().numpy()[ROWS], h_ref) < TOL


def test_step_at_batch_limit(cs, oracle_lib):
    N = P = 16
    w = wl.DECODE.with_(batch=BMAX, nheads=1, dstate=N, headdim=P)
    fx = wl.decode_fixed(w)
    tok = wl.decode_token(w, 0)
    h = torch.from_numpy(fx["h"]).cuda()
    t = {k: torch.from_numpy(np.ascontiguousarray(tok[k])).cuda() for k in ("x", "dt", "B", "C")}
    y = cs.step(h, t["x"], t["dt"], torch.from_numpy(fx["A"]).cuda(), t["B"], t["C"], torch.from_numpy(fx["D"]).cuda())
    torch.cuda.synchronize()
    h_ref, y_ref = oracle_lib.cssd_step(fx["h"][ROWS], tok["x"][ROWS], tok["dt"][ROWS], fx["A"], tok["B"][ROWS],
                                        tok["C"][ROWS], fx["D"])
    assert rel_err(y.cpu().numpy()[ROWS], y_ref) < TOL
    assert rel_err(h.cpu().numpy()[ROWS], h_ref) < TOL
