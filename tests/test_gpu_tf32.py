"""GPU parity of the TF32-operand forward (cssd_chunked_forward_tf32) against
the CPU oracle, and the operand-precision comparison with the default forward.

The default forward takes half operands with a power-of-two scale per tile and
operand on every tensor-core shape (dstate and headdim up to 64, padded to 64
below that, and dstate 128 with headdim 64); cssd_chunked_forward_tf32 keeps
TF32 on the unpadded shapes (headdim 64, dstate 64 or 128) and runs the fp32
CUDA-core kernels on the others.  Where both are 11-bit operand paths the half-operand
error must stay within twice the TF32 error (plus a floor of 1e-5 of the
largest magnitude for cases where both are tiny); the tiny workload (dstate =
headdim = 16) compares half operands with fp32 and is held to the parity bar
only.  Tolerance of the parity checks: max |got - ref| <= 2e-3 * max |ref| per
output tensor.

Run with -s to see the per-workload error table.
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
    return float(np.max(np.abs(np.asarray(got, np.complex128) - ref)) / max(np.max(np.abs(ref)), 1e-30))


def dev(d, keys=KEYS):
    return {k: torch.from_numpy(np.ascontiguousarray(d[k])).cuda() for k in keys}


@pytest.mark.parametrize("N,P,chunk", ((64, 64, 64), (64, 64, 128), (128, 64, 128), (16, 32, 64)))
@pytest.mark.parametrize("T", (1, 65, 300))
@pytest.mark.parametrize("with_h0", (False, True))
def test_tf32_forward(cs, oracle_lib, N, P, chunk, T, with_h0):
    d = wl.random_case(9100 + N + P + T + chunk, 2, T, 3, N, P)
    h0 = wl.random_state(9200 + N, 2, 3, N, P) if with_h0 else None
    y, hf = cs.chunked_forward(**dev(d), chunk=chunk, tf32=True,
                               h0=None if h0 is None else torch.from_numpy(h0).cuda())
    torch.cuda.synchronize()
    y_ref, h_ref = oracle_lib.cssd_naive(**d, h0=h0)
    assert rel_err(y.cpu().numpy(), y_ref) < TOL
    assert rel_err(hf.cpu().numpy(), h_ref) < TOL


def _heads(d, w, heads):
    """The inputs of a subset of heads (all batch rows)."""
    out = {}
    for k in KEYS:
        a = d[k]
        out[k] = np.ascontiguousarray(a[heads] if a.ndim == 1 else a[:, :, heads])
    return out


# workload, heads checked (None = all)
TABLE = (("tiny", None), ("mamba2_layer", None), ("long_seq", [0, 13, 31]), ("pam", None))


@pytest.mark.parametrize("name,heads", TABLE)
def test_half_operands_within_twice_tf32(cs, oracle_lib, name, heads):
    w = wl.WORKLOADS[name]
    d = wl.make_inputs(w)
    d = {k: d[k] for k in KEYS}
    if heads is not None:
        d = _heads(d, w, heads)
    g = dev(d)
    y16, h16 = cs.chunked_forward(**g, chunk=w.chunk)
    y32, h32 = cs.chunked_forward(**g, chunk=w.chunk, tf32=True)
    torch.cuda.synchronize()
    y_ref, h_ref = oracle_lib.cssd_naive(**d)
    e = {"y_default": rel_err(y16.cpu().numpy(), y_ref), "h_default": rel_err(h16.cpu().numpy(), h_ref),
         "y_tf32": rel_err(y32.cpu().numpy(), y_ref), "h_tf32": rel_err(h32.cpu().numpy(), h_ref)}
    print(f"\nerror table {name}: " + " ".join(f"{k}={v:.3e}" for k, v in e.items()))
    for k in ("y", "h"):
        assert e[f"{k}_tf32"] < TOL and e[f"{k}_default"] < TOL
        if w.headdim == 64 and w.dstate in (64, 128):
            assert e[f"{k}_default"] <= 2 * e[f"{k}_tf32"] + 1e-5
