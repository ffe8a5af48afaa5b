"""cssd_chunked_forward_noalloc, the forward for callers that cannot allocate.

Some callers cannot allocate device memory when they call the forward: their
device heap belongs to another allocator, or allocation is not allowed on
their latency-critical path.  This entry point runs on scratch that is part
of the library's device image.  The test calls it through the C ABI twice in a
row (the second call finds the first call's leftovers in the shared scratch)
and checks both results against the ordinary entry point, within the parity
tolerance used everywhere else (2e-3 of the largest reference magnitude).
It runs last so that a failure here leaves every other test already run.
"""

import ctypes

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
    return float(np.max(np.abs(got - ref)) / max(np.max(np.abs(ref)), 1e-30))


def noalloc_call(cs, g, y, h, chunk):
    lib = cs.load()
    Bz, T, H, P = g["x"].shape
    N = g["B"].shape[-1]
    d = cs.Dims(Bz, T, H, N, P)
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.cssd_chunked_forward_noalloc(ctypes.byref(d), p(g["x"]), p(g["dt"]), p(g["A"]), p(g["B"]),
                                            p(g["C"]), p(g["D"]), p(y), p(h), chunk, stream)


@pytest.mark.parametrize("shape", [(2, 300, 3, 64, 64, 64), (1, 257, 2, 16, 32, 64), (2, 130, 2, 128, 64, 128)])
def test_noalloc_matches_forward_on_two_calls(cs, shape):
    Bz, T, H, N, P, chunk = shape
    d = wl.random_case(77 + T, Bz, T, H, N, P)
    g = {k: torch.from_numpy(d[k]).cuda() for k in KEYS}
    y_ref, h_ref = cs.chunked_forward(**g, chunk=chunk)
    y_ref, h_ref = y_ref.cpu().numpy(), h_ref.cpu().numpy()
    for _ in range(2):
        y = torch.full((Bz, T, H, P), float("nan"), dtype=torch.complex64, device="cuda")
        h = torch.full((Bz, H, N, P), float("nan"), dtype=torch.complex64, device="cuda")
        assert noalloc_call(cs, g, y, h, chunk) == 0
        torch.cuda.synchronize()
        assert rel_err(y.cpu().numpy(), y_ref) < TOL
        assert rel_err(h.cpu().numpy(), h_ref) < TOL


def test_noalloc_rejects_sizes_beyond_its_scratch(cs):
    # the tensor-core path keeps 128 KiB of hand-off words per sequence and
    # state half: 160 sequences need 20 MiB
    Bz, T, H, N, P, chunk = 1, 64, 160, 64, 64, 64
    need = cs.workspace_bytes(Bz, T, H, N, P, chunk)
    assert need > cs.NOALLOC_SCRATCH_BYTES
    d = wl.random_case(5, Bz, T, H, N, P)
    g = {k: torch.from_numpy(d[k]).cuda() for k in KEYS}
    y = torch.zeros((Bz, T, H, P), dtype=torch.complex64, device="cuda")
    h = torch.zeros((Bz, H, N, P), dtype=torch.complex64, device="cuda")
    assert noalloc_call(cs, g, y, h, chunk) == -5
    torch.cuda.synchronize()
    assert not torch.any(y != 0).item()
