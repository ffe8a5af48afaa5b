"""cssd_chunked_forward_noalloc, the forward for callers that cannot allocate.

Some callers cannot allocate device memory when they call the forward: their
device heap belongs to another allocator, or allocation is not allowed on
their latency-critical path.  This entry point runs on scratch that is part
of the library's device image, which every call shares and which keeps the
last call's contents.

The test calls it through the C ABI twice in a row per shape.  The second call
takes different inputs (another seed) and fewer sequences and tokens, so any
hand-off word, ticket or error word the kernels failed to clear would hand the
second call the first call's values.  Each call is checked against the
ordinary entry point on its own inputs, the first shape's first call also
against the CPU oracle, all within the parity tolerance used everywhere else
(2e-3 of the largest reference magnitude), and the library's status word must
show no bounded wait giving up.  It runs last so that a failure here leaves
every other test already run.
"""

import ctypes

import numpy as np
import pytest
import torch

import oracle
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


def noalloc_call(cs, g, y, h, chunk, stream=None):
    lib = cs.load()
    Bz, T, H, P = g["x"].shape
    N = g["B"].shape[-1]
    d = cs.Dims(Bz, T, H, N, P)
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    st = torch.cuda.current_stream() if stream is None else stream
    return lib.cssd_chunked_forward_noalloc(ctypes.byref(d), p(g["x"]), p(g["dt"]), p(g["A"]), p(g["B"]),
                                            p(g["C"]), p(g["D"]), p(y), p(h), chunk, ctypes.c_void_p(st.cuda_stream))


# (Bz, T, H) of the first call, (Bz, T, H) of the second, N, P, chunk
SHAPES = [
    ((2, 300, 3), (1, 200, 2), 64, 64, 64),
    ((1, 257, 2), (1, 130, 1), 16, 32, 64),
    ((2, 130, 2), (1, 129, 2), 128, 64, 128),
]


@pytest.mark.parametrize("case", range(len(SHAPES)))
def test_noalloc_matches_forward_on_two_calls(cs, case):
    first, second, N, P, chunk = SHAPES[case]
    side = torch.cuda.Stream()
    cs.device_status(clear=True)
    for call, (Bz, T, H) in enumerate((first, second)):
        d = wl.random_case(77 + 13 * call + T, Bz, T, H, N, P)
        g = {k: torch.from_numpy(d[k]).cuda() for k in KEYS}
        y_ref, h_ref = cs.chunked_forward(**g, chunk=chunk)
        y_ref, h_ref = y_ref.cpu().numpy(), h_ref.cpu().numpy()
        y = torch.full((Bz, T, H, P), float("nan"), dtype=torch.complex64, device="cuda")
        h = torch.full((Bz, H, N, P), float("nan"), dtype=torch.complex64, device="cuda")
        torch.cuda.synchronize()
        # the first call on the default stream, the second on a side stream
        assert noalloc_call(cs, g, y, h, chunk, stream=None if call == 0 else side) == 0
        torch.cuda.synchronize()
        y, h = y.cpu().numpy(), h.cpu().numpy()
        assert rel_err(y, y_ref) < TOL
        assert rel_err(h, h_ref) < TOL
        if case == 0 and call == 0:
            y_or, h_or = oracle.cssd_naive(*(d[k] for k in KEYS))
            assert rel_err(y, y_or) < TOL
            assert rel_err(h, h_or) < TOL
    assert cs.device_status() == 0


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
