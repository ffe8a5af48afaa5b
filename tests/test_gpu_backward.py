"""GPU parity of the gradients (cssd_chunked_backward) against the backward
oracle on the same seeded inputs and upstream gradient.
Bar, per gradient: max |g_gpu - g_ref| <= 2e-3 max |g_ref| (the forward's
bar: the gradients of B and C run through the same TF32 forward kernels)."""

import numpy as np
import pytest
import torch

from complex_valued_state_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

TOL = 2e-3
KEYS = ("gx", "gdt", "gA", "gB", "gC", "gD")


@pytest.fixture(scope="module")
def cs():
    from complex_valued_state_gb300 import build as cbuild
    from complex_valued_state_gb300 import cssd

    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for gpu tests")
    cbuild.build()
    cssd.load()
    return cssd


@pytest.fixture(scope="module")
def orc():
    import oracle

    oracle.build()
    return oracle


def upstream(seed, shape):
    rng = np.random.default_rng(seed)
    return ((rng.standard_normal(shape) + 1j * rng.standard_normal(shape)) / np.sqrt(2)).astype(np.complex64)


def run(cs, d, dy, chunk):
    g = {k: torch.from_numpy(np.ascontiguousarray(d[k])).cuda() for k in ("x", "dt", "A", "B", "C", "D")}
    out = cs.chunked_backward(**g, dy=torch.from_numpy(dy).cuda(), chunk=chunk)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}


def rel_err(got, ref):
    got, ref = np.asarray(got, np.complex128), np.asarray(ref, np.complex128)
    return float(np.max(np.abs(got - ref)) / max(np.max(np.abs(ref)), 1e-30))


@pytest.mark.parametrize("N,P", [(16, 16), (64, 64), (32, 64), (64, 16), (16, 32)])
@pytest.mark.parametrize("T", [1, 63, 65, 200])
def test_matches_oracle(cs, orc, N, P, T):
    d = wl.random_case(N * 7 + P + T, 2, T, 3, N, P)
    dy = upstream(T + N, (2, T, 3, P))
    got = run(cs, d, dy, 64)
    ref = orc.cssd_backward(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], dy)
    for k in KEYS:
        assert rel_err(got[k], ref[k]) < TOL, k


@pytest.mark.parametrize("T,chunk", [(64, 64), (128, 64), (640, 128), (1024, 64)])
def test_chunk_boundary_sums(cs, orc, T, chunk):
    """dstate = headdim = 64 with T a multiple of 64: the step and rate
    gradients come from chunk-local sums plus the inner products of the
    forward and adjoint states at the chunk boundaries."""
    d = wl.random_case(4000 + T + chunk, 2, T, 3, 64, 64)
    dy = upstream(4100 + T, (2, T, 3, 64))
    got = run(cs, d, dy, chunk)
    ref = orc.cssd_backward(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], dy)
    for k in KEYS:
        assert rel_err(got[k], ref[k]) < TOL, k


def test_chunk_128(cs, orc):
    d = wl.random_case(5, 1, 300, 2, 64, 64)
    dy = upstream(6, (1, 300, 2, 64))
    got = run(cs, d, dy, 128)
    ref = orc.cssd_backward(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], dy)
    for k in KEYS:
        assert rel_err(got[k], ref[k]) < TOL, k


def test_deterministic(cs):
    d = wl.random_case(7, 2, 150, 4, 64, 64)
    dy = upstream(8, (2, 150, 4, 64))
    a, b = run(cs, d, dy, 64), run(cs, d, dy, 64)
    for k in KEYS:
        assert np.array_equal(a[k], b[k]), k


def test_mamba2_layer_shape_two_heads(cs, orc):
    """The mamba2_layer shape (batch 4, T 2048, N = P = 64); heads 0 and 23 of
    every batch row against the oracle (gA and gD sum over the batch)."""
    w = wl.MAMBA2_LAYER
    d = wl.make_inputs(w)
    dy = upstream(9, (w.batch, w.seqlen, w.nheads, w.headdim))
    got = run(cs, d, dy, w.chunk)
    for h in (0, 23):
        sub = {k: (d[k][:, :, h:h + 1] if d[k].ndim >= 3 else d[k][h:h + 1]) for k in ("x", "dt", "B", "C")}
        sub["A"], sub["D"] = d["A"][h:h + 1], d["D"][h:h + 1]
        ref = orc.cssd_backward(sub["x"], sub["dt"], sub["A"], sub["B"], sub["C"], sub["D"], dy[:, :, h:h + 1])
        for k in ("gx", "gdt", "gB", "gC"):
            assert rel_err(got[k][:, :, h:h + 1], ref[k]) < TOL, (h, k)
        assert rel_err(got["gA"][h:h + 1], ref["gA"]) < TOL and rel_err(got["gD"][h:h + 1], ref["gD"]) < TOL


@pytest.mark.parametrize("P", [64, 32])
@pytest.mark.parametrize("T,chunk", [(1, 64), (65, 64), (200, 128), (257, 128)])
def test_dstate_128(cs, orc, P, T, chunk):
    """dstate 128: y and gx on the fp32 CUDA-core kernels, the transposed-state
    runs of gB and gC with headdim 128 on the same kernels."""
    d = wl.random_case(6000 + P + T, 2, T, 3, 128, P)
    dy = upstream(6100 + T, (2, T, 3, P))
    got = run(cs, d, dy, chunk)
    ref = orc.cssd_backward(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], dy)
    for k in KEYS:
        assert rel_err(got[k], ref[k]) < TOL, k


def test_long_seq_shape_dstate_128(cs, orc):
    """The long_seq shape (dstate 128, headdim 64, chunk 128, slow decay) over
    4096 tokens on two heads; the oracle keeps every state of the sequence."""
    w = wl.LONG_SEQ.with_(seqlen=4096, nheads=2)
    d = wl.make_inputs(w)
    dy = upstream(12, (w.batch, w.seqlen, w.nheads, w.headdim))
    got = run(cs, d, dy, w.chunk)
    ref = orc.cssd_backward(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], dy)
    for k in KEYS:
        assert rel_err(got[k], ref[k]) < TOL, k
