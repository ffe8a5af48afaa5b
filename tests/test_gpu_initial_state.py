"""GPU parity of the forward started from a given state (cssd_chunked_forward_h0)
and of the forward over host tensors streamed through the device in pieces
(cssd_chunked_forward_host), against the CPU oracle's sequential recurrence
started from the same state.

Bar: max |got - ref| <= 2e-3 * max |ref| (complex modulus) per output tensor,
the tolerance of the workload statement.
"""

import numpy as np
import pytest
import torch

from complex_valued_state_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

TOL = 2e-3
KEYS = ("x", "dt", "A", "B", "C", "D")
SEQ = ("x", "dt", "B", "C")


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


def pinned(d, keys=KEYS):
    return {k: torch.from_numpy(np.ascontiguousarray(d[k])).pin_memory() for k in keys}


SHAPES = ((16, 16), (32, 64), (64, 64), (128, 64), (64, 32))


@pytest.mark.parametrize("N,P", SHAPES)
@pytest.mark.parametrize("chunk", (64, 128))
@pytest.mark.parametrize("T", (1, 65, 200))
def test_forward_from_initial_state(cs, oracle_lib, N, P, chunk, T):
    d = wl.random_case(7100 + N + P + T + chunk, 2, T, 3, N, P)
    h0 = wl.random_state(7200 + N + P, 2, 3, N, P)
    y, hf = cs.chunked_forward(**dev(d), chunk=chunk, h0=torch.from_numpy(h0).cuda())
    torch.cuda.synchronize()
    y_ref, h_ref = oracle_lib.cssd_naive(**d, h0=h0)
    assert rel_err(y.cpu().numpy(), y_ref) < TOL
    assert rel_err(hf.cpu().numpy(), h_ref) < TOL


def test_zero_initial_state_equals_plain_forward(cs):
    d = wl.random_case(7300, 2, 150, 3, 64, 64)
    g = dev(d)
    y0, h0f = cs.chunked_forward(**g, chunk=64)
    y1, h1f = cs.chunked_forward(**g, chunk=64, h0=torch.zeros((2, 3, 64, 64), dtype=torch.complex64, device="cuda"))
    torch.cuda.synchronize()
    assert torch.equal(y0, y1) and torch.equal(h0f, h1f)


@pytest.mark.parametrize("N,P", ((64, 64), (128, 64), (16, 32)))
@pytest.mark.parametrize("T1", (64, 100))
def test_forward_in_two_pieces_equals_whole(cs, oracle_lib, N, P, T1):
    T = 300
    d = wl.random_case(7400 + N + T1, 2, T, 3, N, P)
    first = {k: (v[:, :T1] if k in SEQ else v) for k, v in d.items()}
    rest = {k: (v[:, T1:] if k in SEQ else v) for k, v in d.items()}
    ya, ha = cs.chunked_forward(**dev(first), chunk=64)
    yb, hb = cs.chunked_forward(**dev(rest), chunk=64, h0=ha)
    torch.cuda.synchronize()
    y_ref, h_ref = oracle_lib.cssd_naive(**d)
    assert rel_err(ya.cpu().numpy(), y_ref[:, :T1]) < TOL
    assert rel_err(yb.cpu().numpy(), y_ref[:, T1:]) < TOL
    assert rel_err(hb.cpu().numpy(), h_ref) < TOL


@pytest.mark.parametrize("N,P", ((64, 64), (32, 32)))
def test_continuation_in_place(cs, oracle_lib, N, P):
    d = wl.random_case(7500 + N, 2, 130, 2, N, P)
    h0 = wl.random_state(7501, 2, 2, N, P)
    h = torch.from_numpy(h0).cuda()
    y, hf = cs.chunked_forward(**dev(d), chunk=64, h0=h, h_final=h)
    torch.cuda.synchronize()
    assert hf.data_ptr() == h.data_ptr()
    y_ref, h_ref = oracle_lib.cssd_naive(**d, h0=h0)
    assert rel_err(y.cpu().numpy(), y_ref) < TOL
    assert rel_err(h.cpu().numpy(), h_ref) < TOL


@pytest.mark.parametrize("N,P", ((64, 64), (128, 64), (16, 16)))
@pytest.mark.parametrize("piece", (0, 64, 100, 300))
@pytest.mark.parametrize("with_h0", (False, True))
def test_host_forward(cs, oracle_lib, N, P, piece, with_h0):
    T = 300
    d = wl.random_case(7600 + N + piece, 2, T, 3, N, P)
    h0 = wl.random_state(7601 + N, 2, 3, N, P) if with_h0 else None
    y, hf = cs.chunked_forward_host(**pinned(d), chunk=64, piece_len=piece,
                                    h0=None if h0 is None else torch.from_numpy(h0).pin_memory())
    torch.cuda.synchronize()
    assert y.device.type == "cpu" and hf.device.type == "cpu"
    y_ref, h_ref = oracle_lib.cssd_naive(**d, h0=h0)
    assert rel_err(y.numpy(), y_ref) < TOL
    assert rel_err(hf.numpy(), h_ref) < TOL


def test_host_forward_state_on_device_and_own_buffer(cs, oracle_lib):
    T, N, P = 257, 64, 64
    d = wl.random_case(7700, 2, T, 3, N, P)
    h0 = wl.random_state(7701, 2, 3, N, P)
    buf = torch.empty(cs.host_forward_device_bytes(2, T, 3, N, P, 128, 128), dtype=torch.uint8, device="cuda")
    hf = torch.empty((2, 3, N, P), dtype=torch.complex64, device="cuda")
    s = torch.cuda.Stream()
    y, _ = cs.chunked_forward_host(**pinned(d), chunk=128, piece_len=128, h0=torch.from_numpy(h0).cuda(),
                                   h_final=hf, device_buffer=buf, stream=s)
    s.synchronize()
    y_ref, h_ref = oracle_lib.cssd_naive(**d, h0=h0)
    assert rel_err(y.numpy(), y_ref) < TOL
    assert rel_err(hf.cpu().numpy(), h_ref) < TOL


def test_host_forward_pageable_memory(cs, oracle_lib):
    d = wl.random_case(7800, 1, 200, 2, 64, 64)
    host = {k: torch.from_numpy(np.ascontiguousarray(d[k])) for k in KEYS}
    y = torch.empty((1, 200, 2, 64), dtype=torch.complex64)
    hf = torch.empty((1, 2, 64, 64), dtype=torch.complex64)
    cs.chunked_forward_host(**host, chunk=64, piece_len=64, y=y, h_final=hf)
    torch.cuda.synchronize()
    y_ref, h_ref = oracle_lib.cssd_naive(**d)
    assert rel_err(y.numpy(), y_ref) < TOL and rel_err(hf.numpy(), h_ref) < TOL


def test_host_forward_mamba2_layer_sampled_heads(cs, oracle_lib):
    w = wl.MAMBA2_LAYER
    d = wl.make_inputs(w)
    y, hf = cs.chunked_forward_host(**pinned(d), chunk=w.chunk)
    torch.cuda.synchronize()
    heads = [0, 23]
    sub = {k: (v[heads] if k in ("A", "D") else v[:, :, heads]) for k, v in d.items() if k in KEYS}
    y_ref, h_ref = oracle_lib.cssd_naive(**sub)
    assert rel_err(y.numpy()[:, :, heads], y_ref) < TOL
    assert rel_err(hf.numpy()[:, heads], h_ref) < TOL
    # every head agrees with the device forward over the whole sequence (the
    # pieces restart the rotated frame, so TF32 rounding differs slightly)
    yd, hd = cs.chunked_forward(**dev(d), chunk=w.chunk)
    torch.cuda.synchronize()
    assert rel_err(y.numpy(), yd.cpu().numpy().astype(np.complex128)) < TOL
    assert rel_err(hf.numpy(), hd.cpu().numpy().astype(np.complex128)) < TOL
