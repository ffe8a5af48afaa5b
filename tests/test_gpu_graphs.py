"""The entry points inside CUDA graphs: calls captured on a stream (the
library's host-side checks are legal during capture) and replayed give the
oracle's results.  A decode loop is the case graphs serve: one replay runs many
launch-bound steps without host work between them.

Bar: max |got - ref| <= 2e-3 * max |ref| (complex modulus)."""

import numpy as np
import pytest
import torch

from complex_valued_state_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

TOL = 2e-3


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


@pytest.mark.parametrize("N,P", [(128, 64), (16, 32)])
def test_decode_loop_in_a_graph(cs, oracle_lib, N, P):
    steps = 8
    w = wl.DECODE.with_(batch=4, nheads=6, dstate=N, headdim=P)
    fx = wl.decode_fixed(w)
    toks = [wl.decode_token(w, s) for s in range(steps)]
    A, D = torch.from_numpy(fx["A"]).cuda(), torch.from_numpy(fx["D"]).cuda()
    t = [{k: torch.from_numpy(np.ascontiguousarray(tok[k])).cuda() for k in ("x", "dt", "B", "C")} for tok in toks]
    h = torch.from_numpy(fx["h"]).cuda()
    ys = [torch.empty((w.batch, w.nheads, P), dtype=torch.complex64, device="cuda") for _ in range(steps)]
    # one eager call first (kernel attributes and lazy loading outside the capture), then restore h
    h_keep = h.clone()
    cs.step(h, t[0]["x"], t[0]["dt"], A, t[0]["B"], t[0]["C"], D, y=ys[0])
    h.copy_(h_keep)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for s in range(steps):
            cs.step(h, t[s]["x"], t[s]["dt"], A, t[s]["B"], t[s]["C"], D, y=ys[s])
    h.copy_(h_keep)  # capturing launches nothing; the state is still the initial one
    g.replay()
    torch.cuda.synchronize()
    h_ref = fx["h"].astype(np.complex128)
    for s in range(steps):
        h_ref, y_ref = oracle_lib.cssd_step(h_ref, toks[s]["x"], toks[s]["dt"], fx["A"], toks[s]["B"], toks[s]["C"],
                                            fx["D"])
        assert rel_err(ys[s].cpu().numpy(), y_ref) < TOL, s
    assert rel_err(h.cpu().numpy(), h_ref) < TOL


def test_forward_and_step_in_a_graph(cs, oracle_lib):
    T = 200
    d = wl.random_case(9500, 2, T + 1, 3, 64, 64)
    head = {k: (np.ascontiguousarray(v[:, :T]) if k in ("x", "dt", "B", "C") else v) for k, v in d.items()}
    g_in = {k: torch.from_numpy(head[k]).cuda() for k in head}
    tok = {k: torch.from_numpy(np.ascontiguousarray(d[k][:, T])).cuda() for k in ("x", "dt", "B", "C")}
    y = torch.empty((2, T, 3, 64), dtype=torch.complex64, device="cuda")
    h = torch.empty((2, 3, 64, 64), dtype=torch.complex64, device="cuda")
    y1 = torch.empty((2, 3, 64), dtype=torch.complex64, device="cuda")
    ws = torch.empty(cs.workspace_bytes(2, T, 3, 64, 64, 64), dtype=torch.uint8, device="cuda")

    def run():
        cs.chunked_forward(**g_in, chunk=64, y=y, h_final=h, workspace=ws)
        cs.step(h, tok["x"], tok["dt"], g_in["A"], tok["B"], tok["C"], g_in["D"], y=y1)

    run()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        run()
    y.zero_()
    y1.zero_()
    graph.replay()
    torch.cuda.synchronize()
    y_ref, h_ref = oracle_lib.cssd_naive(**d)
    assert rel_err(y.cpu().numpy(), y_ref[:, :T]) < TOL
    assert rel_err(y1.cpu().numpy(), y_ref[:, T]) < TOL
    assert rel_err(h.cpu().numpy(), h_ref) < TOL
