"""Calls from several host threads at once, each on its own CUDA stream: the
library's per-device caches (kernel attributes, resident-CTA counts, the status
word's address) are filled concurrently, and every result still matches the
oracle.  The binding's foreign calls release the interpreter lock, so the
threads' calls overlap.

Bar: max |got - ref| <= 2e-3 * max |ref| (complex modulus)."""

import threading

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


def test_concurrent_calls_from_host_threads(cs, oracle_lib):
    cases = [wl.random_case(9300 + i, 2, 200 + 17 * i, 3, (64, 128, 64, 16)[i], (64, 64, 64, 32)[i]) for i in range(4)]
    born = wl.make_born_inputs(wl.HTRANSFORMER_ATTN.with_(batch=1, seqlen=150, nheads=2))
    dev = {i: {k: torch.from_numpy(np.ascontiguousarray(cases[i][k])).cuda() for k in KEYS} for i in range(4)}
    bdev = {k: torch.from_numpy(born[k]).cuda() for k in ("q", "k", "v")}
    torch.cuda.synchronize()
    out, errors = {}, []
    start = threading.Barrier(5)

    def forward(i):
        try:
            s = torch.cuda.Stream()
            start.wait()
            with torch.cuda.stream(s):
                y, h = cs.chunked_forward(**dev[i], chunk=64, precise=(i == 2), stream=s)
            s.synchronize()
            out[i] = (y.cpu().numpy(), h.cpu().numpy())
        except Exception as e:  # reported below
            errors.append(e)

    def attention():
        try:
            s = torch.cuda.Stream()
            start.wait()
            psi = cs.born_attention(bdev["q"], bdev["k"], bdev["v"], stream=s)
            s.synchronize()
            out["born"] = psi.cpu().numpy()
        except Exception as e:
            errors.append(e)

    threads = [threading.Thread(target=forward, args=(i,)) for i in range(4)] + [threading.Thread(target=attention)]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=120)
    assert not errors, errors
    for i in range(4):
        y_ref, h_ref = oracle_lib.cssd_naive(**cases[i])
        assert rel_err(out[i][0], y_ref) < TOL and rel_err(out[i][1], h_ref) < TOL, i
    psi_ref = oracle_lib.born_attention(born["q"], born["k"], born["v"], born["tau"])
    assert rel_err(out["born"], psi_ref) < TOL
    assert cs.device_status() == 0
