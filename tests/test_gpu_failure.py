"""Failure detection on the GPU without a fault: the forward's hand-off wait
is bounded; when a predecessor never publishes, the kernel gives up, records
an error bit that the host reads, and the device stays usable."""

import numpy as np
import pytest
import torch

from complex_valued_state_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cs():
    from complex_valued_state_gb300 import build as cbuild
    from complex_valued_state_gb300 import cssd

    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for gpu tests")
    cbuild.build()
    cssd.load()
    return cssd


def test_handoff_wait_gives_up_and_device_stays_usable(cs, oracle_lib):
    cs.device_status(clear=True)
    bits = cs.selftest_handoff_timeout(wait_cycles=2_000_000)  # about a millisecond
    # in all three kernels the hand-off timed out and every tensor-core wait completed
    assert bits == 1 | (1 << 8) | (1 << 16), hex(bits)
    # the library's status word reports it to any caller, and clears on request
    assert cs.device_status() == cs.STATUS_HANDOFF_TIMEOUT
    assert cs.device_status(clear=True) == cs.STATUS_HANDOFF_TIMEOUT
    assert cs.device_status() == 0
    # the same context still computes correct results
    d = wl.random_case(3, 1, 200, 2, 64, 64)
    g = {k: torch.from_numpy(d[k]).cuda() for k in ("x", "dt", "A", "B", "C", "D")}
    y, h = cs.chunked_forward(**g, chunk=64)
    torch.cuda.synchronize()
    y_ref, h_ref = oracle_lib.cssd_naive(**d)
    err = np.max(np.abs(y.cpu().numpy() - y_ref)) / np.max(np.abs(y_ref))
    assert err < 2e-3


def test_status_word_stays_clear_on_normal_work(cs):
    cs.device_status(clear=True)
    d = wl.random_case(4, 2, 300, 3, 64, 64)
    g = {k: torch.from_numpy(d[k]).cuda() for k in ("x", "dt", "A", "B", "C", "D")}
    cs.chunked_forward(**g, chunk=64)
    cs.chunked_forward(**g, chunk=64, precise=True)
    dy = torch.from_numpy(wl.random_case(5, 2, 300, 3, 64, 64)["x"]).cuda()
    cs.chunked_backward(**g, dy=dy, chunk=64)
    bi = wl.make_born_inputs(wl.HTRANSFORMER_ATTN.with_(batch=1, seqlen=200, nheads=2))
    cs.born_attention(*(torch.from_numpy(bi[k]).cuda() for k in ("q", "k", "v")))
    assert cs.device_status() == 0
