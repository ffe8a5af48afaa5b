"""The C ABI library on the host: it loads, exports every declared symbol, and
rejects bad arguments before touching CUDA (no GPU needed, nothing launched)."""

import ctypes
import os
import re

import pytest

from complex_valued_state_gb300 import build as cbuild
from complex_valued_state_gb300 import cssd

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "cssd.h")


@pytest.fixture(scope="module")
def lib():
    cbuild.build()
    return cssd.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(cssd_\w+)\s*\(", text, flags=re.M)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert set(cssd.EXPORTS) <= set(names)
    for n in names:
        assert hasattr(lib, n), n
        assert ctypes.cast(getattr(lib, n), ctypes.c_void_p).value


def test_status_strings(lib):
    for code in cssd.STATUS:
        s = cssd.status_string(code)
        assert isinstance(s, str) and s and s != "unknown status"
    assert cssd.status_string(12345) == "unknown status"


def test_workspace_bytes(lib):
    # tensor-core path (headdim 64, dstate 64 or 128): two slots of tagged
    # 8-byte hand-off words per sequence and 64-row state half, plus per-chunk phases
    got = cssd.workspace_bytes(4, 2048, 24, 64, 64, 64)
    assert got >= 4 * 24 * 2 * 2 * 64 * 64 * 8 + 4 * 24 * 32 * 4
    assert cssd.workspace_bytes(1, 65536, 32, 128, 64, 128) >= 32 * 2 * 2 * 2 * 64 * 64 * 8 + 32 * 1024 * 4
    # CUDA-core path: every chunk's end state plus per-chunk decay totals
    got = cssd.workspace_bytes(1, 4096, 8, 32, 32, 128)
    assert got >= 8 * 32 * 32 * 32 * 8
    # tensor cores: one prep launch up to 64 chunks of 64 tokens, two beyond, then the chunk kernel
    assert cssd.forward_launches(4, 2048, 24, 64, 64, 64) == 2
    assert cssd.forward_launches(4, 4096, 24, 64, 64, 64) == 2
    assert cssd.forward_launches(4, 4097, 24, 64, 64, 64) == 3
    assert cssd.forward_launches(1, 65536, 32, 128, 64, 128) == 3
    assert cssd.forward_launches(1, 4096, 8, 32, 32, 128) == 2  # padded to the tensor-core tile
    assert cssd.forward_launches(1, 4096, 8, 128, 32, 128) == 3  # CUDA-core kernels
    assert cssd.workspace_bytes(1, 65, 1, 16, 16, 64) > cssd.workspace_bytes(1, 64, 1, 16, 16, 64)
    assert cssd.workspace_bytes(1, 64, 1, 16, 16, 96) == 0  # unsupported chunk
    assert cssd.workspace_bytes(1, 0, 1, 16, 16, 64) == 0  # empty sequence
    assert cssd.workspace_bytes(1, 64, 1, 48, 16, 64) == 0  # unsupported N
    # split precision: the forward's workspace, except at dstate 128 (the
    # CUDA-core kernels keep every chunk's state)
    assert cssd.precise_workspace_bytes(4, 2048, 24, 64, 64, 64) == cssd.workspace_bytes(4, 2048, 24, 64, 64, 64)
    assert cssd.precise_workspace_bytes(1, 4096, 8, 32, 32, 128) == cssd.workspace_bytes(1, 4096, 8, 32, 32, 128)
    assert cssd.precise_workspace_bytes(1, 8192, 32, 128, 64, 128) >= 32 * 64 * 128 * 64 * 8
    assert cssd.precise_workspace_bytes(1, 64, 1, 48, 16, 64) == 0


def _fwd(lib, dims, ptrs=None, chunk=64, ws=None, ws_bytes=0):
    p = ptrs or {}
    args = [p.get(k, 0x10000 + 0x100 * i) for i, k in enumerate(("x", "dt", "A", "B", "C", "D", "y", "h"))]
    d = None if dims is None else ctypes.byref(cssd.Dims(*dims))
    return lib.cssd_chunked_forward(d, *[ctypes.c_void_p(a) if a else None for a in args], chunk,
                                    ctypes.c_void_p(ws) if ws else None, ctypes.c_size_t(ws_bytes), None)


def _step(lib, dims, ptrs=None):
    p = ptrs or {}
    args = [p.get(k, 0x10000 + 0x100 * i) for i, k in enumerate(("h", "x", "dt", "A", "B", "C", "D", "y"))]
    d = None if dims is None else ctypes.byref(cssd.Dims(*dims))
    return lib.cssd_step(d, *[ctypes.c_void_p(a) if a else None for a in args], None)


def test_argument_errors_are_caught_on_the_host(lib):
    ok = (1, 64, 1, 16, 16)
    assert _fwd(lib, None) == -1
    assert _fwd(lib, (0, 64, 1, 16, 16)) == -2
    assert _fwd(lib, (1, 0, 1, 16, 16)) == -2
    assert _fwd(lib, (1, 64, -3, 16, 16)) == -2
    assert _fwd(lib, (1, 64, 1, 24, 16)) == -3
    assert _fwd(lib, (1, 64, 1, 16, 128)) == -3
    assert _fwd(lib, ok, chunk=32) == -3
    assert _fwd(lib, ok, {"x": 0}) == -1
    assert _fwd(lib, ok, {"D": 0}) == -1
    assert _fwd(lib, ok, {"x": 0x10008}) == -4  # complex64 arrays want 16-byte alignment
    assert _fwd(lib, ok, {"dt": 0x10102}) == -4
    assert _fwd(lib, ok, ws=0x900000, ws_bytes=16) == -5
    assert _fwd(lib, (70000, 64, 1, 16, 16)) == -2  # beyond the grid limit
    assert _fwd(lib, (60000, 64 * 60000, 1, 16, 16)) == -2  # (batch, head, tile) count beyond 32 bits
    assert _step(lib, None) == -1
    assert _step(lib, (1, 1, 1, 16, 16), {"h": 0}) == -1
    assert _step(lib, (1, 1, 1, 16, 8)) == -3
    assert _step(lib, (1, 1, 1, 16, 16), {"y": 0x10004}) == -4


def test_constant_input_argument_errors(lib):
    ok = cssd.Dims(1, 1, 1, 16, 16)
    args = [ctypes.c_void_p(0x10000 + 0x100 * i) for i in range(8)]  # h, x, dt, A, B, C, D, y
    h, x, dt, A, B, C, D, y = args
    assert lib.cssd_step_n(ctypes.byref(ok), h, x, dt, A, B, C, D, -1, y, None) == -2
    assert lib.cssd_step_n(None, h, x, dt, A, B, C, D, 5, y, None) == -1
    assert lib.cssd_step_n(ctypes.byref(ok), None, x, dt, A, B, C, D, 5, y, None) == -1
    assert lib.cssd_step_n(ctypes.byref(ok), ctypes.c_void_p(0x10008), x, dt, A, B, C, D, 5, y, None) == -4
    assert lib.cssd_step_n(ctypes.byref(cssd.Dims(1, 1, 1, 24, 16)), h, x, dt, A, B, C, D, 5, y, None) == -3
    assert lib.cssd_step_infinite(ctypes.byref(ok), x, dt, A, B, C, D, None, None) == -1
    assert lib.cssd_step_infinite(ctypes.byref(ok), x, dt, A, ctypes.c_void_p(0x10404), C, D, y, None) == -4
    assert lib.cssd_step_infinite(ctypes.byref(cssd.Dims(0, 1, 1, 16, 16)), x, dt, A, B, C, D, y, None) == -2


def test_cayley_scan_argument_errors(lib):
    ok = cssd.Dims(1, 8, 2, 16, 0)
    p = [ctypes.c_void_p(0x10000 + 0x100 * i) for i in range(7)]  # phi, u, b, C, psi0, y, psi_final
    f = lib.cssd_cayley_scan
    assert f(None, *p, 64, ctypes.c_float(-30.0), None) == -1
    assert f(ctypes.byref(cssd.Dims(1, 0, 2, 16, 0)), *p, 64, ctypes.c_float(-30.0), None) == -2
    assert f(ctypes.byref(ok), *p, 0, ctypes.c_float(-30.0), None) == -2  # chunk
    assert f(ctypes.byref(ok), *p, 64, ctypes.c_float(1.0), None) == -2  # clamp above 0
    assert f(ctypes.byref(ok), *p, 64, ctypes.c_float(-100.0), None) == -2  # e^100 would overflow
    assert f(ctypes.byref(ok), *p, 64, ctypes.c_float(float("nan")), None) == -2
    q = list(p)
    q[0] = None
    assert f(ctypes.byref(ok), *q, 64, ctypes.c_float(-30.0), None) == -1
    q = list(p)
    q[2] = ctypes.c_void_p(0x10204)  # complex64 wants 8-byte alignment
    assert f(ctypes.byref(ok), *q, 64, ctypes.c_float(float("-inf")), None) == -4


def test_backward_argument_errors(lib):
    ok = cssd.Dims(1, 8, 2, 64, 64)
    p = [ctypes.c_void_p(0x10000 + 0x100 * i) for i in range(14)]  # x dt A B C D dy gx gdt gA gB gC gD ws
    f = lib.cssd_chunked_backward
    assert f(None, *p[:13], 64, p[13], 1 << 40, None) == -1
    assert f(ctypes.byref(cssd.Dims(1, 8, 2, 48, 64)), *p[:13], 64, p[13], 1 << 40, None) == -3
    assert f(ctypes.byref(cssd.Dims(1, 8, 2, 64, 128)), *p[:13], 64, p[13], 1 << 40, None) == -3
    assert f(ctypes.byref(ok), *p[:13], 32, p[13], 1 << 40, None) == -3  # chunk
    q = list(p)
    q[6] = None  # dy
    assert f(ctypes.byref(ok), *q[:13], 64, q[13], 1 << 40, None) == -1
    q = list(p)
    q[7] = ctypes.c_void_p(0x10708)  # gx 8-byte aligned only
    assert f(ctypes.byref(ok), *q[:13], 64, q[13], 1 << 40, None) == -4
    assert f(ctypes.byref(ok), *p[:13], 64, p[13], 16, None) == -5  # workspace too small
    assert lib.cssd_backward_workspace_bytes(ctypes.byref(ok), 64) > 0
    assert lib.cssd_backward_workspace_bytes(ctypes.byref(cssd.Dims(1, 8, 2, 128, 64)), 64) > 0  # dstate 128
    assert lib.cssd_backward_workspace_bytes(ctypes.byref(cssd.Dims(1, 8, 2, 64, 128)), 64) == 0  # headdim 128


def test_born_attention_argument_errors(lib):
    ok = cssd.Dims(1, 8, 2, 16, 0)
    p = [ctypes.c_void_p(0x10000 + 0x100 * i) for i in range(4)]  # q, k, v, psi
    f = lib.cssd_born_attention
    assert f(None, *p, None) == -1
    assert f(ctypes.byref(cssd.Dims(1, 0, 2, 16, 0)), *p, None) == -2
    assert f(ctypes.byref(cssd.Dims(1, 8, 2, 24, 0)), *p, None) == -3  # width not 16 or 32
    q = list(p)
    q[3] = None
    assert f(ctypes.byref(ok), *q, None) == -1
    q = list(p)
    q[1] = ctypes.c_void_p(0x10108)  # 8-byte aligned only
    assert f(ctypes.byref(ok), *q, None) == -4


def test_initial_state_and_host_forward_argument_errors(lib):
    ok = cssd.Dims(1, 64, 1, 16, 16)
    p = [ctypes.c_void_p(0x10000 + 0x100 * i) for i in range(9)]  # x dt A B C D h0 y h_final
    f = lib.cssd_chunked_forward_h0
    assert f(None, *p, 64, None, 0, None) == -1
    assert f(ctypes.byref(cssd.Dims(1, 64, 1, 24, 16)), *p, 64, None, 0, None) == -3
    q = list(p)
    q[6] = ctypes.c_void_p(0x10608)  # h0 is complex64 state: 16-byte alignment
    assert f(ctypes.byref(ok), *q, 64, None, 0, None) == -4
    q = list(p)
    q[7] = None  # y
    assert f(ctypes.byref(ok), *q, 64, None, 0, None) == -1
    assert f(ctypes.byref(ok), *p, 64, ctypes.c_void_p(0x900000), 16, None) == -5
    f = lib.cssd_chunked_forward_tf32  # same arguments and checks as the h0 forward
    assert f(None, *p, 64, None, 0, None) == -1
    assert f(ctypes.byref(ok), *p, 128 + 1, None, 0, None) == -3
    assert f(ctypes.byref(cssd.Dims(1, 64, 1, 24, 16)), *p, 64, None, 0, None) == -3
    q = list(p)
    q[3] = ctypes.c_void_p(0x10308)  # B: 16-byte alignment
    assert f(ctypes.byref(ok), *q, 64, None, 0, None) == -4
    assert f(ctypes.byref(ok), *p, 64, ctypes.c_void_p(0x900000), 16, None) == -5
    f = lib.cssd_chunked_forward_precise  # same arguments and checks
    assert f(None, *p, 64, None, 0, None) == -1
    assert f(ctypes.byref(ok), *p, 128 + 1, None, 0, None) == -3
    # dstate 128 with headdim 64 is accepted (the fp32 CUDA-core kernels): the
    # call gets as far as the workspace check
    assert f(ctypes.byref(cssd.Dims(1, 64, 1, 128, 64)), *p, 64, ctypes.c_void_p(0x900000), 16, None) == -5
    q = list(p)
    q[6] = ctypes.c_void_p(0x10604)
    assert f(ctypes.byref(ok), *q, 64, None, 0, None) == -4
    assert f(ctypes.byref(ok), *p, 64, ctypes.c_void_p(0x900000), 16, None) == -5

    g = lib.cssd_chunked_forward_host
    assert g(None, *p, 64, 0, None, 0, None) == -1
    assert g(ctypes.byref(cssd.Dims(1, 0, 1, 16, 16)), *p, 64, 0, None, 0, None) == -2
    assert g(ctypes.byref(ok), *p, 64, -1, None, 0, None) == -2  # piece length
    assert g(ctypes.byref(ok), *p, 96, 0, None, 0, None) == -3  # chunk
    assert g(ctypes.byref(cssd.Dims(1, 64, 1, 16, 8)), *p, 64, 0, None, 0, None) == -3
    q = list(p)
    q[0] = None
    assert g(ctypes.byref(ok), *q, 64, 0, None, 0, None) == -1
    assert g(ctypes.byref(ok), *p, 64, 0, ctypes.c_void_p(0x900010), 1 << 30, None) == -4  # buffer alignment
    assert g(ctypes.byref(ok), *p, 64, 0, ctypes.c_void_p(0x900000), 16, None) == -5  # buffer size

    # device bytes: two slots of one piece's x, dt, B, C, y plus two states and the piece's workspace
    m = cssd.Dims(4, 2048, 24, 64, 64)
    in_per_token = 4 * 24 * (8 * 64 + 4 + 16 * 64)  # x, dt, B, C
    piece = (48 << 20) // in_per_token // 64 * 64  # default: ~48 MB of inputs, whole chunks (320 tokens)
    auto = lib.cssd_host_forward_device_bytes(ctypes.byref(m), 64, 0)
    assert auto >= 2 * piece * (in_per_token + 4 * 24 * 8 * 64) + 2 * 4 * 24 * 64 * 64 * 8
    assert lib.cssd_host_forward_device_bytes(ctypes.byref(m), 64, piece) == auto
    assert lib.cssd_host_forward_device_bytes(ctypes.byref(m), 64, 128) < auto
    assert lib.cssd_host_forward_device_bytes(ctypes.byref(m), 64, 1 << 20) == \
        lib.cssd_host_forward_device_bytes(ctypes.byref(m), 64, 2048)  # a piece never exceeds the sequence
    assert lib.cssd_host_forward_device_bytes(ctypes.byref(m), 64, -1) == 0
    assert lib.cssd_host_forward_device_bytes(ctypes.byref(m), 96, 0) == 0


def test_device_status_argument_errors(lib):
    assert lib.cssd_device_status(None, 0, None) == -1


def test_selftest_argument_errors(lib):
    bits = ctypes.c_int(0)
    assert lib.cssd_selftest_handoff_timeout(1000, None, None) == -1
    assert lib.cssd_selftest_handoff_timeout(0, ctypes.byref(bits), None) == -2


def test_binding_rejects_wrong_dtypes_and_shapes():
    import torch

    x = torch.zeros((1, 8, 1, 16), dtype=torch.complex64)
    dt = torch.zeros((1, 8, 1))
    A = torch.zeros(1, dtype=torch.complex64)
    B = torch.zeros((1, 8, 1, 16), dtype=torch.complex64)
    D = torch.zeros(1)
    with pytest.raises(TypeError):
        cssd.chunked_forward(x, dt.double(), A, B, B, D)
    with pytest.raises(ValueError):
        cssd.chunked_forward(x, dt[:, :4], A, B, B, D)
    with pytest.raises(ValueError):
        cssd.chunked_forward(x, dt, A, B.transpose(1, 3), B, D)
