"""ctypes binding of libcssd (argument marshalling only).

Every function here takes torch tensors that already live on a CUDA device,
checks dtype / shape / contiguity, and passes raw pointers and sizes to the C
ABI declared in ``include/cssd.h``.  All arithmetic runs in the library's
kernels.  If ``libcssd.so`` is missing the first call raises: there is no CPU
fallback.
"""

from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libcssd.so")

CSSD_OK = 0
STATUS = {
    0: "CSSD_OK",
    -1: "CSSD_ERR_NULL",
    -2: "CSSD_ERR_DIMS",
    -3: "CSSD_ERR_UNSUPPORTED",
    -4: "CSSD_ERR_ALIGN",
    -5: "CSSD_ERR_WORKSPACE",
    -6: "CSSD_ERR_CUDA",
    -7: "CSSD_ERR_DEVICE",
}

# Every symbol include/cssd.h declares.
EXPORTS = ("cssd_workspace_bytes", "cssd_precise_workspace_bytes", "cssd_forward_launches", "cssd_chunked_forward", "cssd_chunked_forward_h0",
           "cssd_chunked_forward_precise", "cssd_chunked_forward_tf32",
           "cssd_host_forward_device_bytes", "cssd_chunked_forward_host",
           "cssd_backward_workspace_bytes", "cssd_chunked_backward",
           "cssd_chunked_forward_noalloc", "cssd_step", "cssd_step_n", "cssd_step_infinite", "cssd_cayley_scan", "cssd_born_attention",
           "cssd_profile_events", "cssd_device_status",
           "cssd_selftest_handoff_timeout", "cssd_status_string")

# Scratch array size of cssd_chunked_forward_noalloc (bytes).
NOALLOC_SCRATCH_BYTES = 16 << 20


class Dims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in ("batch", "seqlen", "nheads", "dstate", "headdim")]


class CssdError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)} ({status_string(status)})")


_lock = threading.Lock()
_lib = None


def load(path: str = LIB_PATH):
    """Load libcssd.so and declare its signatures (raises if it is not built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise RuntimeError(f"{path} is not built; run complex_valued_state_gb300.build.build() first")
            lib = ctypes.CDLL(path)
            vp, dims_p = ctypes.c_void_p, ctypes.POINTER(Dims)
            lib.cssd_workspace_bytes.argtypes = [dims_p, ctypes.c_int]
            lib.cssd_workspace_bytes.restype = ctypes.c_size_t
            lib.cssd_precise_workspace_bytes.argtypes = [dims_p, ctypes.c_int]
            lib.cssd_precise_workspace_bytes.restype = ctypes.c_size_t
            lib.cssd_forward_launches.argtypes = [dims_p, ctypes.c_int]
            lib.cssd_forward_launches.restype = ctypes.c_int
            lib.cssd_chunked_forward.argtypes = [dims_p] + [vp] * 8 + [ctypes.c_int, vp, ctypes.c_size_t, vp]
            lib.cssd_chunked_forward.restype = ctypes.c_int
            lib.cssd_chunked_forward_h0.argtypes = [dims_p] + [vp] * 9 + [ctypes.c_int, vp, ctypes.c_size_t, vp]
            lib.cssd_chunked_forward_h0.restype = ctypes.c_int
            lib.cssd_chunked_forward_precise.argtypes = [dims_p] + [vp] * 9 + [ctypes.c_int, vp, ctypes.c_size_t, vp]
            lib.cssd_chunked_forward_precise.restype = ctypes.c_int
            lib.cssd_chunked_forward_tf32.argtypes = [dims_p] + [vp] * 9 + [ctypes.c_int, vp, ctypes.c_size_t, vp]
            lib.cssd_chunked_forward_tf32.restype = ctypes.c_int
            lib.cssd_host_forward_device_bytes.argtypes = [dims_p, ctypes.c_int, ctypes.c_int64]
            lib.cssd_host_forward_device_bytes.restype = ctypes.c_size_t
            lib.cssd_chunked_forward_host.argtypes = [dims_p] + [vp] * 9 + [ctypes.c_int, ctypes.c_int64, vp,
                                                                           ctypes.c_size_t, vp]
            lib.cssd_chunked_forward_host.restype = ctypes.c_int
            lib.cssd_chunked_forward_noalloc.argtypes = [dims_p] + [vp] * 8 + [ctypes.c_int, vp]
            lib.cssd_chunked_forward_noalloc.restype = ctypes.c_int
            lib.cssd_step.argtypes = [dims_p] + [vp] * 8 + [vp]
            lib.cssd_step.restype = ctypes.c_int
            lib.cssd_step_n.argtypes = [dims_p] + [vp] * 7 + [ctypes.c_int64, vp, vp]
            lib.cssd_step_n.restype = ctypes.c_int
            lib.cssd_step_infinite.argtypes = [dims_p] + [vp] * 7 + [vp]
            lib.cssd_step_infinite.restype = ctypes.c_int
            lib.cssd_cayley_scan.argtypes = [dims_p] + [vp] * 7 + [ctypes.c_int, ctypes.c_float, vp]
            lib.cssd_cayley_scan.restype = ctypes.c_int
            lib.cssd_backward_workspace_bytes.argtypes = [dims_p, ctypes.c_int]
            lib.cssd_backward_workspace_bytes.restype = ctypes.c_size_t
            lib.cssd_chunked_backward.argtypes = [dims_p] + [vp] * 13 + [ctypes.c_int, vp, ctypes.c_size_t, vp]
            lib.cssd_chunked_backward.restype = ctypes.c_int
            lib.cssd_born_attention.argtypes = [dims_p] + [vp] * 4 + [vp]
            lib.cssd_born_attention.restype = ctypes.c_int
            lib.cssd_device_status.argtypes = [ctypes.POINTER(ctypes.c_uint), ctypes.c_int, vp]
            lib.cssd_device_status.restype = ctypes.c_int
            lib.cssd_profile_events.argtypes = [vp, vp]
            lib.cssd_profile_events.restype = ctypes.c_int
            lib.cssd_selftest_handoff_timeout.argtypes = [ctypes.c_longlong, ctypes.POINTER(ctypes.c_int), vp]
            lib.cssd_selftest_handoff_timeout.restype = ctypes.c_int
            lib.cssd_status_string.argtypes = [ctypes.c_int]
            lib.cssd_status_string.restype = ctypes.c_char_p
            _lib = lib
    return _lib


def status_string(status: int) -> str:
    return load().cssd_status_string(int(status)).decode()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check(t, name, dtype, shape, device):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.device != device:
        raise ValueError(f"{name} must be on {device}, got {t.device}")


def _stream_handle(stream, device):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


# Bits of the device status word (cssd_device_status).
STATUS_HANDOFF_TIMEOUT = 1
STATUS_CHUNK_MMA_TIMEOUT = 2
STATUS_BORN_MMA_TIMEOUT = 4


def device_status(clear: bool = False, device=None, stream=None) -> int:
    """The library's device status word (bits STATUS_*; 0 = no bounded wait has
    given up), read after the work already on `stream`; cleared when `clear`."""
    lib = load()
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    bits = ctypes.c_uint(0)
    st = lib.cssd_device_status(ctypes.byref(bits), 1 if clear else 0, _stream_handle(stream, dev))
    if st != CSSD_OK:
        raise CssdError(st, "cssd_device_status")
    return int(bits.value)


def profile_events(begin=None, end=None):
    """Record `begin` / `end` (torch.cuda.Event, created with enable_timing and
    recorded once so that they exist) around the dominant kernel of later
    forward calls from this thread; None, None = off."""

    def h(e):
        if e is None:
            return None
        if not e.cuda_event:
            raise ValueError("event not created yet: record it once first")
        return ctypes.c_void_p(e.cuda_event)

    st = load().cssd_profile_events(h(begin), h(end))
    if st != CSSD_OK:
        raise CssdError(st, "cssd_profile_events")


def selftest_handoff_timeout(wait_cycles: int = 2_000_000, stream=None) -> int:
    """Run the tensor-core forward kernels with a predecessor chunk that never
    publishes; return their error bits: the TF32 kernel's in bits 0-7, the
    dstate-64 half-operand kernel's in bits 8-15, the dstate-128 one's in bits
    16-23 (bit 0 of each set = the bounded hand-off wait gave up)."""
    import torch as _t

    bits = ctypes.c_int(-1)
    st = load().cssd_selftest_handoff_timeout(int(wait_cycles), ctypes.byref(bits),
                                              _stream_handle(stream, _t.device("cuda", _t.cuda.current_device())))
    if st != CSSD_OK:
        raise CssdError(st, "cssd_selftest_handoff_timeout")
    return int(bits.value)


def workspace_bytes(batch: int, seqlen: int, nheads: int, dstate: int, headdim: int, chunk: int) -> int:
    d = Dims(batch, seqlen, nheads, dstate, headdim)
    return int(load().cssd_workspace_bytes(ctypes.byref(d), int(chunk)))


def precise_workspace_bytes(batch: int, seqlen: int, nheads: int, dstate: int, headdim: int, chunk: int) -> int:
    d = Dims(batch, seqlen, nheads, dstate, headdim)
    return int(load().cssd_precise_workspace_bytes(ctypes.byref(d), int(chunk)))


def forward_launches(batch: int, seqlen: int, nheads: int, dstate: int, headdim: int, chunk: int) -> int:
    d = Dims(batch, seqlen, nheads, dstate, headdim)
    return int(load().cssd_forward_launches(ctypes.byref(d), int(chunk)))


def chunked_forward(x, dt, A, B, C, D, *, chunk: int = 64, y=None, h_final=None, want_state: bool = True,
                    workspace=None, stream=None, h0=None, precise: bool = False, tf32: bool = False):
    """cssd_chunked_forward (cssd_chunked_forward_h0 when `h0` is given,
    cssd_chunked_forward_precise when `precise`, cssd_chunked_forward_tf32 when
    `tf32`) on device tensors; returns (y, h_final or None).

    x complex64 [Bz,T,H,P]; dt float32 [Bz,T,H]; A complex64 [H];
    B, C complex64 [Bz,T,H,N]; D float32 [H]; h0 complex64 [Bz,H,N,P], the
    state before the first token (zero when None).  `workspace` is an optional
    uint8 device tensor of at least workspace_bytes(...) bytes
    (precise_workspace_bytes(...) with `precise`).
    """
    lib = load()
    dev = x.device
    Bz, T, H, P = x.shape
    N = B.shape[-1]
    c64, f32 = torch.complex64, torch.float32
    _check(x, "x", c64, (Bz, T, H, P), dev)
    _check(dt, "dt", f32, (Bz, T, H), dev)
    _check(A, "A", c64, (H,), dev)
    _check(B, "B", c64, (Bz, T, H, N), dev)
    _check(C, "C", c64, (Bz, T, H, N), dev)
    _check(D, "D", f32, (H,), dev)
    if y is None:
        y = torch.empty((Bz, T, H, P), dtype=c64, device=dev)
    _check(y, "y", c64, (Bz, T, H, P), dev)
    if h_final is None and want_state:
        h_final = torch.empty((Bz, H, N, P), dtype=c64, device=dev)
    if h_final is not None:
        _check(h_final, "h_final", c64, (Bz, H, N, P), dev)
    ws_bytes = 0
    if workspace is not None:
        if workspace.device != dev or not workspace.is_contiguous():
            raise ValueError("workspace must be a contiguous tensor on the inputs' device")
        ws_bytes = workspace.numel() * workspace.element_size()
    d = Dims(Bz, T, H, N, P)
    if precise and tf32:
        raise ValueError("precise and tf32 select different entry points; pass at most one")
    if precise or tf32:
        if h0 is not None:
            _check(h0, "h0", c64, (Bz, H, N, P), dev)
        name = "cssd_chunked_forward_precise" if precise else "cssd_chunked_forward_tf32"
        st = getattr(lib, name)(ctypes.byref(d), _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(h0),
                                _ptr(y), _ptr(h_final), int(chunk), _ptr(workspace), ctypes.c_size_t(ws_bytes),
                                _stream_handle(stream, dev))
        if st != CSSD_OK:
            raise CssdError(st, name)
        return y, h_final
    if h0 is None:
        st = lib.cssd_chunked_forward(ctypes.byref(d), _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
                                      _ptr(y), _ptr(h_final), int(chunk), _ptr(workspace),
                                      ctypes.c_size_t(ws_bytes), _stream_handle(stream, dev))
        if st != CSSD_OK:
            raise CssdError(st, "cssd_chunked_forward")
        return y, h_final
    _check(h0, "h0", c64, (Bz, H, N, P), dev)
    st = lib.cssd_chunked_forward_h0(ctypes.byref(d), _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
                                     _ptr(h0), _ptr(y), _ptr(h_final), int(chunk), _ptr(workspace),
                                     ctypes.c_size_t(ws_bytes), _stream_handle(stream, dev))
    if st != CSSD_OK:
        raise CssdError(st, "cssd_chunked_forward_h0")
    return y, h_final


def host_forward_device_bytes(batch: int, seqlen: int, nheads: int, dstate: int, headdim: int, chunk: int,
                              piece_len: int = 0) -> int:
    d = Dims(batch, seqlen, nheads, dstate, headdim)
    return int(load().cssd_host_forward_device_bytes(ctypes.byref(d), int(chunk), int(piece_len)))


def chunked_forward_host(x, dt, A, B, C, D, *, chunk: int = 64, piece_len: int = 0, y=None, h_final=None, h0=None,
                         want_state: bool = True, device_buffer=None, device=None, stream=None):
    """cssd_chunked_forward_host: the forward over host tensors (pin them for
    copies that overlap the compute), streamed through `device` (default: the
    current CUDA device) in pieces of `piece_len` tokens (0: library's choice).

    Shapes as chunked_forward.  y and h_final are host tensors (pinned when
    created here) unless passed in; h_final may also be a device tensor, h0
    a host or device tensor.  Returns (y, h_final); they are complete once
    `stream` (default: the device's current stream) has run past the call.
    """
    lib = load()
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    Bz, T, H, P = x.shape
    N = B.shape[-1]
    c64, f32 = torch.complex64, torch.float32

    def chk(t, name, dtype, shape):
        if not isinstance(t, torch.Tensor):
            raise TypeError(f"{name} must be a torch.Tensor")
        if t.dtype != dtype or tuple(t.shape) != tuple(shape) or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous {dtype} tensor of shape {tuple(shape)}")
        if t.device.type == "cuda" and t.device != dev:
            raise ValueError(f"{name} must be on the host or on {dev}")

    chk(x, "x", c64, (Bz, T, H, P))
    chk(dt, "dt", f32, (Bz, T, H))
    chk(A, "A", c64, (H,))
    chk(B, "B", c64, (Bz, T, H, N))
    chk(C, "C", c64, (Bz, T, H, N))
    chk(D, "D", f32, (H,))
    if y is None:
        y = torch.empty((Bz, T, H, P), dtype=c64, pin_memory=True)
    chk(y, "y", c64, (Bz, T, H, P))
    if h_final is None and want_state:
        h_final = torch.empty((Bz, H, N, P), dtype=c64, pin_memory=True)
    if h_final is not None:
        chk(h_final, "h_final", c64, (Bz, H, N, P))
    if h0 is not None:
        chk(h0, "h0", c64, (Bz, H, N, P))
    nbytes = 0
    if device_buffer is not None:
        if device_buffer.device != dev or not device_buffer.is_contiguous():
            raise ValueError("device_buffer must be a contiguous tensor on the device")
        nbytes = device_buffer.numel() * device_buffer.element_size()
    d = Dims(Bz, T, H, N, P)
    st = lib.cssd_chunked_forward_host(ctypes.byref(d), _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
                                       _ptr(h0), _ptr(y), _ptr(h_final), int(chunk), int(piece_len),
                                       _ptr(device_buffer), ctypes.c_size_t(nbytes), _stream_handle(stream, dev))
    if st != CSSD_OK:
        raise CssdError(st, "cssd_chunked_forward_host")
    return y, h_final


def backward_workspace_bytes(batch: int, seqlen: int, nheads: int, dstate: int, headdim: int, chunk: int) -> int:
    d = Dims(batch, seqlen, nheads, dstate, headdim)
    return int(load().cssd_backward_workspace_bytes(ctypes.byref(d), int(chunk)))


def chunked_backward(x, dt, A, B, C, D, dy, *, chunk: int = 64, grads=None, workspace=None, stream=None):
    """cssd_chunked_backward on device tensors; returns a dict gx, gdt, gA, gB,
    gC, gD (complex inputs: dL/dRe + i dL/dIm; real ones: dL/dw).

    Inputs as chunked_forward; dy complex64 [Bz,T,H,P] is the upstream
    gradient.  `grads` may hold preallocated outputs under the same keys.
    """
    lib = load()
    dev = x.device
    Bz, T, H, P = x.shape
    N = B.shape[-1]
    c64, f32 = torch.complex64, torch.float32
    _check(x, "x", c64, (Bz, T, H, P), dev)
    _check(dt, "dt", f32, (Bz, T, H), dev)
    _check(A, "A", c64, (H,), dev)
    _check(B, "B", c64, (Bz, T, H, N), dev)
    _check(C, "C", c64, (Bz, T, H, N), dev)
    _check(D, "D", f32, (H,), dev)
    _check(dy, "dy", c64, (Bz, T, H, P), dev)
    g = dict(grads or {})
    shapes = {"gx": ((Bz, T, H, P), c64), "gdt": ((Bz, T, H), f32), "gA": ((H,), c64), "gB": ((Bz, T, H, N), c64),
              "gC": ((Bz, T, H, N), c64), "gD": ((H,), f32)}
    for k, (shp, dtp) in shapes.items():
        if k not in g:
            g[k] = torch.empty(shp, dtype=dtp, device=dev)
        _check(g[k], k, dtp, shp, dev)
    ws_bytes = 0
    if workspace is not None:
        if workspace.device != dev or not workspace.is_contiguous():
            raise ValueError("workspace must be a contiguous tensor on the inputs' device")
        ws_bytes = workspace.numel() * workspace.element_size()
    d = Dims(Bz, T, H, N, P)
    st = lib.cssd_chunked_backward(ctypes.byref(d), _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(dy),
                                   _ptr(g["gx"]), _ptr(g["gdt"]), _ptr(g["gA"]), _ptr(g["gB"]), _ptr(g["gC"]),
                                   _ptr(g["gD"]), int(chunk), _ptr(workspace), ctypes.c_size_t(ws_bytes),
                                   _stream_handle(stream, dev))
    if st != CSSD_OK:
        raise CssdError(st, "cssd_chunked_backward")
    return g


def chunked_forward_noalloc(x, dt, A, B, C, D, *, chunk: int = 64, y=None, h_final=None, want_state: bool = True,
                            stream=None):
    """cssd_chunked_forward_noalloc: the forward on the library's fixed scratch
    array, for callers that cannot allocate device memory; returns (y, h_final).

    The outputs must be passed in (y, h_final) for the call itself to allocate
    nothing; when they are omitted this wrapper creates them with torch first.
    """
    lib = load()
    dev = x.device
    Bz, T, H, P = x.shape
    N = B.shape[-1]
    c64, f32 = torch.complex64, torch.float32
    _check(x, "x", c64, (Bz, T, H, P), dev)
    _check(dt, "dt", f32, (Bz, T, H), dev)
    _check(A, "A", c64, (H,), dev)
    _check(B, "B", c64, (Bz, T, H, N), dev)
    _check(C, "C", c64, (Bz, T, H, N), dev)
    _check(D, "D", f32, (H,), dev)
    if y is None:
        y = torch.empty((Bz, T, H, P), dtype=c64, device=dev)
    _check(y, "y", c64, (Bz, T, H, P), dev)
    if h_final is None and want_state:
        h_final = torch.empty((Bz, H, N, P), dtype=c64, device=dev)
    if h_final is not None:
        _check(h_final, "h_final", c64, (Bz, H, N, P), dev)
    d = Dims(Bz, T, H, N, P)
    st = lib.cssd_chunked_forward_noalloc(ctypes.byref(d), _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
                                          _ptr(y), _ptr(h_final), int(chunk), _stream_handle(stream, dev))
    if st != CSSD_OK:
        raise CssdError(st, "cssd_chunked_forward_noalloc")
    return y, h_final


def _check_step_inputs(dev, Bz, H, N, P, x, dt, A, B, C, D, y):
    c64, f32 = torch.complex64, torch.float32
    _check(x, "x", c64, (Bz, H, P), dev)
    _check(dt, "dt", f32, (Bz, H), dev)
    _check(A, "A", c64, (H,), dev)
    _check(B, "B", c64, (Bz, H, N), dev)
    _check(C, "C", c64, (Bz, H, N), dev)
    _check(D, "D", f32, (H,), dev)
    if y is None:
        y = torch.empty((Bz, H, P), dtype=c64, device=dev)
    _check(y, "y", c64, (Bz, H, P), dev)
    return y


def step(h, x, dt, A, B, C, D, *, y=None, stream=None):
    """cssd_step on device tensors: h updated in place; returns y.

    h complex64 [Bz,H,N,P]; x complex64 [Bz,H,P]; dt float32 [Bz,H];
    A complex64 [H]; B, C complex64 [Bz,H,N]; D float32 [H].
    """
    lib = load()
    dev = h.device
    Bz, H, N, P = h.shape
    _check(h, "h", torch.complex64, (Bz, H, N, P), dev)
    y = _check_step_inputs(dev, Bz, H, N, P, x, dt, A, B, C, D, y)
    d = Dims(Bz, 1, H, N, P)
    st = lib.cssd_step(ctypes.byref(d), _ptr(h), _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(y),
                       _stream_handle(stream, dev))
    if st != CSSD_OK:
        raise CssdError(st, "cssd_step")
    return y


def step_n(h, x, dt, A, B, C, D, nsteps, *, y=None, stream=None):
    """cssd_step_n: `nsteps` steps of the same token in closed form; h updated
    in place; returns the n-th step's y.  Shapes as in step()."""
    lib = load()
    dev = h.device
    Bz, H, N, P = h.shape
    _check(h, "h", torch.complex64, (Bz, H, N, P), dev)
    y = _check_step_inputs(dev, Bz, H, N, P, x, dt, A, B, C, D, y)
    d = Dims(Bz, 1, H, N, P)
    st = lib.cssd_step_n(ctypes.byref(d), _ptr(h), _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
                         ctypes.c_int64(int(nsteps)), _ptr(y), _stream_handle(stream, dev))
    if st != CSSD_OK:
        raise CssdError(st, "cssd_step_n")
    return y


def step_infinite(x, dt, A, B, C, D, *, y=None, stream=None):
    """cssd_step_infinite: the output of the same token held forever (no
    state); returns y [Bz,H,P].  Shapes as in step()."""
    lib = load()
    dev = x.device
    Bz, H, P = x.shape
    N = B.shape[-1]
    y = _check_step_inputs(dev, Bz, H, N, P, x, dt, A, B, C, D, y)
    d = Dims(Bz, 1, H, N, P)
    st = lib.cssd_step_infinite(ctypes.byref(d), _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(y),
                                _stream_handle(stream, dev))
    if st != CSSD_OK:
        raise CssdError(st, "cssd_step_infinite")
    return y


def cayley_scan(phi, u, b, C, *, psi0=None, chunk=64, log_clamp=-30.0, y=None, psi_final=None, stream=None):
    """cssd_cayley_scan on device tensors; returns (y, psi_final).

    phi, u float32 [Bz,T,H,N]; b, C complex64 [Bz,T,H,N]; psi0 complex64
    [Bz,H,N] or None.  log_clamp=-inf evaluates the recurrence exactly; a
    finite value (the paper's -30) runs the paper's clamped chunked scan.
    """
    lib = load()
    dev = phi.device
    Bz, T, H, N = phi.shape
    c64, f32 = torch.complex64, torch.float32
    _check(phi, "phi", f32, (Bz, T, H, N), dev)
    _check(u, "u", f32, (Bz, T, H, N), dev)
    _check(b, "b", c64, (Bz, T, H, N), dev)
    _check(C, "C", c64, (Bz, T, H, N), dev)
    if psi0 is not None:
        _check(psi0, "psi0", c64, (Bz, H, N), dev)
    if y is None:
        y = torch.empty((Bz, T, H, N), dtype=c64, device=dev)
    _check(y, "y", c64, (Bz, T, H, N), dev)
    if psi_final is None:
        psi_final = torch.empty((Bz, H, N), dtype=c64, device=dev)
    _check(psi_final, "psi_final", c64, (Bz, H, N), dev)
    d = Dims(Bz, T, H, N, 0)
    st = lib.cssd_cayley_scan(ctypes.byref(d), _ptr(phi), _ptr(u), _ptr(b), _ptr(C), _ptr(psi0), _ptr(y),
                              _ptr(psi_final), int(chunk), ctypes.c_float(float(log_clamp)),
                              _stream_handle(stream, dev))
    if st != CSSD_OK:
        raise CssdError(st, "cssd_cayley_scan")
    return y, psi_final


def born_attention(q, k, v, *, psi=None, stream=None):
    """cssd_born_attention on device tensors; returns psi.

    q, k, v complex64 [Bz,T,H,D] (D = 16 or 32).  The temperature of the
    scores cancels in the normalisation and is not an argument.
    """
    lib = load()
    dev = q.device
    Bz, T, H, D = q.shape
    c64 = torch.complex64
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check(t, n, c64, (Bz, T, H, D), dev)
    if psi is None:
        psi = torch.empty((Bz, T, H, D), dtype=c64, device=dev)
    _check(psi, "psi", c64, (Bz, T, H, D), dev)
    d = Dims(Bz, T, H, D, 0)
    st = lib.cssd_born_attention(ctypes.byref(d), _ptr(q), _ptr(k), _ptr(v), _ptr(psi), _stream_handle(stream, dev))
    if st != CSSD_OK:
        raise CssdError(st, "cssd_born_attention")
    return psi
