"""CPU oracle for the complex SSD — TEST INFRASTRUCTURE ONLY.

Plain double-precision C (``cssd_oracle.c``) behind a ctypes wrapper.  Only the
tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may
import this package; the CUDA library and its Python binding never do.

Inputs are the float32 / complex64 arrays of ``complex_valued_state_gb300.workloads``
(promoted exactly to double here); outputs are complex128 / float64.

Pins: every function here is checked in ``tests/test_oracle.py`` against
results fixed independently of this code (closed forms, brute-force sums,
special cases and the numbers the pages print).
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRCS = [os.path.join(_HERE, "cssd_oracle.c"), os.path.join(_HERE, "cayley_oracle.c"),
         os.path.join(_HERE, "born_oracle.c"), os.path.join(_HERE, "backward_oracle.c")]
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP over independent (batch, head) pairs)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < max(os.path.getmtime(f) for f in _SRCS):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fcx-limited-range", "-fPIC", "-shared", "-fopenmp",
               *_SRCS, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            i64, dp = ctypes.c_int64, ctypes.c_void_p
            lib.oracle_threads.restype = ctypes.c_int
            lib.oracle_cssd_naive.argtypes = [i64] * 5 + [dp] * 9
            lib.oracle_cssd_step.argtypes = [i64] * 4 + [dp] * 8
            lib.oracle_cssd_chunked.argtypes = [i64] * 6 + [dp] * 8
            lib.oracle_geom_closed_form.argtypes = [i64] * 5 + [dp] * 10
            lib.oracle_cayley_coefficients.argtypes = [i64] + [dp] * 3
            lib.oracle_cayley_recurrence.argtypes = [i64] * 4 + [dp] * 7
            lib.oracle_cayley_chunked.argtypes = [i64] * 5 + [ctypes.c_double] + [dp] * 7
            lib.oracle_born_attention.argtypes = [i64] * 4 + [dp] * 5
            lib.oracle_cssd_backward.argtypes = [i64] * 5 + [dp] * 13
            lib.oracle_born_attention_feature_map.argtypes = [i64] * 4 + [dp] * 4
            for f in (lib.oracle_cssd_naive, lib.oracle_cssd_step, lib.oracle_cssd_chunked,
                      lib.oracle_geom_closed_form, lib.oracle_cayley_coefficients, lib.oracle_cayley_recurrence,
                      lib.oracle_cayley_chunked, lib.oracle_born_attention, lib.oracle_born_attention_feature_map,
                      lib.oracle_cssd_backward):
                f.restype = None
            _lib = lib
    return _lib


def _c(a):
    return np.ascontiguousarray(a, dtype=np.complex128)


def _r(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def _p(a):
    return None if a is None else a.ctypes.data


def threads() -> int:
    """OpenMP threads the oracle uses (OMP_NUM_THREADS, else all cores)."""
    return int(_load().oracle_threads())


def cssd_naive(x, dt, A, B, C, D, h0=None, want_state=True):
    """Sequential recurrence; returns (y [Bz,T,H,P], h_final [Bz,H,N,P])."""
    lib = _load()
    x, dt, A, B, C, D = _c(x), _r(dt), _c(A), _c(B), _c(C), _r(D)
    Bz, T, H, P = x.shape
    N = B.shape[-1]
    h0 = None if h0 is None else _c(h0)
    y = np.empty((Bz, T, H, P), np.complex128)
    hf = np.empty((Bz, H, N, P), np.complex128) if want_state else None
    lib.oracle_cssd_naive(Bz, T, H, N, P, _p(x), _p(dt), _p(A), _p(B), _p(C), _p(D), _p(h0),
                          _p(y), _p(hf))
    return y, hf


def cssd_step(h, x, dt, A, B, C, D):
    """One decode token; returns (h_new [Bz,H,N,P], y [Bz,H,P])."""
    lib = _load()
    h = _c(h).copy()
    x, dt, A, B, C, D = _c(x), _r(dt), _c(A), _c(B), _c(C), _r(D)
    Bz, H, N, P = h.shape
    y = np.empty((Bz, H, P), np.complex128)
    lib.oracle_cssd_step(Bz, H, N, P, _p(h), _p(x), _p(dt), _p(A), _p(B), _p(C), _p(D), _p(y))
    return h, y


def cssd_chunked(x, dt, A, B, C, D, chunk: int):
    """Chunkwise decomposition (theorem form); returns (y, h_final)."""
    lib = _load()
    x, dt, A, B, C, D = _c(x), _r(dt), _c(A), _c(B), _c(C), _r(D)
    Bz, T, H, P = x.shape
    N = B.shape[-1]
    y = np.empty((Bz, T, H, P), np.complex128)
    hf = np.empty((Bz, H, N, P), np.complex128)
    lib.oracle_cssd_chunked(Bz, T, H, N, P, int(chunk), _p(x), _p(dt), _p(A), _p(B), _p(C), _p(D),
                            _p(y), _p(hf))
    return y, hf


def geom_closed_form(h0, x, dt, A, B, C, D, nsteps: int):
    """Constant input held for `nsteps` decode steps from h0, in closed form.

    Returns (h_n [Bz,H,N,P], y_n [Bz,H,P], y_inf [Bz,H,P])."""
    lib = _load()
    h0 = _c(h0)
    x, dt, A, B, C, D = _c(x), _r(dt), _c(A), _c(B), _c(C), _r(D)
    Bz, H, N, P = h0.shape
    hn = np.empty_like(h0)
    yn = np.empty((Bz, H, P), np.complex128)
    yinf = np.empty((Bz, H, P), np.complex128)
    lib.oracle_geom_closed_form(Bz, H, N, P, int(nsteps), _p(h0), _p(x), _p(dt), _p(A), _p(B), _p(C),
                                _p(D), _p(hn), _p(yn), _p(yinf))
    return hn, yn, yinf


# ---- per-coordinate Cayley-phase recurrence ("Complex Phase-State Dynamics
# Reduce the Optimization Steps of Sequence Models", sections 5.2-5.5 and
# Appendix A, Algorithms 1-2)

def cayley_coefficients(phi, u):
    """Algorithm 1: a = sigmoid(u) (1 + i phi) / (1 - i phi), elementwise."""
    lib = _load()
    phi, u = _r(phi), _r(u)
    a = np.empty(phi.shape, np.complex128)
    lib.oracle_cayley_coefficients(phi.size, _p(phi), _p(u), _p(a))
    return a


def cayley_recurrence(phi, u, b, C, psi0=None):
    """Equation (2) step by step; returns (y [Bz,T,H,N], psi_final [Bz,H,N])."""
    lib = _load()
    phi, u, b, C = _r(phi), _r(u), _c(b), _c(C)
    Bz, T, H, N = phi.shape
    p0 = None if psi0 is None else _c(psi0)
    y = np.empty((Bz, T, H, N), np.complex128)
    pf = np.empty((Bz, H, N), np.complex128)
    lib.oracle_cayley_recurrence(Bz, T, H, N, _p(phi), _p(u), _p(b), _p(C), None if p0 is None else _p(p0),
                                 _p(y), _p(pf))
    return y, pf


def cayley_chunked(phi, u, b, C, chunk: int, log_clamp: float = -30.0, psi0=None):
    """Algorithm 2 (chunked polar scan, cumulative log-gate clamped to
    [log_clamp, 0]); returns (y, psi_final)."""
    lib = _load()
    phi, u, b, C = _r(phi), _r(u), _c(b), _c(C)
    Bz, T, H, N = phi.shape
    p0 = None if psi0 is None else _c(psi0)
    y = np.empty((Bz, T, H, N), np.complex128)
    pf = np.empty((Bz, H, N), np.complex128)
    lib.oracle_cayley_chunked(Bz, T, H, N, int(chunk), float(log_clamp), _p(phi), _p(u), _p(b), _p(C),
                              None if p0 is None else _p(p0), _p(y), _p(pf))
    return y, pf


def born_attention(q, k, v, tau):
    """Causal Born attention, Algorithm 3 step by step: q, k, v [Bz,T,H,D]
    complex, tau [Bz,T,H] real; returns psi [Bz,T,H,D] (0 where a row's
    scores are all zero)."""
    lib = _load()
    q, k, v, tau = _c(q), _c(k), _c(v), _r(tau)
    Bz, T, H, D = q.shape
    psi = np.empty((Bz, T, H, D), np.complex128)
    lib.oracle_born_attention(Bz, T, H, D, _p(q), _p(k), _p(v), _p(tau), _p(psi))
    return psi


def born_attention_feature_map(q, k, v):
    """The same quantity through the recurrent feature-map form
    (|<q|k>|^2 = q^H k k^H q, carried as D x D matrices); used only to pin
    born_attention.  O(T D^4) per head: small cases only."""
    lib = _load()
    q, k, v = _c(q), _c(k), _c(v)
    Bz, T, H, D = q.shape
    psi = np.empty((Bz, T, H, D), np.complex128)
    lib.oracle_born_attention_feature_map(Bz, T, H, D, _p(q), _p(k), _p(v), _p(psi))
    return psi


def cssd_backward(x, dt, A, B, C, D, dy):
    """Gradients of the forward with respect to every input, given the
    upstream gradient dy [Bz,T,H,P] (complex): returns a dict gx, gdt, gA, gB,
    gC, gD (complex inputs get dL/dRe + i dL/dIm, real ones dL/dw).  Keeps
    every forward state: small cases only."""
    lib = _load()
    x, dt, A, B, C, D, dy = _c(x), _r(dt), _c(A), _c(B), _c(C), _r(D), _c(dy)
    Bz, T, H, P = x.shape
    N = B.shape[-1]
    g = dict(gx=np.empty_like(x), gdt=np.empty_like(dt), gA=np.empty_like(A), gB=np.empty_like(B),
             gC=np.empty_like(C), gD=np.empty_like(D))
    lib.oracle_cssd_backward(Bz, T, H, N, P, _p(x), _p(dt), _p(A), _p(B), _p(C), _p(D), _p(dy),
                             _p(g["gx"]), _p(g["gdt"]), _p(g["gA"]), _p(g["gB"]), _p(g["gC"]), _p(g["gD"]))
    return g
