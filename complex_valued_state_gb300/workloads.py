"""Seeded synthetic inputs for the complex SSD forward and decode step.

This module only draws random numbers and lays them out; it holds none of the
recurrence's arithmetic, so both the CUDA path and the CPU oracle can consume
its arrays without sharing any computation.

Shapes (all row-major, complex64 interleaved as [re, im]):
    x   [Bz, T, H, P]   complex64   token content
    dt  [Bz, T, H]      float32     raw step, discretised later as softplus(dt)
    A   [H]             complex64   per-head continuous-time rate
    B   [Bz, T, H, N]   complex64   input coupling
    C   [Bz, T, H, N]   complex64   readout
    D   [H]             float32     skip
    h   [Bz, H, N, P]   complex64   decode state (decode workload only)

Distributions follow the workloads of the pages: complex Gaussians with
re, im ~ N(0, 1/2); B and C scaled by 1/sqrt(N); dt ~ N(-1, 0.5) (0.5 read as
the standard deviation); A = -exp(U[ln 0.5, ln 4]) + i U[-pi, pi]; D ~ N(0, 1).
Draw order: x, B, C, dt, A_re, A_im, D, then h.  numpy's PCG64 generator is
used, so a seed gives the same arrays on every machine.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

# softplus(-1), the step at the mean of dt, used only to place the long-sequence
# decay rates: ln(1 + e^-1).
_SOFTPLUS_MINUS_ONE = math.log1p(math.exp(-1.0))


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    seqlen: int
    nheads: int
    dstate: int  # N
    headdim: int  # P
    chunk: int
    seed: int
    kind: str = "gaussian"  # gaussian | slow_decay | pam | decode
    steps: int = 0  # decode workloads: consecutive single-token calls
    note: str = field(default="", compare=False)

    @property
    def units(self) -> int:
        """Token-heads processed by one forward pass (Bz * T * H)."""
        return self.batch * self.seqlen * self.nheads

    def with_(self, **kw) -> "Workload":
        d = dict(self.__dict__)
        d.update(kw)
        return Workload(**d)


TINY = Workload("tiny", 1, 256, 1, 16, 16, 64, seed=0)
MAMBA2_LAYER = Workload("mamba2_layer", 4, 2048, 24, 64, 64, 64, seed=1)
LONG_SEQ = Workload("long_seq", 1, 65536, 32, 128, 64, 128, seed=2, kind="slow_decay")
PAM = Workload("pam", 8, 1024, 12, 64, 64, 64, seed=3, kind="pam")
DECODE = Workload("decode", 256, 1, 32, 128, 64, 64, seed=4, kind="decode", steps=1000)
# Per-coordinate Cayley-phase scan at the H-Mamba shapes (16 heads of 16 complex
# coordinates, 1024-token sequences, chunk 64) and its per-accelerator training
# batch of 256 sequences; headdim is unused by this recurrence.
HMAMBA_SCAN = Workload("hmamba_scan", 256, 1024, 16, 16, 16, 64, seed=5, kind="cayley")
# Causal Born attention at the H-Transformer shapes (16 heads of width D = N = 16,
# 1024-token sequences) and the same per-accelerator batch of 256 sequences;
# dstate holds the head width D, headdim and chunk are unused.
HTRANSFORMER_ATTN = Workload("htransformer_attn", 256, 1024, 16, 16, 16, 64, seed=6, kind="born")

WORKLOADS = {w.name: w for w in (TINY, MAMBA2_LAYER, LONG_SEQ, PAM, DECODE, HMAMBA_SCAN, HTRANSFORMER_ATTN)}


def _cgauss(rng: np.random.Generator, shape, scale: float = 1.0) -> np.ndarray:
    """Complex Gaussian with re, im ~ N(0, 1/2) each, times `scale`."""
    s = np.float32(scale * math.sqrt(0.5))
    out = np.empty(tuple(shape) + (2,), dtype=np.float32)
    out[...] = rng.standard_normal(out.shape, dtype=np.float32)
    out *= s
    return out.view(np.complex64).reshape(shape)


def _unit_phase(rng: np.random.Generator, shape) -> np.ndarray:
    phi = rng.uniform(-math.pi, math.pi, size=shape)
    return (np.cos(phi) + 1j * np.sin(phi)).astype(np.complex64)


def _rate_A(rng: np.random.Generator, H: int) -> np.ndarray:
    a_re = -np.exp(rng.uniform(math.log(0.5), math.log(4.0), size=H))
    a_im = rng.uniform(-math.pi, math.pi, size=H)
    return (a_re + 1j * a_im).astype(np.complex64)


def make_inputs(w: Workload, seed: int | None = None) -> dict:
    """Arrays for one forward pass of workload `w` (see the module docstring)."""
    rng = np.random.default_rng(w.seed if seed is None else seed)
    Bz, T, H, N, P = w.batch, w.seqlen, w.nheads, w.dstate, w.headdim
    if w.kind == "pam":
        return _make_pam(rng, w)
    x = _cgauss(rng, (Bz, T, H, P))
    B = _cgauss(rng, (Bz, T, H, N), 1.0 / math.sqrt(N))
    C = _cgauss(rng, (Bz, T, H, N), 1.0 / math.sqrt(N))
    dt = (rng.standard_normal((Bz, T, H), dtype=np.float32) * np.float32(0.5) - np.float32(1.0)).astype(np.float32)
    if w.kind == "slow_decay":
        # Per-head decay rho ~ U[0.9, 0.9999] at the mean step dt = -1:
        # Re A = ln(rho) / softplus(-1).
        rho = rng.uniform(0.9, 0.9999, size=H)
        a_re = np.log(rho) / _SOFTPLUS_MINUS_ONE
        a_im = rng.uniform(-math.pi, math.pi, size=H)
        A = (a_re + 1j * a_im).astype(np.complex64)
    else:
        A = _rate_A(rng, H)
    D = rng.standard_normal(H).astype(np.float32)
    out = dict(x=x, dt=dt, A=A, B=B, C=C, D=D)
    if w.kind == "decode":
        out["h"] = _cgauss(rng, (Bz, H, N, P))
    return out


def _make_pam(rng: np.random.Generator, w: Workload) -> dict:
    """Phase-associative memory stated on the SSD interface.

    The memory S_t = gamma S_{t-1} + V_t (x) conj(K_t), read as S_t Q_t / sqrt(d),
    is the SSD with h^T = S, B = conj(K), x = V, C = Q / sqrt(d), D = 0, and a
    constant real per-step decay gamma, reached through A = ln(gamma) + 0i and
    dt = ln(e - 1) so that softplus(dt) = 1.  Draw order: Q, K, V, gamma.
    The raw Q, K, V, gamma are returned too.
    """
    Bz, T, H, d = w.batch, w.seqlen, w.nheads, w.dstate
    assert w.dstate == w.headdim
    Q = _unit_phase(rng, (Bz, T, H, d))
    K = _unit_phase(rng, (Bz, T, H, d))
    V = _unit_phase(rng, (Bz, T, H, d))
    gamma = rng.uniform(0.9, 0.999, size=H)
    dt_one = np.float32(math.log(math.e - 1.0))
    return dict(
        x=V,
        dt=np.full((Bz, T, H), dt_one, dtype=np.float32),
        A=(np.log(gamma) + 0j).astype(np.complex64),
        B=np.conj(K).astype(np.complex64),
        C=(Q / np.float32(math.sqrt(d))).astype(np.complex64),
        D=np.zeros(H, dtype=np.float32),
        Q=Q,
        K=K,
        V=V,
        gamma=gamma,
    )


def decode_fixed(w: Workload = DECODE) -> dict:
    """A, D and the initial state h for the decode workload (fixed over steps)."""
    rng = np.random.default_rng(w.seed)
    A = _rate_A(rng, w.nheads)
    D = rng.standard_normal(w.nheads).astype(np.float32)
    h = _cgauss(rng, (w.batch, w.nheads, w.dstate, w.headdim))
    return dict(A=A, D=D, h=h)


def decode_token(w: Workload, step: int) -> dict:
    """Fresh per-token inputs for decode call number `step` (mamba2_layer laws).

    Each step has its own generator, seeded from (seed, step), so any subset of
    steps can be regenerated independently.
    """
    rng = np.random.default_rng([w.seed, 1 + step])
    Bz, H, N, P = w.batch, w.nheads, w.dstate, w.headdim
    x = _cgauss(rng, (Bz, H, P))
    B = _cgauss(rng, (Bz, H, N), 1.0 / math.sqrt(N))
    C = _cgauss(rng, (Bz, H, N), 1.0 / math.sqrt(N))
    dt = (rng.standard_normal((Bz, H), dtype=np.float32) * np.float32(0.5) - np.float32(1.0)).astype(np.float32)
    return dict(x=x, B=B, C=C, dt=dt)


def random_case(seed: int, Bz: int, T: int, H: int, N: int, P: int, *, dt_mean: float = -1.0,
                dt_std: float = 0.5, a_scale: float = 1.0) -> dict:
    """Small general case for parity sweeps: the mamba2_layer laws at any shape.

    `a_scale` multiplies A (a_scale = 0 gives A = 0).
    """
    rng = np.random.default_rng(seed)
    x = _cgauss(rng, (Bz, T, H, P))
    B = _cgauss(rng, (Bz, T, H, N), 1.0 / math.sqrt(N))
    C = _cgauss(rng, (Bz, T, H, N), 1.0 / math.sqrt(N))
    dt = (rng.standard_normal((Bz, T, H), dtype=np.float32) * np.float32(dt_std) + np.float32(dt_mean)).astype(np.float32)
    A = (_rate_A(rng, H) * np.complex64(a_scale)).astype(np.complex64)
    D = rng.standard_normal(H).astype(np.float32)
    return dict(x=x, dt=dt, A=A, B=B, C=C, D=D)


def random_state(seed: int, Bz: int, H: int, N: int, P: int) -> np.ndarray:
    """An initial state h0 [Bz,H,N,P] complex64: complex Gaussian, as the decode
    workload's state."""
    return _cgauss(np.random.default_rng(seed), (Bz, H, N, P))


def make_cayley_inputs(w: Workload = HMAMBA_SCAN, seed: int | None = None, *, gate_mean: float = 0.0) -> dict:
    """Inputs of the per-coordinate Cayley-phase scan (workload `w`'s shapes).

        phi  [Bz,T,H,N] float32    phase parameter, phi = dt/2 (delta + omega)
        u    [Bz,T,H,N] float32    gate logits
        b    [Bz,T,H,N] complex64  input projection
        C    [Bz,T,H,N] complex64  readout projection
        psi0 [Bz,H,N]   complex64  initial state

    Recipe (the H-Mamba substrate's parameterisation and initialisation): step
    sizes dt ~ U[0.1, 0.6] per (batch, token, head) (the range of a softplus
    step floored at 0.1); shifts delta ~ N(0, 0.1^2); base frequencies omega_k
    on a geometric grid over two decades, [0.05, 5], with alternating sign;
    gate logits u ~ N(gate_mean, 1) (near zero at initialisation, so gates
    near 1/2); b, C complex Gaussian with re, im ~ N(0, 1/2); psi0 a complex
    Gaussian prior per head normalised to unit norm, shared by the batch.
    Draw order: dt, delta, u, b, C, prior.
    """
    rng = np.random.default_rng(w.seed if seed is None else seed)
    Bz, T, H, N = w.batch, w.seqlen, w.nheads, w.dstate
    dt = rng.uniform(0.1, 0.6, size=(Bz, T, H, 1)).astype(np.float32)
    delta = (rng.standard_normal((Bz, T, H, N), dtype=np.float32) * np.float32(0.1)).astype(np.float32)
    omega = np.geomspace(0.05, 5.0, N).astype(np.float32) * np.where(np.arange(N) % 2 == 0, 1, -1).astype(np.float32)
    phi = (np.float32(0.5) * dt * (delta + omega)).astype(np.float32)
    del delta
    u = (rng.standard_normal((Bz, T, H, N), dtype=np.float32) + np.float32(gate_mean)).astype(np.float32)
    b = _cgauss(rng, (Bz, T, H, N))
    C = _cgauss(rng, (Bz, T, H, N))
    prior = _cgauss(rng, (H, N)).astype(np.complex128)
    prior /= np.linalg.norm(prior, axis=1, keepdims=True)
    psi0 = np.broadcast_to(prior.astype(np.complex64), (Bz, H, N)).copy()
    return dict(phi=phi, u=u, b=b, C=C, psi0=psi0)


def make_born_inputs(w: Workload = HTRANSFORMER_ATTN, seed: int | None = None) -> dict:
    """Inputs of causal Born attention (workload `w`'s shapes, D = w.dstate).

        q, k, v [Bz,T,H,D] complex64   queries, keys, values
        tau     [Bz,T,H]   float32     positive temperatures

    Recipe: q, k, v complex Gaussian with re, im ~ N(0, 1/2); queries and keys
    then carry the H-Transformer's per-position phase, component a of position
    t multiplied by e^{i t omega_a} with the base frequencies omega on a
    geometric grid over two decades, [0.05, 5], with alternating sign (the
    initialisation the phase-state paper describes); tau ~ U[0.5, 2].  Draw
    order: q, k, v, tau.
    """
    rng = np.random.default_rng(w.seed if seed is None else seed)
    Bz, T, H, D = w.batch, w.seqlen, w.nheads, w.dstate
    q = _cgauss(rng, (Bz, T, H, D))
    k = _cgauss(rng, (Bz, T, H, D))
    v = _cgauss(rng, (Bz, T, H, D))
    tau = rng.uniform(0.5, 2.0, size=(Bz, T, H)).astype(np.float32)
    omega = np.geomspace(0.05, 5.0, D) * np.where(np.arange(D) % 2 == 0, 1.0, -1.0)
    ang = np.arange(T, dtype=np.float64)[:, None] * omega[None, :]  # [T, D]
    rot = np.exp(1j * ang).astype(np.complex64)[None, :, None, :]
    q = (q * rot).astype(np.complex64)
    k = (k * rot).astype(np.complex64)
    return dict(q=q, k=k, v=v, tau=tau)
