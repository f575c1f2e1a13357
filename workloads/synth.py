"""Workload definitions and seeded input generators.

The five workloads are the Mamba-shaped layers the method is measured on:

* ``tiny``      B=2, L=64, D=16, N=4, fp32 — small enough for the oracle's
                finite-difference checks and exact comparison;
* ``mamba130m`` B=8, L=2048, d_model=768, D=1536, N=16, fp32;
* ``mamba1p4b`` B=4, L=2048, d_model=2048, D=4096, N=16, bf16 activations with
                fp32 state and fp32 gradients (the throughput workload);
* ``short``     B=4096, L=32, D=64, N=16, fp32 — many short sequences, where the
                cross-batch reductions of dA/dB/dC dominate;
* ``long``      B=1, L=16384, D=2048, N=16, bf16, long-memory step sizes,
                checkpoint every 256 steps.

Distributions (all drawn in float64 with ``numpy.random.Generator(PCG64)``):

* ``dt_bias[d] = softplus^{-1}(u)``, ``u = exp(Uniform(ln lo, ln hi))`` per
  channel (``[lo, hi] = [1e-3, 1e-1]``, long memory ``[1e-4, 1e-2]``);
* ``delta[b,t,d] = softplus(0.5 * eps[b,t,d] + dt_bias[d])``, ``eps ~ N(0,1)``;
* ``x, z, Bm, Cm, dy ~ N(0,1)``; ``A[d,n] = -(n+1)``; ``Dv[d] = 1``; no h0.

Every array is rounded to the workload's activation dtype (fp32 or bf16,
round-to-nearest-even) and returned as float64 holding exactly the rounded
values, so that the oracle and the CUDA path see identical numbers.  The
three generator streams (scan, conv1d, RMSNorm) are independent PCG64 streams
keyed by ``(seed, stream)`` so each can be drawn without the others.
"""

from __future__ import annotations

import dataclasses
from dataclasses import dataclass

import numpy as np

_STREAM_SCAN, _STREAM_CONV, _STREAM_RMS = 0, 1, 2


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    L: int
    D: int  # d_inner: scan / conv channels
    N: int  # SSM state size
    d_conv: int
    d_model: int  # RMSNorm width
    dtype: str  # activation dtype: "f32" or "bf16"
    dt_lo: float
    dt_hi: float
    chunk: int  # checkpoint interval of the scan
    desc: str = ""

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)

    @property
    def elems(self) -> int:
        return self.B * self.L * self.D


CONFIGS = {
    "tiny": Workload("tiny", 2, 64, 16, 4, 4, 8, "f32", 1e-3, 1e-1, 64,
                     "tiny fp32 scan fwd+bwd: B=2, L=64, d_inner=16, N=4, d_conv=4"),
    "mamba130m": Workload("mamba130m", 8, 2048, 1536, 16, 4, 768, "f32", 1e-3, 1e-1, 8,
                          "Mamba-130M-shaped layer: B=8, L=2048, d_model=768, d_inner=1536, N=16, fp32"),
    "mamba1p4b": Workload("mamba1p4b", 4, 2048, 4096, 16, 4, 2048, "bf16", 1e-3, 1e-1, 8,
                          "Mamba-1.4B-shaped layer: B=4, L=2048, d_model=2048, d_inner=4096, N=16, "
                          "bf16 x/delta/B/C/z/dy, fp32 state and grads"),
    "short": Workload("short", 4096, 32, 64, 16, 4, 32, "f32", 1e-3, 1e-1, 8,
                      "short-sequence many-batch scan: B=4096, L=32, d_inner=64, N=16, fp32"),
    "long": Workload("long", 1, 16384, 2048, 16, 4, 1024, "bf16", 1e-4, 1e-2, 256,
                     "long-context scan: B=1, L=16384, d_inner=2048, N=16, bf16, long-memory delta, "
                     "checkpoint every 256 steps"),
}


def get_config(name: str) -> Workload:
    return CONFIGS[name]


def _rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64([int(seed), int(stream)]))


def round_to(a: np.ndarray, dtype: str) -> np.ndarray:
    """Round float64 values to the activation dtype (RNE) and return them as float64."""
    a = np.asarray(a, dtype=np.float64)
    if dtype == "f32":
        return a.astype(np.float32).astype(np.float64)
    if dtype == "bf16":
        # Round-to-nearest-even onto the bf16 grid via float32 bits; inputs here
        # are finite and far from the float32 range limits.
        f = a.astype(np.float32)
        bits = f.view(np.uint32).astype(np.uint64)
        lsb = (bits >> np.uint64(16)) & np.uint64(1)
        bits = (bits + np.uint64(0x7FFF) + lsb) & np.uint64(0xFFFF0000)
        return bits.astype(np.uint32).view(np.float32).astype(np.float64)
    raise ValueError(f"unknown dtype {dtype!r}")


def _softplus(v: np.ndarray) -> np.ndarray:
    return np.logaddexp(0.0, v)


def _softplus_inv(u: np.ndarray) -> np.ndarray:
    return np.log(np.expm1(u))


def make_scan_inputs(wl: Workload, seed: int = 0) -> dict:
    """Inputs of the selective scan for workload ``wl``.

    Returns float64 arrays (exactly representable in ``wl.dtype`` for the
    activations, in fp32 for A and Dv): ``x, delta, z, dy`` of shape [B,L,D],
    ``Bm, Cm`` of shape [B,L,N], ``A`` [D,N], ``Dv`` [D], plus ``dt_bias`` [D] and
    ``delta_raw`` [B,L,D] = 0.5*eps, the pre-bias, pre-softplus value whose
    softplus(delta_raw + dt_bias) is ``delta`` before rounding.
    Draw order: dt_bias, eps, x, z, Bm, Cm, dy.
    """
    rng = _rng(seed, _STREAM_SCAN)
    B, L, D, N = wl.B, wl.L, wl.D, wl.N
    u = np.exp(rng.uniform(np.log(wl.dt_lo), np.log(wl.dt_hi), size=D))
    dt_bias = _softplus_inv(u)
    eps = rng.standard_normal((B, L, D))
    x = rng.standard_normal((B, L, D))
    z = rng.standard_normal((B, L, D))
    Bm = rng.standard_normal((B, L, N))
    Cm = rng.standard_normal((B, L, N))
    dy = rng.standard_normal((B, L, D))
    delta = _softplus(0.5 * eps + dt_bias[None, None, :])
    A = -np.broadcast_to(np.arange(1, N + 1, dtype=np.float64), (D, N)).copy()
    Dv = np.ones(D)
    r = lambda a: round_to(a, wl.dtype)
    return {
        "x": r(x), "delta": r(delta), "z": r(z), "Bm": r(Bm), "Cm": r(Cm), "dy": r(dy),
        "A": round_to(A, "f32"), "Dv": round_to(Dv, "f32"), "dt_bias": round_to(dt_bias, "f32"),
        "delta_raw": r(0.5 * eps),
    }


def make_conv_inputs(wl: Workload, seed: int = 0) -> dict:
    """Inputs of the depthwise causal conv1d backward.

    ``dout`` [B,L,D] fp32 ~ N(0,1) (the gradient after the SiLU backward),
    ``x`` [B,L,D] in ``wl.dtype`` ~ N(0,1), ``w`` [D,d_conv] fp32 ~ U(+-1/sqrt(d_conv)).
    """
    rng = _rng(seed, _STREAM_CONV)
    B, L, D, K = wl.B, wl.L, wl.D, wl.d_conv
    dout = rng.standard_normal((B, L, D))
    x = rng.standard_normal((B, L, D))
    bound = 1.0 / np.sqrt(K)
    w = rng.uniform(-bound, bound, size=(D, K))
    return {"dout": round_to(dout, "f32"), "x": round_to(x, wl.dtype), "w": round_to(w, "f32")}


RMS_EPS = 1e-5


def make_rmsnorm_inputs(wl: Workload, seed: int = 0, rows: int | None = None, dim: int | None = None) -> dict:
    """Inputs of the RMSNorm backward over ``[rows, dim]`` (default ``[B*L, d_model]``).

    ``x, dy`` ~ N(0,1) in ``wl.dtype``; ``scale = 1 + 0.1*N(0,1)`` fp32; ``rms``
    is the statistic the forward saves, ``sqrt(mean(x^2) + 1e-5)`` per row, in fp32.
    """
    rng = _rng(seed, _STREAM_RMS)
    R = wl.B * wl.L if rows is None else rows
    H = wl.d_model if dim is None else dim
    x = round_to(rng.standard_normal((R, H)), wl.dtype)
    dy = round_to(rng.standard_normal((R, H)), wl.dtype)
    scale = round_to(1.0 + 0.1 * rng.standard_normal(H), "f32")
    rms = round_to(np.sqrt(np.mean(x * x, axis=1) + RMS_EPS), "f32")
    return {"x": x, "dy": dy, "scale": scale, "rms": rms}
