"""PyTorch-facing calls of libssscan: argument checks, output allocation and the
C-ABI call on the current CUDA stream.  No arithmetic of the method is done here.

Names and argument order follow include/ssscan.h:

* ``ss_scan_fwd(x, delta, A, Bm, Cm, Dv, z, h0=None, chunk=64, workspace=None)``
  -> ``(y, ckpt, h_last)``
* ``ss_scan_bwd(x, delta, A, Bm, Cm, Dv, z, ckpt, dy, dh_last=None, chunk=64, dA=None, dD=None, ...)``
  -> dict of gradients
* ``conv1d_causal_bwd(dout, x, w, dw=None, db=None)`` -> ``(dx, dw, db)``
* ``rmsnorm_bwd(dy, x, scale, rms, dscale=None)`` -> ``(dx, dscale)``
* ``conv1d_causal_fwd(x, w, bias=None, silu=False)`` -> ``out``
* ``conv1d_causal_silu_bwd(dact, x, w, bias=None, dw=None, db=None)`` -> ``(dx, dw, db)``
* ``rmsnorm_fwd(x, scale, eps)`` -> ``(y, rms)``
* ``ss_scan_step(x, delta, A, Bm, Cm, Dv, z, h)`` -> ``y`` (h updated in place)
* ``ss_scan_fwd_summary(x, delta, A, Bm)`` -> ``(h_end, delta_sum)``;
  ``ss_scan_bwd_summary(delta, A, Cm, z, dy)`` -> ``(g_start, delta_sum)``;
  ``ss_scan_carries(A, delta_sum, summ, init=None, reverse=False)`` -> ``carry``
  (the pieces of a sequence-sharded scan; ``sharded.py`` runs them over ranks)
* ``conv1d_causal_step(x, conv_state, w, bias=None, silu=False)`` -> ``out`` (state updated in place)

Activations are ``torch.float32`` or ``torch.bfloat16`` CUDA tensors, contiguous;
parameters, states and gradients are ``torch.float32``.
"""

from __future__ import annotations

import ctypes

import torch

from . import _capi
from ._capi import SS_BF16, SS_F32, check, load

_DT = {torch.float32: SS_F32, torch.bfloat16: SS_BF16}


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _req(t, name, shape=None, dtype=None, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous (strided views are not accepted)")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    return t


def _act_dtype(x):
    if x.dtype not in _DT:
        raise ValueError(f"activations must be float32 or bfloat16, got {x.dtype}")
    return _DT[x.dtype]


def num_chunks(L: int, chunk: int) -> int:
    return load().ss_scan_num_chunks(L, chunk)


def scan_fwd_workspace_size(B, L, D, N, chunk, dtype) -> int:
    return load().ss_scan_fwd_workspace_size(B, L, D, N, chunk, _DT[dtype])


def ss_scan_fwd(x, delta, A, Bm, Cm, Dv, z, h0=None, chunk: int = 64, want_h_last: bool = True, workspace=None,
                dt_bias=None, delta_softplus: bool = False):
    """Forward scan -> ``(y, ckpt, h_last)``.  With ``dt_bias`` / ``delta_softplus`` the
    recurrence uses softplus(delta + dt_bias) (or delta + dt_bias), computed in the kernel."""
    lib = load()
    B, L, D = x.shape
    N = A.shape[1]
    dev, dt = x.device, x.dtype
    _act_dtype(x)
    for name, t in (("x", x), ("delta", delta), ("z", z)):
        _req(t, name, (B, L, D), dt, dev)
    for name, t in (("Bm", Bm), ("Cm", Cm)):
        _req(t, name, (B, L, N), dt, dev)
    _req(A, "A", (D, N), torch.float32, dev)
    _req(Dv, "Dv", (D,), torch.float32, dev)
    if h0 is not None:
        _req(h0, "h0", (B, D, N), torch.float32, dev)
    if dt_bias is not None:
        _req(dt_bias, "dt_bias", (D,), torch.float32, dev)
    nck = num_chunks(L, chunk) if L > 0 and chunk > 0 else 0
    y = torch.empty_like(x)
    ckpt = torch.empty((B, max(nck, 1), D, N), device=dev, dtype=torch.float32)
    h_last = torch.empty((B, D, N), device=dev, dtype=torch.float32) if want_h_last else None
    ws_bytes = lib.ss_scan_fwd_workspace_size(B, L, D, N, chunk, _DT[dt])
    if workspace is None and ws_bytes > 0:
        workspace = torch.empty(ws_bytes, device=dev, dtype=torch.uint8)
    ws_have = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = lib.ss_scan_fwd(_p(x), _p(delta), _p(A), _p(Bm), _p(Cm), _p(Dv), _p(z), _p(h0), _p(y), _p(ckpt), _p(h_last),
                         B, L, D, N, chunk, _DT[dt], _p(dt_bias), int(bool(delta_softplus)), _p(workspace), ws_have,
                         _stream())
    check(rc, "ss_scan_fwd")
    return y, ckpt, h_last


def scan_bwd_workspace_size(B, L, D, N, chunk, dtype) -> int:
    return load().ss_scan_bwd_workspace_size(B, L, D, N, chunk, _DT[dtype])


def ss_scan_bwd(x, delta, A, Bm, Cm, Dv, z, ckpt, dy, dh_last=None, chunk: int = 64, dA=None, dD=None,
                want_dh0: bool = True, workspace=None, out=None, dt_bias=None, delta_softplus: bool = False,
                d_dt_bias=None):
    """Gradients of sum(y*dy) (+ sum(h_last*dh_last)).  dA and dD accumulate into the
    given tensors (zeros when None); the rest are returned freshly (or written into ``out``).
    With the fused discretisation (same ``dt_bias`` / ``delta_softplus`` as the forward),
    ``ddelta`` is the gradient of the raw delta and ``d_dt_bias`` accumulates (zeros when None)."""
    lib = load()
    B, L, D = x.shape
    N = A.shape[1]
    dev, dt = x.device, x.dtype
    _act_dtype(x)
    for name, t in (("x", x), ("delta", delta), ("z", z), ("dy", dy)):
        _req(t, name, (B, L, D), dt, dev)
    for name, t in (("Bm", Bm), ("Cm", Cm)):
        _req(t, name, (B, L, N), dt, dev)
    _req(A, "A", (D, N), torch.float32, dev)
    _req(Dv, "Dv", (D,), torch.float32, dev)
    _req(ckpt, "ckpt", (B, num_chunks(L, chunk), D, N), torch.float32, dev)
    if dh_last is not None:
        _req(dh_last, "dh_last", (B, D, N), torch.float32, dev)
    f32 = dict(device=dev, dtype=torch.float32)
    if out is None:
        out = {
            "dx": torch.empty((B, L, D), **f32), "ddelta": torch.empty((B, L, D), **f32),
            "dz": torch.empty((B, L, D), **f32), "dB": torch.empty((B, L, N), **f32),
            "dC": torch.empty((B, L, N), **f32),
            "dh0": torch.empty((B, D, N), **f32) if want_dh0 else None,
        }
    fused = dt_bias is not None or delta_softplus
    if dt_bias is not None:
        _req(dt_bias, "dt_bias", (D,), torch.float32, dev)
    if fused:
        out["d_dt_bias"] = (torch.zeros((D,), **f32) if d_dt_bias is None
                            else _req(d_dt_bias, "d_dt_bias", (D,), torch.float32, dev))
    out["dA"] = torch.zeros((D, N), **f32) if dA is None else _req(dA, "dA", (D, N), torch.float32, dev)
    out["dD"] = torch.zeros((D,), **f32) if dD is None else _req(dD, "dD", (D,), torch.float32, dev)
    ws_bytes = lib.ss_scan_bwd_workspace_size(B, L, D, N, chunk, _DT[dt])
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 16), device=dev, dtype=torch.uint8)
    rc = lib.ss_scan_bwd(_p(x), _p(delta), _p(A), _p(Bm), _p(Cm), _p(Dv), _p(z), _p(ckpt), _p(dy), _p(dh_last),
                         _p(out["dx"]), _p(out["ddelta"]), _p(out["dz"]), _p(out["dA"]), _p(out["dB"]), _p(out["dC"]),
                         _p(out["dD"]), _p(out.get("dh0")), B, L, D, N, chunk, _DT[dt], _p(dt_bias),
                         int(bool(delta_softplus)), _p(out.get("d_dt_bias")), _p(workspace),
                         workspace.numel() * workspace.element_size(), _stream())
    check(rc, "ss_scan_bwd")
    return out


def ss_scan_fwd_summary(x, delta, A, Bm, dt_bias=None, delta_softplus: bool = False):
    """Forward summary of one piece of a sequence -> ``(h_end [B,D,N], delta_sum [B,D])``:
    the state the piece reaches from a zero start and its sum of (discretised) delta."""
    lib = load()
    B, L, D = x.shape
    N = A.shape[1]
    dev, dt = x.device, x.dtype
    _act_dtype(x)
    _req(x, "x", (B, L, D), dt, dev)
    _req(delta, "delta", (B, L, D), dt, dev)
    _req(Bm, "Bm", (B, L, N), dt, dev)
    _req(A, "A", (D, N), torch.float32, dev)
    if dt_bias is not None:
        _req(dt_bias, "dt_bias", (D,), torch.float32, dev)
    h_end = torch.empty((B, D, N), device=dev, dtype=torch.float32)
    dsum = torch.empty((B, D), device=dev, dtype=torch.float32)
    rc = lib.ss_scan_fwd_summary(_p(x), _p(delta), _p(A), _p(Bm), _p(h_end), _p(dsum), B, L, D, N, _DT[dt],
                                 _p(dt_bias), int(bool(delta_softplus)), _stream())
    check(rc, "ss_scan_fwd_summary")
    return h_end, dsum


def ss_scan_bwd_summary(delta, A, Cm, z, dy, dt_bias=None, delta_softplus: bool = False):
    """Backward summary of one piece -> ``(g_start [B,D,N], delta_sum [B,D])``: the adjoint the
    piece sends out of its first step when no carry arrives at its end, and its sum of delta."""
    lib = load()
    B, L, D = delta.shape
    N = A.shape[1]
    dev, dt = delta.device, delta.dtype
    _act_dtype(delta)
    for name, t in (("delta", delta), ("z", z), ("dy", dy)):
        _req(t, name, (B, L, D), dt, dev)
    _req(Cm, "Cm", (B, L, N), dt, dev)
    _req(A, "A", (D, N), torch.float32, dev)
    if dt_bias is not None:
        _req(dt_bias, "dt_bias", (D,), torch.float32, dev)
    g_start = torch.empty((B, D, N), device=dev, dtype=torch.float32)
    dsum = torch.empty((B, D), device=dev, dtype=torch.float32)
    rc = lib.ss_scan_bwd_summary(_p(delta), _p(A), _p(Cm), _p(z), _p(dy), _p(g_start), _p(dsum), B, L, D, N, _DT[dt],
                                 _p(dt_bias), int(bool(delta_softplus)), _stream())
    check(rc, "ss_scan_bwd_summary")
    return g_start, dsum


def ss_scan_carries(A, delta_sum, summ, init=None, reverse: bool = False):
    """Compose P pieces' affine maps (piece-major ``delta_sum [P,B,D]``, ``summ [P,B,D,N]``)
    -> ``carry [P,B,D,N]``: the state entering each piece (forward) or the carry arriving
    at its end (``reverse``), starting from ``init`` (zeros when None)."""
    lib = load()
    P, B, D, N = summ.shape
    dev = summ.device
    _req(A, "A", (D, N), torch.float32, dev)
    _req(delta_sum, "delta_sum", (P, B, D), torch.float32, dev)
    _req(summ, "summ", (P, B, D, N), torch.float32, dev)
    if init is not None:
        _req(init, "init", (B, D, N), torch.float32, dev)
    carry = torch.empty((P, B, D, N), device=dev, dtype=torch.float32)
    rc = lib.ss_scan_carries(_p(A), _p(delta_sum), _p(summ), _p(init), _p(carry), P, B, D, N, int(bool(reverse)),
                             _stream())
    check(rc, "ss_scan_carries")
    return carry


def conv1d_causal_bwd(dout, x, w, dw=None, db=None, workspace=None):
    lib = load()
    B, L, D = x.shape
    K = w.shape[1]
    dev = x.device
    xdt = _act_dtype(x)
    _req(dout, "dout", (B, L, D), torch.float32, dev)
    _req(x, "x", (B, L, D), x.dtype, dev)
    _req(w, "w", (D, K), torch.float32, dev)
    dw = torch.zeros((D, K), device=dev, dtype=torch.float32) if dw is None else _req(dw, "dw", (D, K), torch.float32, dev)
    db = torch.zeros((D,), device=dev, dtype=torch.float32) if db is None else _req(db, "db", (D,), torch.float32, dev)
    dx = torch.empty((B, L, D), device=dev, dtype=torch.float32)
    ws_bytes = lib.conv1d_causal_bwd_workspace_size(B, L, D, K)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 16), device=dev, dtype=torch.uint8)
    rc = lib.conv1d_causal_bwd(_p(dout), _p(x), _p(w), _p(dx), _p(dw), _p(db), B, L, D, K, xdt, _p(workspace),
                               workspace.numel() * workspace.element_size(), _stream())
    check(rc, "conv1d_causal_bwd")
    return dx, dw, db


def conv1d_causal_silu_bwd(dact, x, w, bias=None, dw=None, db=None, workspace=None):
    """Backward through silu(conv1d(x) + bias) given dL/d(silu output); dw, db accumulate."""
    lib = load()
    B, L, D = x.shape
    K = w.shape[1]
    dev = x.device
    xdt = _act_dtype(x)
    _req(dact, "dact", (B, L, D), torch.float32, dev)
    _req(x, "x", (B, L, D), x.dtype, dev)
    _req(w, "w", (D, K), torch.float32, dev)
    if bias is not None:
        _req(bias, "bias", (D,), torch.float32, dev)
    dw = torch.zeros((D, K), device=dev, dtype=torch.float32) if dw is None else _req(dw, "dw", (D, K), torch.float32, dev)
    db = torch.zeros((D,), device=dev, dtype=torch.float32) if db is None else _req(db, "db", (D,), torch.float32, dev)
    dx = torch.empty((B, L, D), device=dev, dtype=torch.float32)
    ws_bytes = lib.conv1d_causal_bwd_workspace_size(B, L, D, K)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 16), device=dev, dtype=torch.uint8)
    rc = lib.conv1d_causal_silu_bwd(_p(dact), _p(x), _p(w), _p(bias), _p(dx), _p(dw), _p(db), B, L, D, K, xdt,
                                    _p(workspace), workspace.numel() * workspace.element_size(), _stream())
    check(rc, "conv1d_causal_silu_bwd")
    return dx, dw, db


def rmsnorm_bwd(dy, x, scale, rms, dscale=None, workspace=None):
    lib = load()
    R, H = x.shape
    dev = x.device
    dt = _act_dtype(x)
    _req(dy, "dy", (R, H), x.dtype, dev)
    _req(x, "x", (R, H), x.dtype, dev)
    _req(scale, "scale", (H,), torch.float32, dev)
    _req(rms, "rms", (R,), torch.float32, dev)
    dscale = torch.zeros((H,), device=dev, dtype=torch.float32) if dscale is None else _req(
        dscale, "dscale", (H,), torch.float32, dev)
    dx = torch.empty((R, H), device=dev, dtype=torch.float32)
    ws_bytes = lib.rmsnorm_bwd_workspace_size(R, H)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 16), device=dev, dtype=torch.uint8)
    rc = lib.rmsnorm_bwd(_p(dy), _p(x), _p(scale), _p(rms), _p(dx), _p(dscale), R, H, dt, _p(workspace),
                         workspace.numel() * workspace.element_size(), _stream())
    check(rc, "rmsnorm_bwd")
    return dx, dscale


def conv1d_causal_fwd(x, w, bias=None, silu: bool = False, out=None):
    """Depthwise causal conv1d (+ optional SiLU); ``out`` has x's dtype."""
    lib = load()
    B, L, D = x.shape
    K = w.shape[1]
    dev = x.device
    xdt = _act_dtype(x)
    _req(x, "x", (B, L, D), x.dtype, dev)
    _req(w, "w", (D, K), torch.float32, dev)
    if bias is not None:
        _req(bias, "bias", (D,), torch.float32, dev)
    out = torch.empty_like(x) if out is None else _req(out, "out", (B, L, D), x.dtype, dev)
    rc = lib.conv1d_causal_fwd(_p(x), _p(w), _p(bias), _p(out), B, L, D, K, int(bool(silu)), xdt, _stream())
    check(rc, "conv1d_causal_fwd")
    return out


def rmsnorm_fwd(x, scale, eps: float, want_rms: bool = True):
    """RMSNorm forward: ``(y, rms)`` with y in x's dtype and rms fp32 (None unless ``want_rms``)."""
    lib = load()
    R, H = x.shape
    dev = x.device
    dt = _act_dtype(x)
    _req(x, "x", (R, H), x.dtype, dev)
    _req(scale, "scale", (H,), torch.float32, dev)
    y = torch.empty_like(x)
    rms = torch.empty((R,), device=dev, dtype=torch.float32) if want_rms else None
    rc = lib.rmsnorm_fwd(_p(x), _p(scale), float(eps), _p(y), _p(rms), R, H, dt, _stream())
    check(rc, "rmsnorm_fwd")
    return y, rms


def ss_scan_step(x, delta, A, Bm, Cm, Dv, z, h):
    """One decode step for B sequences: updates ``h`` [B,D,N] in place and returns y [B,D]."""
    lib = load()
    B, D = x.shape
    N = A.shape[1]
    dev, dt = x.device, x.dtype
    _act_dtype(x)
    for name, t in (("x", x), ("delta", delta), ("z", z)):
        _req(t, name, (B, D), dt, dev)
    for name, t in (("Bm", Bm), ("Cm", Cm)):
        _req(t, name, (B, N), dt, dev)
    _req(A, "A", (D, N), torch.float32, dev)
    _req(Dv, "Dv", (D,), torch.float32, dev)
    _req(h, "h", (B, D, N), torch.float32, dev)
    y = torch.empty_like(x)
    rc = lib.ss_scan_step(_p(x), _p(delta), _p(A), _p(Bm), _p(Cm), _p(Dv), _p(z), _p(h), _p(y), B, D, N, _DT[dt],
                          _stream())
    check(rc, "ss_scan_step")
    return y


def conv1d_causal_step(x, conv_state, w, bias=None, silu: bool = False):
    """One conv step for B sequences: shifts ``conv_state`` [B,D,K] in place and returns out [B,D]."""
    lib = load()
    B, D = x.shape
    K = w.shape[1]
    dev = x.device
    xdt = _act_dtype(x)
    _req(conv_state, "conv_state", (B, D, K), torch.float32, dev)
    _req(w, "w", (D, K), torch.float32, dev)
    if bias is not None:
        _req(bias, "bias", (D,), torch.float32, dev)
    out = torch.empty_like(x)
    rc = lib.conv1d_causal_step(_p(x), _p(conv_state), _p(w), _p(bias), _p(out), B, D, K, int(bool(silu)), xdt,
                                _stream())
    check(rc, "conv1d_causal_step")
    return out


def count_nonfinite(t, workspace=None) -> int:
    """Number of NaN / +-Inf values in a dense fp32 or bf16 CUDA tensor (synchronises the current stream)."""
    lib = load()
    dt = _act_dtype(t)
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError("count_nonfinite: t must be a contiguous CUDA tensor")
    wsz = lib.ss_count_nonfinite_workspace_size()
    ws = workspace if workspace is not None else torch.empty((wsz,), device=t.device, dtype=torch.uint8)
    out = torch.empty((1,), device=t.device, dtype=torch.int64)
    rc = lib.ss_count_nonfinite(_p(t), t.numel(), dt, _p(out), _p(ws), ws.numel() * ws.element_size(), _stream())
    check(rc, "ss_count_nonfinite")
    return int(out.item())


def device_status() -> int:
    """Reads and clears the library's device error word (synchronises the current stream)."""
    return load().ss_device_status(_stream())
