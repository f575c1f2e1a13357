"""Depthwise causal conv1d: forward and backward in float64 (oracle; test infrastructure only).

Per channel d the causal filter reads the shift register of the last d_conv
inputs, newest at tap d_conv-1 (mamba-rs ``backward_ops.rs``,
``backward_conv1d_step``: "current x_branch feeds into position d_conv - 1"):

    state_t[d, k] = x[t - (d_conv-1) + k, d]      (x at negative time = 0)
    out[t, d]     = bias[d] + sum_k w[d, k] * state_t[d, k]

Full-sequence backward, given dout = dL/dout (the gradient after the SiLU
backward):

    dx[s, d] = sum_k dout[s + (d_conv-1) - k, d] * w[d, k]   (terms past the end dropped)
    dw[d, k] = sum_{b,t} dout[t, d] * state_t[d, k]
    db[d]    = sum_{b,t} dout[t, d]

The per-step function of the pages, which treats the shift register as saved
state and sends the input gradient through the newest tap only, is kept as
``conv1d_step_bwd_ref``; the full-sequence dw and db equal its per-step
contributions summed over time.
"""

from __future__ import annotations

import numpy as np


def _state(x: np.ndarray, k: int, K: int) -> np.ndarray:
    """state[:, t, :] for tap k: x shifted right by (K-1-k) steps with zero fill. x [B,L,D]."""
    shift = K - 1 - k
    out = np.zeros_like(x)
    if shift < x.shape[1]:
        out[:, shift:, :] = x[:, : x.shape[1] - shift, :]
    return out


def conv1d_causal_fwd_ref(x, w, bias=None):
    """out [B,L,D] = bias + sum_k w[:,k] * state_k."""
    x = np.asarray(x, np.float64)
    w = np.asarray(w, np.float64)
    K = w.shape[1]
    out = np.zeros_like(x) if bias is None else np.broadcast_to(np.asarray(bias, np.float64), x.shape).copy()
    for k in range(K):
        out += _state(x, k, K) * w[None, None, :, k]
    return out


def silu_ref(v):
    """SiLU, the activation after the conv: v * sigmoid(v) = v / (1 + exp(-v)), float64."""
    v = np.asarray(v, np.float64)
    return v / (1.0 + np.exp(-v))


def conv1d_causal_silu_fwd_ref(x, w, bias=None):
    """The conv -> SiLU branch: silu(conv1d_causal_fwd_ref(x, w, bias))."""
    return silu_ref(conv1d_causal_fwd_ref(x, w, bias))


def conv1d_causal_bwd_ref(dout, x, w):
    """Returns (dx [B,L,D], dw [D,K], db [D]) for the loss sum(out * dout)."""
    dout = np.asarray(dout, np.float64)
    x = np.asarray(x, np.float64)
    w = np.asarray(w, np.float64)
    Bsz, L, D = x.shape
    K = w.shape[1]
    dx = np.zeros_like(x)
    for k in range(K):
        shift = K - 1 - k  # out[t] reads x[t - shift] through tap k
        if shift < L:
            dx[:, : L - shift, :] += dout[:, shift:, :] * w[None, None, :, k]
    dw = np.empty((D, K))
    for k in range(K):
        dw[:, k] = np.sum(dout * _state(x, k, K), axis=(0, 1))
    db = np.sum(dout, axis=(0, 1))
    return dx, dw, db


def conv1d_step_fwd_ref(state, x_t, w, bias=None, silu: bool = False):
    """One step of the causal conv for B sequences: state [B,D,K] (newest input at
    K-1) shifts one tap towards 0 and takes x_t [B,D] at K-1; the output is
    act(bias + sum_k w[:,k] state[..., k]).  Returns (new_state, out)."""
    state = np.asarray(state, np.float64)
    new = np.concatenate([state[:, :, 1:], np.asarray(x_t, np.float64)[:, :, None]], axis=2)
    out = np.sum(new * np.asarray(w, np.float64)[None, :, :], axis=2)
    if bias is not None:
        out = out + np.asarray(bias, np.float64)[None, :]
    return new, (silu_ref(out) if silu else out)


def dsilu_ref(v):
    """d/dv silu(v) = s (1 + v (1 - s)), s = 1 / (1 + exp(-v)), float64."""
    v = np.asarray(v, np.float64)
    s = 1.0 / (1.0 + np.exp(-v))
    return s * (1.0 + v * (1.0 - s))


def conv1d_causal_silu_bwd_ref(dact, x, w, bias=None):
    """Backward of silu(conv1d_causal_fwd_ref(x, w, bias)) for the loss sum(act * dact).

    Chain rule: the conv receives g = dact * silu'(pre) at its output and
    conv1d_causal_bwd_ref does the rest; the bias gradient equals db.
    Returns (dx, dw, db)."""
    pre = conv1d_causal_fwd_ref(x, w, bias)
    return conv1d_causal_bwd_ref(np.asarray(dact, np.float64) * dsilu_ref(pre), x, w)


def conv1d_step_bwd_ref(d_out, conv_state, w, dw, db):
    """One timestep of the pages' conv1d backward (mamba-rs ``backward_conv1d_step``).

    d_out [D], conv_state [D,K] (newest input at K-1), w [D,K].  Accumulates
    into dw [D,K] and db [D] in place and returns dx [D] = d_out * w[:, K-1].
    """
    d_out = np.asarray(d_out, np.float64)
    db += d_out
    dw += d_out[:, None] * np.asarray(conv_state, np.float64)
    return d_out * np.asarray(w, np.float64)[:, -1]
