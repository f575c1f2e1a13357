"""RMSNorm forward and backward in float64 (oracle; test infrastructure only).

Forward, per row b of x [R, H]:  rms_b = sqrt(mean_i x[b,i]^2 + eps),
y[b,i] = x[b,i] * scale[i] / rms_b.  The backward receives the saved ``rms``
(the root mean square itself, not its inverse) and follows the formula of
mamba-rs ``backward_ops.rs``, ``backward_rms_norm``:

    inv      = 1 / rms_b
    dot_b    = inv^2 * sum_i dy[b,i] * scale[i] * x[b,i]
    dx[b,i]  = inv * (scale[i] * dy[b,i] - x[b,i] * dot_b / H)
    dscale[i] = sum_b dy[b,i] * x[b,i] * inv

This dx is the full gradient through rms(x): eps enters only through the saved rms.
"""

from __future__ import annotations

import numpy as np


def rmsnorm_fwd_ref(x, scale, eps: float):
    """Returns (y [R,H], rms [R])."""
    x = np.asarray(x, np.float64)
    rms = np.sqrt(np.mean(x * x, axis=1) + eps)
    return x * np.asarray(scale, np.float64)[None, :] / rms[:, None], rms


def rmsnorm_bwd_ref(dy, x, scale, rms):
    """Returns (dx [R,H], dscale [H]) for the loss sum(y * dy)."""
    dy = np.asarray(dy, np.float64)
    x = np.asarray(x, np.float64)
    scale = np.asarray(scale, np.float64)
    inv = 1.0 / np.asarray(rms, np.float64)
    H = x.shape[1]
    dot = np.sum(dy * scale[None, :] * x, axis=1) * inv * inv
    dx = inv[:, None] * (scale[None, :] * dy - x * dot[:, None] / H)
    dscale = np.sum(dy * x * inv[:, None], axis=0)
    return dx, dscale
