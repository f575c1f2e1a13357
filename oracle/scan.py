"""Selective-scan forward and backward in float64 (oracle; test infrastructure only).

Definition (the diagonal selective SSM the pages train by backpropagation
through time; rustytorch ``backward_cuda`` commit message, mamba-rs crate
description):

    a_t[d,n] = exp(delta_t[d] * A[d,n])
    h_t[d,n] = a_t[d,n] * h_{t-1}[d,n] + delta_t[d] * B_t[n] * x_t[d]     (h_{-1} = h0, else 0)
    s_t[d]   = sum_n C_t[n] * h_t[d,n] + D[d] * x_t[d]
    y_t[d]   = s_t[d] * silu(z_t[d]),    silu(z) = z * sigmoid(z)

Shapes: x, delta, z, y, dy: [B, L, D]; Bm, Cm: [B, L, N]; A: [D, N]; Dv: [D];
h0, h_last: [B, D, N]; checkpoints [B, ceil(L/chunk), D, N] with
ckpt[b, c, d, :] = the state just before step c*chunk (c = 0 holds h0 or zeros).

Backward of the scalar loss sum(y * dy), by hand (reverse mode):

    ds_t = dy_t * silu(z_t)
    dz_t = dy_t * s_t * sigmoid(z_t) * (1 + z_t * (1 - sigmoid(z_t)))
    G_t  = dL/dh_t = ds_t * C_t + a_{t+1} * G_{t+1}            (a_L G_L := dh_last, else 0)
    q_t  = G_t * a_t * h_{t-1}
    d delta_t = sum_n (q_t * A + G_t * B_t * x_t)
    dx_t      = ds_t * D + delta_t * sum_n G_t * B_t
    dA        = sum_{b,t} q_t * delta_t
    dB_t[n]   = sum_d G_t * delta_t * x_t
    dC_t[n]   = sum_d ds_t * h_t
    dD        = sum_{b,t} ds_t * x_t
    dh0       = a_0 * G_0

The backward keeps float64 copies of the state every ``segment`` steps and
recomputes the states of one segment at a time while walking backwards; the
recomputation repeats the same float64 operations in the same order, so the
values are those of a full stored history.
"""

from __future__ import annotations

import numpy as np


def _sigmoid(z: np.ndarray) -> np.ndarray:
    return 1.0 / (1.0 + np.exp(-z))


def _step(h: np.ndarray, delta_t: np.ndarray, x_t: np.ndarray, B_t: np.ndarray, A: np.ndarray):
    """One step of the recurrence. h [B,D,N], delta_t/x_t [B,D], B_t [B,N], A [D,N]."""
    a = np.exp(delta_t[:, :, None] * A[None, :, :])
    h_new = a * h + (delta_t * x_t)[:, :, None] * B_t[:, None, :]
    return a, h_new


def scan_fwd_ref(x, delta, A, Bm, Cm, Dv, z, h0=None, chunk: int | None = None):
    """Forward scan. Returns (y [B,L,D], h_last [B,D,N], ckpt [B,ceil(L/chunk),D,N] or None)."""
    x, delta, z = (np.asarray(v, np.float64) for v in (x, delta, z))
    A, Bm, Cm, Dv = (np.asarray(v, np.float64) for v in (A, Bm, Cm, Dv))
    Bsz, L, D = x.shape
    N = A.shape[1]
    h = np.zeros((Bsz, D, N)) if h0 is None else np.array(h0, dtype=np.float64, copy=True)
    y = np.empty((Bsz, L, D))
    ckpt = None
    if chunk:
        ckpt = np.empty((Bsz, -(-L // chunk), D, N))
    for t in range(L):
        if chunk and t % chunk == 0:
            ckpt[:, t // chunk] = h
        _, h = _step(h, delta[:, t], x[:, t], Bm[:, t], A)
        s = np.sum(h * Cm[:, t, None, :], axis=-1) + Dv[None, :] * x[:, t]
        y[:, t] = s * (z[:, t] * _sigmoid(z[:, t]))
    return y, h, ckpt


def delta_softplus_ref(delta_raw, dt_bias=None, softplus: bool = True):
    """The discretisation step in front of the scan: delta = softplus(raw + dt_bias)
    (softplus(v) = log(1 + e^v), evaluated as log(e^0 + e^v) by numpy.logaddexp),
    or raw + dt_bias without the softplus.  dt_bias [D] or None (zero)."""
    v = np.asarray(delta_raw, np.float64)
    if dt_bias is not None:
        v = v + np.asarray(dt_bias, np.float64)
    return np.logaddexp(0.0, v) if softplus else v


def scan_fwd_fused_ref(x, delta_raw, A, Bm, Cm, Dv, z, dt_bias=None, softplus: bool = True, h0=None,
                       chunk: int | None = None):
    """scan_fwd_ref on delta = delta_softplus_ref(delta_raw, dt_bias, softplus)."""
    return scan_fwd_ref(x, delta_softplus_ref(delta_raw, dt_bias, softplus), A, Bm, Cm, Dv, z, h0=h0, chunk=chunk)


def scan_bwd_fused_ref(x, delta_raw, A, Bm, Cm, Dv, z, dy, dt_bias=None, softplus: bool = True, h0=None,
                       dh_last=None):
    """Gradient through the fused discretisation: scan_bwd_ref on the transformed
    delta, then the chain rule into the raw delta (softplus' = sigmoid) and the
    bias (d dt_bias[d] = sum over b, t of that raw-delta gradient).  Returns the
    scan_bwd_ref dict with 'ddelta' replaced and 'd_dt_bias' added."""
    v = np.asarray(delta_raw, np.float64)
    if dt_bias is not None:
        v = v + np.asarray(dt_bias, np.float64)
    delta = np.logaddexp(0.0, v) if softplus else v
    g = dict(scan_bwd_ref(x, delta, A, Bm, Cm, Dv, z, dy, h0=h0, dh_last=dh_last))
    if softplus:
        g["ddelta"] = g["ddelta"] * _sigmoid(v)
    g["d_dt_bias"] = np.sum(g["ddelta"], axis=(0, 1))
    return g


def scan_step_ref(h, x_t, delta_t, A, B_t, C_t, Dv, z_t):
    """One recurrent step for B sequences (the single-step updater of the
    rustytorch mamba_step_equivalence.rs test): h [B,D,N], x_t/delta_t/z_t [B,D],
    B_t/C_t [B,N].  Returns (h_new [B,D,N], y_t [B,D])."""
    h = np.asarray(h, np.float64)
    x_t, delta_t, z_t = (np.asarray(v, np.float64) for v in (x_t, delta_t, z_t))
    A, B_t, C_t, Dv = (np.asarray(v, np.float64) for v in (A, B_t, C_t, Dv))
    _, h_new = _step(h, delta_t, x_t, B_t, A)
    s = np.sum(h_new * C_t[:, None, :], axis=-1) + Dv[None, :] * x_t
    return h_new, s * (z_t * _sigmoid(z_t))


def scan_bwd_ref(x, delta, A, Bm, Cm, Dv, z, dy, h0=None, dh_last=None, segment: int | None = None):
    """Reverse-mode gradient of sum(y * dy) + sum(h_last * dh_last) w.r.t. every input of ``scan_fwd_ref``.

    ``dh_last`` [B,D,N] (optional) is the gradient arriving on the final state from
    a later segment; it lets a sequence split in two be differentiated piecewise.
    Returns a dict with dx, ddelta, dz [B,L,D]; dA [D,N]; dB, dC [B,L,N]; dD [D];
    dh0 [B,D,N] (the gradient w.r.t. the initial state, zeros-based when h0 is None).
    """
    x, delta, z, dy = (np.asarray(v, np.float64) for v in (x, delta, z, dy))
    A, Bm, Cm, Dv = (np.asarray(v, np.float64) for v in (A, Bm, Cm, Dv))
    Bsz, L, D = x.shape
    N = A.shape[1]
    if segment is None:
        # keep one segment of float64 states at or below ~256 MB
        segment = max(1, min(L, (256 << 20) // max(1, Bsz * D * N * 8)))

    # forward pass: store the state entering every segment
    h = np.zeros((Bsz, D, N)) if h0 is None else np.array(h0, dtype=np.float64, copy=True)
    seg_starts = list(range(0, L, segment))
    seg_state = {}
    for t in range(L):
        if t % segment == 0:
            seg_state[t] = h
        _, h = _step(h, delta[:, t], x[:, t], Bm[:, t], A)

    dx = np.empty((Bsz, L, D))
    ddelta = np.empty((Bsz, L, D))
    dz = np.empty((Bsz, L, D))
    dB = np.empty((Bsz, L, N))
    dC = np.empty((Bsz, L, N))
    dA = np.zeros((D, N))
    dD = np.zeros(D)
    # G = dL/dh_t carried backwards; past the last step G_L * a_L stands for dh_last
    if dh_last is None:
        G = np.zeros((Bsz, D, N))
        a_next = np.zeros((Bsz, D, N))
    else:
        G = np.array(dh_last, dtype=np.float64, copy=True)
        a_next = np.ones((Bsz, D, N))

    for t0 in reversed(seg_starts):
        t1 = min(L, t0 + segment)
        # recompute the states of this segment: hist[i] = h_{t0+i-1}
        hist = [seg_state[t0]]
        avals = []
        for t in range(t0, t1):
            a, hn = _step(hist[-1], delta[:, t], x[:, t], Bm[:, t], A)
            avals.append(a)
            hist.append(hn)
        for t in reversed(range(t0, t1)):
            i = t - t0
            a_t, h_prev, h_t = avals[i], hist[i], hist[i + 1]
            x_t, d_t, z_t, dy_t = x[:, t], delta[:, t], z[:, t], dy[:, t]
            B_t, C_t = Bm[:, t], Cm[:, t]
            sig = _sigmoid(z_t)
            s_t = np.sum(h_t * C_t[:, None, :], axis=-1) + Dv[None, :] * x_t
            ds = dy_t * (z_t * sig)
            dz[:, t] = dy_t * s_t * sig * (1.0 + z_t * (1.0 - sig))
            G = ds[:, :, None] * C_t[:, None, :] + a_next * G
            q = G * a_t * h_prev
            GB = np.sum(G * B_t[:, None, :], axis=-1)
            ddelta[:, t] = np.sum(q * A[None, :, :], axis=-1) + GB * x_t
            dx[:, t] = ds * Dv[None, :] + d_t * GB
            dA += np.sum(q * d_t[:, :, None], axis=0)
            dB[:, t] = np.sum(G * (d_t * x_t)[:, :, None], axis=1)
            dC[:, t] = np.sum(ds[:, :, None] * h_t, axis=1)
            dD += np.sum(ds * x_t, axis=0)
            a_next = a_t
    dh0 = a_next * G
    return {"dx": dx, "ddelta": ddelta, "dz": dz, "dA": dA, "dB": dB, "dC": dC, "dD": dD, "dh0": dh0}
