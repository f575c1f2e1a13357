"""Pins for the conv1d-backward and RMSNorm-backward oracles (CPU only)."""

import numpy as np
import pytest

from oracle import (conv1d_causal_bwd_ref, conv1d_causal_fwd_ref, conv1d_step_bwd_ref, rmsnorm_bwd_ref,
                    rmsnorm_fwd_ref)
from tests._util import max_rel_err

# ------------------------------------------------------------------ conv1d


def _conv_inputs(rng, B=2, L=9, D=3, K=4):
    return rng.standard_normal((B, L, D)), rng.standard_normal((D, K)), rng.standard_normal(D), rng.standard_normal((B, L, D))


@pytest.mark.parametrize("K", [1, 2, 3, 4])
def test_conv_forward_matches_numpy_convolve(K):
    rng = np.random.default_rng(20 + K)
    x, w, b, _ = _conv_inputs(rng, K=K)
    out = conv1d_causal_fwd_ref(x, w, b)
    for bb in range(2):
        for d in range(3):
            ref = np.convolve(x[bb, :, d], w[d, ::-1])[: x.shape[1]] + b[d]
            np.testing.assert_allclose(out[bb, :, d], ref, rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("K", [1, 2, 3, 4])
def test_conv_backward_is_toeplitz_transpose(K):
    """dx = T^T dout with T the causal Toeplitz matrix of each channel's filter (scipy.linalg.toeplitz)."""
    scipy_linalg = pytest.importorskip("scipy.linalg")
    rng = np.random.default_rng(30 + K)
    x, w, _, dout = _conv_inputs(rng, L=11, K=K)
    dx, dw, db = conv1d_causal_bwd_ref(dout, x, w)
    L = x.shape[1]
    for d in range(3):
        col = np.zeros(L)
        col[:K] = w[d, ::-1]  # out[t] = sum_j T[t, j] x[j], T[t, t-i] = w[K-1-i]
        T = scipy_linalg.toeplitz(col, np.zeros(L))
        for bb in range(2):
            np.testing.assert_allclose(dx[bb, :, d], T.T @ dout[bb, :, d], rtol=1e-12, atol=1e-13)
        # dw[d, k] = correlation of dout with x delayed by K-1-k
        for k in range(K):
            ref = sum(np.correlate(dout[bb, :, d], np.concatenate([np.zeros(K - 1 - k), x[bb, : L - (K - 1 - k), d]]))[0]
                      for bb in range(2))
            np.testing.assert_allclose(dw[d, k], ref, rtol=1e-12)
    np.testing.assert_allclose(db, dout.sum(axis=(0, 1)), rtol=1e-13)


def test_conv_backward_finite_differences():
    rng = np.random.default_rng(40)
    x, w, b, dout = _conv_inputs(rng, B=2, L=6, D=2, K=3)
    dx, dw, db = conv1d_causal_bwd_ref(dout, x, w)
    loss = lambda: float(np.sum(conv1d_causal_fwd_ref(x, w, b) * dout))
    for arr, g in ((x, dx), (w, dw), (b, db)):
        fd = np.empty_like(arr)
        for idx in np.ndindex(arr.shape):
            v0 = arr[idx]
            arr[idx] = v0 + 1e-6
            lp = loss()
            arr[idx] = v0 - 1e-6
            lm = loss()
            arr[idx] = v0
            fd[idx] = (lp - lm) / 2e-6
        assert max_rel_err(g, fd) < 1e-8


@pytest.mark.parametrize("K", [1, 4])
def test_conv_full_sequence_equals_summed_step_formula(K):
    """dw, db are the per-step contributions of the pages' step function summed over time;
    with K=1 the input gradient is the step function's newest-tap gradient."""
    rng = np.random.default_rng(50 + K)
    x, w, _, dout = _conv_inputs(rng, B=2, L=8, D=3, K=K)
    dx, dw, db = conv1d_causal_bwd_ref(dout, x, w)
    dw_s = np.zeros_like(w)
    db_s = np.zeros(3)
    for bb in range(2):
        state = np.zeros((3, K))
        for t in range(x.shape[1]):
            state = np.concatenate([state[:, 1:], x[bb, t][:, None]], axis=1)  # newest input at K-1
            dx_t = conv1d_step_bwd_ref(dout[bb, t], state, w, dw_s, db_s)
            if K == 1:
                np.testing.assert_allclose(dx[bb, t], dx_t, rtol=1e-14)
    np.testing.assert_allclose(dw, dw_s, rtol=1e-12)
    np.testing.assert_allclose(db, db_s, rtol=1e-12)


# ----------------------------------------------------------------- RMSNorm


def test_rmsnorm_backward_finite_differences():
    """FD through y = x*scale/sqrt(mean(x^2)+eps), rms recomputed from x, for dx and dscale."""
    rng = np.random.default_rng(60)
    R, H, eps = 3, 7, 1e-5
    x = rng.standard_normal((R, H))
    scale = 1 + 0.1 * rng.standard_normal(H)
    dy = rng.standard_normal((R, H))
    _, rms = rmsnorm_fwd_ref(x, scale, eps)
    dx, dscale = rmsnorm_bwd_ref(dy, x, scale, rms)
    loss = lambda: float(np.sum(rmsnorm_fwd_ref(x, scale, eps)[0] * dy))
    for arr, g in ((x, dx), (scale, dscale)):
        fd = np.empty_like(arr)
        for idx in np.ndindex(arr.shape):
            v0 = arr[idx]
            arr[idx] = v0 + 1e-6
            lp = loss()
            arr[idx] = v0 - 1e-6
            lm = loss()
            arr[idx] = v0
            fd[idx] = (lp - lm) / 2e-6
        assert max_rel_err(g, fd) < 1e-8


def test_rmsnorm_scale_invariance():
    """With eps=0, y is invariant to scaling each row of x, so sum_i x_i dx_i = 0 per row."""
    rng = np.random.default_rng(61)
    x = rng.standard_normal((5, 33))
    scale = 1 + 0.1 * rng.standard_normal(33)
    dy = rng.standard_normal((5, 33))
    _, rms = rmsnorm_fwd_ref(x, scale, 0.0)
    dx, _ = rmsnorm_bwd_ref(dy, x, scale, rms)
    np.testing.assert_allclose(np.sum(x * dx, axis=1), 0.0, atol=1e-12)


def test_rmsnorm_rows_independent_and_dscale_sums_rows():
    rng = np.random.default_rng(62)
    x = rng.standard_normal((6, 10))
    scale = rng.standard_normal(10)
    dy = rng.standard_normal((6, 10))
    rms = np.sqrt(np.mean(x * x, 1) + 1e-5)
    dx, dscale = rmsnorm_bwd_ref(dy, x, scale, rms)
    parts = [rmsnorm_bwd_ref(dy[i : i + 1], x[i : i + 1], scale, rms[i : i + 1]) for i in range(6)]
    np.testing.assert_array_equal(np.concatenate([p[0] for p in parts]), dx)
    np.testing.assert_allclose(sum(p[1] for p in parts), dscale, rtol=1e-13)


# ------------------------------------------------------------------ forward producers (conv -> SiLU, RMSNorm)


def test_silu_matches_scipy_expit():
    """silu(v) = v * sigmoid(v), checked against SciPy's logistic function."""
    special = pytest.importorskip("scipy.special")
    from oracle import silu_ref
    v = np.concatenate([np.linspace(-60, 60, 1201), [-1e-8, 0.0, 1e-8]])
    np.testing.assert_allclose(silu_ref(v), v * special.expit(v), rtol=1e-14, atol=1e-300)


def test_silu_limits():
    from oracle import silu_ref
    assert silu_ref(0.0) == 0.0
    assert abs(silu_ref(40.0) - 40.0) < 1e-14 * 40
    assert abs(silu_ref(-40.0)) < 1e-15
    # odd part: silu(v) - silu(-v) = v
    v = np.linspace(-5, 5, 41)
    np.testing.assert_allclose(silu_ref(v) - silu_ref(-v), v, atol=1e-14)


def test_conv_silu_is_silu_of_conv():
    from oracle import conv1d_causal_silu_fwd_ref, silu_ref
    rng = np.random.default_rng(70)
    x, w, b, _ = _conv_inputs(rng, B=2, L=11, D=5, K=4)
    out = conv1d_causal_fwd_ref(x, w, b)
    np.testing.assert_array_equal(conv1d_causal_silu_fwd_ref(x, w, b), silu_ref(out))


def test_rmsnorm_fwd_rms_is_scaled_euclidean_norm():
    """eps = 0: rms is |x_r| / sqrt(H) (numpy.linalg.norm), and y with unit scale has unit RMS."""
    rng = np.random.default_rng(71)
    x = rng.standard_normal((7, 40))
    y, rms = rmsnorm_fwd_ref(x, np.ones(40), 0.0)
    np.testing.assert_allclose(rms, np.linalg.norm(x, axis=1) / np.sqrt(40), rtol=1e-14)
    np.testing.assert_allclose(np.sqrt(np.mean(y * y, axis=1)), 1.0, rtol=1e-14)
    scale = 1 + 0.1 * rng.standard_normal(40)
    y2, _ = rmsnorm_fwd_ref(x, scale, 0.0)
    np.testing.assert_allclose(y2, y * scale[None, :], rtol=1e-14)


def test_rmsnorm_fwd_eps_enters_under_the_root():
    x = np.array([[3.0, 4.0]])  # mean square 12.5
    _, rms = rmsnorm_fwd_ref(x, np.ones(2), 0.5)
    assert rms[0] == np.sqrt(13.0)


def test_dsilu_matches_scipy_expit_derivative():
    """silu'(v) = expit(v) + v expit(v) (1 - expit(v)), from SciPy's logistic function."""
    special = pytest.importorskip("scipy.special")
    from oracle import dsilu_ref
    v = np.linspace(-30, 30, 601)
    e = special.expit(v)
    np.testing.assert_allclose(dsilu_ref(v), e + v * e * (1 - e), rtol=1e-13, atol=1e-300)


def test_conv_silu_backward_finite_differences():
    """Central differences of sum(silu(conv(x, w) + b) * dact) in x, w and the bias."""
    from oracle import conv1d_causal_silu_bwd_ref, conv1d_causal_silu_fwd_ref
    rng = np.random.default_rng(72)
    x, w, b, dact = _conv_inputs(rng, B=2, L=7, D=3, K=4)
    dx, dw, db = conv1d_causal_silu_bwd_ref(dact, x, w, b)
    loss = lambda: float(np.sum(conv1d_causal_silu_fwd_ref(x, w, b) * dact))
    for arr, g in ((x, dx), (w, dw), (b, db)):
        fd = np.empty_like(arr)
        for idx in np.ndindex(arr.shape):
            v0 = arr[idx]
            arr[idx] = v0 + 1e-6
            lp = loss()
            arr[idx] = v0 - 1e-6
            lm = loss()
            arr[idx] = v0
            fd[idx] = (lp - lm) / 2e-6
        assert max_rel_err(g, fd) < 1e-8


@pytest.mark.parametrize("K,silu", [(1, False), (3, True), (4, False), (4, True)])
def test_conv_step_chain_equals_sequence(K, silu):
    """L single conv steps from a zero shift register reproduce the full-sequence conv (+SiLU)."""
    from oracle import conv1d_causal_silu_fwd_ref, conv1d_step_fwd_ref
    rng = np.random.default_rng(73 + K)
    x, w, b, _ = _conv_inputs(rng, B=2, L=8, D=3, K=K)
    ref = (conv1d_causal_silu_fwd_ref if silu else conv1d_causal_fwd_ref)(x, w, b)
    state = np.zeros((2, 3, K))
    for t in range(8):
        state, out = conv1d_step_fwd_ref(state, x[:, t], w, b, silu=silu)
        np.testing.assert_allclose(out, ref[:, t], rtol=1e-14, atol=1e-14)
    np.testing.assert_array_equal(state[:, :, -1], x[:, -1])
