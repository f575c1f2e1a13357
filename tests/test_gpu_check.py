"""ss_count_nonfinite on the GPU: exact counts of NaN / +-Inf planted at known
places (vector body and ragged tail, both dtypes), zero on finite data."""
import numpy as np
import pytest

from gpu_util import ss_module

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ss():
    return ss_module()


@pytest.mark.parametrize("n", [0, 1, 7, 8, 9, 1000, 4099, 10_000_003])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_count_nonfinite_matches_numpy(ss, n, dtype):
    import torch
    rng = np.random.default_rng(n + (1 if dtype == "bf16" else 0))
    a = rng.standard_normal(n).astype(np.float32)
    k = min(n, 37)
    if k:
        idx = rng.choice(n, k, replace=False)
        a[idx] = rng.choice(np.array([np.nan, np.inf, -np.inf], dtype=np.float32), k)
        a[n - 1] = np.nan  # the last element sits in the ragged tail unless n is a multiple of the vector
    t = torch.from_numpy(a)
    if dtype == "bf16":
        t = t.to(torch.bfloat16)
    expect = int((~torch.isfinite(t.float())).sum())
    assert ss.count_nonfinite(t.cuda()) == expect


def test_count_nonfinite_finite_gradients(ss):
    import torch
    g = torch.randn(4, 2048, 4096, device="cuda") * 1e30  # large but finite
    assert ss.count_nonfinite(g) == 0
    g[3, 2047, 4095] = float("inf")
    g[0, 0, 0] = float("nan")
    assert ss.count_nonfinite(g) == 2
