"""rmsnorm_bwd_noalloc: the RMSNorm backward for callers that cannot allocate
device memory (its scratch is a fixed array inside the library).  Called
through the C ABI, twice in a row, and compared with rmsnorm_bwd, which takes
a caller-allocated workspace, and with the float64 oracle.  This file is
collected last on purpose."""

import ctypes

import numpy as np
import pytest

from oracle import rmsnorm_bwd_ref
from tests._util import TOL, assert_close
from tests.gpu_util import dev, host, ss_module
from workloads import CONFIGS, make_rmsnorm_inputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("rows,dim,dtype", [(3000, 2048, "bf16"), (517, 768, "f32"), (64, 8192, "f32")])
def test_noalloc_matches_allocating_entry_point(rows, dim, dtype):
    ss_module()
    import torch
    from mamba_selective_ssm_gb300 import _capi

    lib = _capi.load()
    wl = CONFIGS["tiny"].with_(dtype=dtype)
    r = make_rmsnorm_inputs(wl, seed=rows, rows=rows, dim=dim)
    dy, x = dev(r["dy"], dtype), dev(r["x"], dtype)
    scale, rms = dev(r["scale"]), dev(r["rms"])
    sdt = _capi.SS_BF16 if dtype == "bf16" else _capi.SS_F32
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)

    ref_dx = torch.empty((rows, dim), device="cuda")
    ref_ds = torch.zeros(dim, device="cuda")
    ws = torch.empty(lib.rmsnorm_bwd_workspace_size(rows, dim), device="cuda", dtype=torch.uint8)
    assert lib.rmsnorm_bwd(p(dy), p(x), p(scale), p(rms), p(ref_dx), p(ref_ds), rows, dim, sdt, p(ws), ws.numel(),
                           stream) == 0
    odx, ods = rmsnorm_bwd_ref(r["dy"], r["x"], r["scale"], r["rms"])
    for _ in range(2):  # the shared scratch keeps the previous call's partials
        dx = torch.full((rows, dim), float("nan"), device="cuda")
        ds = torch.zeros(dim, device="cuda")
        assert lib.rmsnorm_bwd_noalloc(p(dy), p(x), p(scale), p(rms), p(dx), p(ds), rows, dim, sdt, stream) == 0
        torch.cuda.synchronize()
        assert_close(host(dx), host(ref_dx), TOL["f32"], "dx")
        assert_close(host(ds), host(ref_ds), TOL["f32"], "dscale")
        # and against the float64 oracle itself, at the parity bar of the other RMSNorm tests
        assert_close(host(dx), odx, TOL["f32"], "dx vs oracle")
        assert_close(host(ds), ods, TOL["f32"], "dscale vs oracle")


def test_noalloc_rejects_dim_beyond_its_scratch():
    ss_module()
    from mamba_selective_ssm_gb300 import _capi

    lib = _capi.load()
    fake = [ctypes.c_void_p(0x10000 + 256 * i) for i in range(6)]
    assert lib.rmsnorm_bwd_noalloc(*fake, 16, 8200, _capi.SS_F32, None) == _capi.SS_ERR_DIM
