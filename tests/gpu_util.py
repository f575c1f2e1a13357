"""Helpers for the GPU parity tests: build/load the library, move seeded inputs
to the device in the workload dtype, and run the oracle on the same values."""

import numpy as np
import pytest

TORCH_DT = {"f32": "float32", "bf16": "bfloat16"}


def ss_module():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mamba_selective_ssm_gb300 as ss
    ss.build()
    ss.load()
    return ss


def dev(a, dtype="f32"):
    """float64 numpy (already on the dtype's grid) -> CUDA tensor of that dtype (exact)."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float64))
    return t.to(getattr(torch, TORCH_DT[dtype])).cuda().contiguous()


def host(t):
    return t.detach().to("cpu").double().numpy()


def scan_inputs_on_device(inp, dtype):
    return {
        "x": dev(inp["x"], dtype), "delta": dev(inp["delta"], dtype), "z": dev(inp["z"], dtype),
        "Bm": dev(inp["Bm"], dtype), "Cm": dev(inp["Cm"], dtype), "dy": dev(inp["dy"], dtype),
        "A": dev(inp["A"]), "Dv": dev(inp["Dv"]),
    }


def run_gpu_scan(ss, d, chunk, h0=None, dh_last=None, dA0=None, dD0=None):
    y, ckpt, h_last = ss.ss_scan_fwd(d["x"], d["delta"], d["A"], d["Bm"], d["Cm"], d["Dv"], d["z"], h0=h0, chunk=chunk)
    g = ss.ss_scan_bwd(d["x"], d["delta"], d["A"], d["Bm"], d["Cm"], d["Dv"], d["z"], ckpt, d["dy"], dh_last=dh_last,
                       chunk=chunk, dA=dA0, dD=dD0)
    return y, ckpt, h_last, g
