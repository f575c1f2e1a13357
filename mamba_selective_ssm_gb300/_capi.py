"""ctypes declarations of libssscan.so (include/ssscan.h).

Only argument marshalling lives here; every step of the computation runs in
the library's CUDA kernels.  Loading fails loudly when the library is missing.
"""

from __future__ import annotations

import ctypes
import os

from . import _build

SS_OK = 0
SS_ERR_NULL = -1
SS_ERR_DIM = -2
SS_ERR_UNSUPPORTED = -3
SS_ERR_ALIGN = -4
SS_ERR_WORKSPACE = -5
SS_ERR_CUDA = -6
SS_ERR_DEVICE = -7
SS_F32 = 0
SS_BF16 = 1

_vp = ctypes.c_void_p
_i = ctypes.c_int
_sz = ctypes.c_size_t

# name -> (restype, argtypes), in the order of include/ssscan.h
SIGNATURES = {
    "ss_strerror": (ctypes.c_char_p, [_i]),
    "ss_scan_num_chunks": (_i, [_i, _i]),
    "ss_scan_fwd_workspace_size": (_sz, [_i] * 6),
    "ss_scan_fwd": (_i, [_vp] * 11 + [_i] * 6 + [_vp, _i, _vp, _sz, _vp]),
    "ss_scan_bwd_workspace_size": (_sz, [_i] * 6),
    "ss_scan_bwd": (_i, [_vp] * 18 + [_i] * 6 + [_vp, _i, _vp, _vp, _sz, _vp]),
    "ss_scan_fwd_summary": (_i, [_vp] * 6 + [_i] * 5 + [_vp, _i, _vp]),
    "ss_scan_bwd_summary": (_i, [_vp] * 7 + [_i] * 5 + [_vp, _i, _vp]),
    "ss_scan_carries": (_i, [_vp] * 5 + [_i] * 5 + [_vp]),
    "conv1d_causal_bwd_workspace_size": (_sz, [_i] * 4),
    "conv1d_causal_bwd": (_i, [_vp] * 6 + [_i] * 5 + [_vp, _sz, _vp]),
    "conv1d_causal_silu_bwd": (_i, [_vp] * 7 + [_i] * 5 + [_vp, _sz, _vp]),
    "rmsnorm_bwd_workspace_size": (_sz, [_i, _i]),
    "rmsnorm_bwd": (_i, [_vp] * 6 + [_i] * 3 + [_vp, _sz, _vp]),
    "rmsnorm_bwd_noalloc": (_i, [_vp] * 6 + [_i] * 3 + [_vp]),
    "conv1d_causal_fwd": (_i, [_vp] * 4 + [_i] * 6 + [_vp]),
    "rmsnorm_fwd": (_i, [_vp, _vp, ctypes.c_float, _vp, _vp, _i, _i, _i, _vp]),
    "ss_scan_step": (_i, [_vp] * 9 + [_i] * 4 + [_vp]),
    "conv1d_causal_step": (_i, [_vp] * 5 + [_i] * 5 + [_vp]),
    "ss_count_nonfinite_workspace_size": (_sz, []),
    "ss_count_nonfinite": (_i, [_vp, _sz, _i, _vp, _vp, _sz, _vp]),
    "ss_device_status": (_i, [_vp]),
}

_LIB = None


class SSError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {strerror(code)} (status {code})")


def load(path: str | None = None):
    """Load libssscan.so (built in-tree by _build.build())."""
    global _LIB
    if _LIB is not None and path is None:
        return _LIB
    path = path or _build.LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(
            f"libssscan.so not found at {path}; build it with mamba_selective_ssm_gb300._build.build() "
            "(there is no fallback implementation)")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path == _build.LIB_PATH:
        _LIB = lib
    return lib


def strerror(code: int) -> str:
    return load().ss_strerror(code).decode()


def check(code: int, where: str) -> None:
    if code != SS_OK:
        raise SSError(code, where)
