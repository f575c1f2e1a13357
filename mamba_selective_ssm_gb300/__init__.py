"""GB300-native Mamba selective scan: forward and backward of the diagonal
selective SSM, the depthwise causal conv1d (+SiLU) and RMSNorm forward and
backward, as hand-written sm_103a CUDA kernels behind the C ABI in
include/ssscan.h.

The Python layer only checks arguments, allocates outputs with PyTorch and
calls the library on the current CUDA stream.
"""

from ._build import build
from ._capi import SSError, load
from .ops import (conv1d_causal_bwd, conv1d_causal_fwd, conv1d_causal_silu_bwd, conv1d_causal_step, count_nonfinite, device_status, num_chunks, rmsnorm_bwd, rmsnorm_fwd,
                  scan_bwd_workspace_size, scan_fwd_workspace_size, ss_scan_bwd, ss_scan_bwd_summary, ss_scan_carries,
                  ss_scan_fwd, ss_scan_fwd_summary, ss_scan_step)

__all__ = [
    "build", "load", "SSError", "ss_scan_fwd", "ss_scan_bwd", "scan_fwd_workspace_size", "scan_bwd_workspace_size",
    "ss_scan_step", "ss_scan_fwd_summary", "ss_scan_bwd_summary", "ss_scan_carries", "conv1d_causal_step", "conv1d_causal_fwd", "conv1d_causal_bwd", "conv1d_causal_silu_bwd", "rmsnorm_fwd", "rmsnorm_bwd", "num_chunks", "count_nonfinite", "device_status",
]
