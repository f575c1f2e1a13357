"""Float64 CPU oracle for the selective-scan forward/backward, the depthwise causal
conv1d backward and the RMSNorm backward.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call, link
or execute this package: only the test-suite, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` use it.  It shares no code, header, table
or helper with the CUDA library; both sides are fed by the seeded generators
in ``workloads/``.

Each function is the plain definition of what the method computes, written
out in NumPy float64 with a sequential loop over time, no blocking, fusion or
reordering beyond what the definition states:

* ``scan.scan_fwd_ref`` / ``scan.scan_bwd_ref`` — the diagonal selective SSM
  ``h_t = exp(delta_t*A) * h_{t-1} + delta_t*B_t*x_t``,
  ``y_t = (C_t . h_t + D*x_t) * silu(z_t)`` and its reverse-mode gradient
  (backpropagation through time through the SSM state: the "sequential scan
  reverse-pass" of the rustytorch ``backward_cuda`` commit message);
* ``conv1d.conv1d_causal_bwd_ref`` / ``conv1d.conv1d_step_bwd_ref`` — the
  depthwise causal conv1d backward, full-sequence and per-step (mamba-rs
  ``backward_ops.rs``, ``backward_conv1d_step``);
* ``rmsnorm.rmsnorm_bwd_ref`` — the RMSNorm backward (mamba-rs
  ``backward_ops.rs``, ``backward_rms_norm``).

Pins (tests/test_oracle_*.py, CPU only): central finite differences, the L=1
closed form, the A->0 cumulative-sum limit, the constant-input geometric
series, a bidiagonal linear solve, step/segment equivalence, numpy.correlate,
and RMSNorm scale invariance.
"""

from .conv1d import (conv1d_causal_bwd_ref, conv1d_causal_fwd_ref, conv1d_causal_silu_bwd_ref,
                     conv1d_causal_silu_fwd_ref, conv1d_step_bwd_ref, conv1d_step_fwd_ref, dsilu_ref, silu_ref)
from .rmsnorm import rmsnorm_bwd_ref, rmsnorm_fwd_ref
from .scan import (delta_softplus_ref, scan_bwd_fused_ref, scan_bwd_ref, scan_fwd_fused_ref, scan_fwd_ref,
                   scan_step_ref)

__all__ = [
    "scan_fwd_ref", "scan_bwd_ref", "scan_step_ref", "conv1d_step_fwd_ref", "delta_softplus_ref",
    "scan_fwd_fused_ref", "scan_bwd_fused_ref",
    "conv1d_causal_fwd_ref", "conv1d_causal_silu_fwd_ref", "silu_ref", "dsilu_ref", "conv1d_causal_bwd_ref",
    "conv1d_causal_silu_bwd_ref", "conv1d_step_bwd_ref",
    "rmsnorm_fwd_ref", "rmsnorm_bwd_ref",
]
