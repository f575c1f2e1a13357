"""Seeded synthetic inputs shared by the oracle tests, the GPU parity tests and the bench.

This package only draws random numbers in the shapes and distributions of the
Mamba-shaped workloads; it holds none of the selective-scan, conv1d or RMSNorm
backward arithmetic.  Both the float64 oracle and the CUDA path consume what it
returns, and neither imports the other.
"""

from .synth import (CONFIGS, RMS_EPS, Workload, get_config, make_conv_inputs, make_rmsnorm_inputs, make_scan_inputs,
                    round_to)

__all__ = ["CONFIGS", "RMS_EPS", "Workload", "get_config", "make_scan_inputs", "make_conv_inputs",
           "make_rmsnorm_inputs", "round_to"]
