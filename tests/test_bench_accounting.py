"""The algorithmic bytes bench.py divides by (CPU only).

Worked by hand for each workload at one checkpoint per 256 steps, with
E = B*L*D elements and e the activation bytes:
  scan forward  = E*4e + B*L*N*2e + C          (read x, delta, z; write y; read B_t, C_t; write checkpoints)
  scan backward = E*(4e + 12) + B*L*N*(2e + 8) + C   (read x, delta, z, dy; write dx, ddelta, dz fp32;
                                                      read B_t, C_t; write dB, dC fp32; read checkpoints)
  C = B*D*(ceil(L/256) - 1)*N*4; bench also counts the parameter bytes (A and D read by both passes, dA and
  dD read and written by the backward: 4*(D*N + D)*4 bytes, 1.1 MB at D = 4096), which the totals below leave out.
  mamba130m (fp32):  E = 25.17 M: 1124.6 MB      mamba1p4b (bf16): E = 33.55 M: 956.3 MB
  short (fp32):      E = 8.39 M:   419.4 MB      long (bf16, chunk 256): 960.2 MB
"""
import pytest

from workloads import CONFIGS


@pytest.mark.parametrize("name,mb", [("mamba130m", 1124.6), ("mamba1p4b", 956.3), ("short", 419.4), ("long", 960.2)])
def test_scan_bytes_per_step(name, mb):
    import bench
    a = bench.algorithmic_bytes(CONFIGS[name], 256)
    got = (a["scan_fwd"] + a["scan_bwd"]) / 1e6
    assert abs(got - mb) <= 1.5, (name, got, mb)


def test_side_kernel_bytes():
    import bench
    a = bench.algorithmic_bytes(CONFIGS["mamba1p4b"], 8)
    E = 4 * 2048 * 4096
    assert abs(a["conv1d_bwd"] - E * (4 + 2 + 4)) < 1e6          # read g fp32, x bf16; write dx fp32
    assert abs(a["rmsnorm_bwd"] - 8192 * 2048 * (2 + 2 + 4)) < 1e6  # read dy, x bf16; write dx fp32


def test_checkpoint_overhead():
    """At a checkpoint every 8 steps the 1.4B layer's scan writes (forward) and reads (backward) all
    2048/8 = 256 checkpoints of B*D*N fp32 = 1 MiB each (268.4 MB); the count allows 2048/256 - 1 = 7 (7.3 MB)."""
    import bench
    wl = CONFIGS["mamba1p4b"]
    got = bench.checkpoint_overhead_bytes(wl, 8)
    assert got == 4 * 4096 * 16 * 4 * (256 - 7)
    assert bench.checkpoint_overhead_bytes(CONFIGS["long"], 256) == 1 * 2048 * 16 * 4  # only the first
