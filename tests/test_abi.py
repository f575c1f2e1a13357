"""The C ABI on the host: the library builds and loads, exports every symbol that
include/ssscan.h declares, and rejects bad arguments with the documented
status codes before touching the GPU (CPU only; no kernel is launched)."""

import ctypes
import os
import re
import shutil

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ssscan.h")


@pytest.fixture(scope="module")
def lib():
    if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
        pytest.skip("nvcc not available")
    from mamba_selective_ssm_gb300 import _build, _capi
    _build.build()
    return _capi.load()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", text, flags=re.M)) - {"defined"})


def test_header_declares_the_four_entry_points():
    names = _declared_functions()
    for n in ("ss_scan_fwd", "ss_scan_bwd", "conv1d_causal_bwd", "rmsnorm_bwd", "ss_strerror"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    from mamba_selective_ssm_gb300._capi import SIGNATURES
    names = _declared_functions()
    assert set(names) == set(SIGNATURES), (names, sorted(SIGNATURES))
    for n in names:
        assert hasattr(lib, n), n


def test_strerror_covers_codes(lib):
    for c in range(-7, 1):
        assert lib.ss_strerror(c) and b"unknown" not in lib.ss_strerror(c)
    assert b"unknown" in lib.ss_strerror(-99)


def _fake(addr=0x10000):
    return ctypes.c_void_p(addr)


def test_scan_fwd_validation(lib):
    from mamba_selective_ssm_gb300 import _capi as c
    p = [_fake(0x10000 + 256 * i) for i in range(11)]

    def call(ptrs=p, B=2, L=64, D=16, N=4, chunk=64, dtype=c.SS_F32):
        return lib.ss_scan_fwd(*ptrs, B, L, D, N, chunk, dtype, None, 0, None, 0, None)

    q = list(p)
    q[0] = None
    assert call(q) == c.SS_ERR_NULL
    q = list(p)
    q[7] = None  # h0 optional -> only later checks fail
    assert call(q, B=0) == c.SS_ERR_DIM
    assert call(B=0) == c.SS_ERR_DIM
    assert call(L=-1) == c.SS_ERR_DIM
    assert call(chunk=0) == c.SS_ERR_DIM
    assert call(N=5) == c.SS_ERR_UNSUPPORTED
    assert call(N=32) == c.SS_ERR_UNSUPPORTED
    assert call(dtype=7) == c.SS_ERR_UNSUPPORTED
    assert call(chunk=24) == c.SS_ERR_UNSUPPORTED
    assert call(D=12) == c.SS_ERR_ALIGN
    assert call(L=63, N=4, dtype=c.SS_BF16) == c.SS_ERR_ALIGN  # B_t rows of 8*63 bytes
    q = list(p)
    q[3] = _fake(0x10004)
    assert call(q) == c.SS_ERR_ALIGN


def test_scan_fwd_workspace(lib):
    """A small B*D cuts the sequence into segments, whose summaries need scratch;
    a layer with enough (batch row, channel) pairs needs none."""
    from mamba_selective_ssm_gb300 import _capi as c
    ws = lib.ss_scan_fwd_workspace_size(2, 64, 16, 4, 64, c.SS_F32)
    # end states [B, P, D, N] and sums of delta [B, P, D] for P = 64 / 16 segments
    assert ws >= 2 * 4 * 16 * 4 * 4 + 2 * 4 * 16 * 4
    assert lib.ss_scan_fwd_workspace_size(8, 2048, 4096, 16, 8, c.SS_BF16) == 0
    assert lib.ss_scan_fwd_workspace_size(2, 64, 16, 5, 64, c.SS_F32) == 0  # invalid N
    p = [_fake(0x10000 + 256 * i) for i in range(11)]
    f = lambda w, n: lib.ss_scan_fwd(*p, 2, 64, 16, 4, 64, c.SS_F32, None, 0, w, n, None)
    assert f(None, 0) == c.SS_ERR_WORKSPACE
    assert f(_fake(0x90000), ws - 1) == c.SS_ERR_WORKSPACE
    assert f(_fake(0x90008), ws) == c.SS_ERR_ALIGN


def test_scan_bwd_validation_and_workspace(lib):
    from mamba_selective_ssm_gb300 import _capi as c
    ws = lib.ss_scan_bwd_workspace_size(2, 64, 16, 4, 64, c.SS_F32)
    assert ws > 0
    # dB/dC partials per 64-channel tile + dA/dD partials per CTA row
    assert ws >= 1 * 2 * 64 * 2 * 4 * 4 + 2 * 16 * 4 * 4 + 2 * 16 * 4
    assert lib.ss_scan_bwd_workspace_size(0, 64, 16, 4, 64, 0) == 0
    assert lib.ss_scan_bwd_workspace_size(2, 64, 16, 4, 4096, 0) == 0  # window states exceed shared memory
    p = [_fake(0x10000 + 256 * i) for i in range(18)]

    def call(ptrs=p, B=2, L=64, D=16, N=4, chunk=64, dtype=c.SS_F32, w=_fake(0x90000), wsz=ws):
        return lib.ss_scan_bwd(*ptrs, B, L, D, N, chunk, dtype, None, 0, None, w, wsz, None)

    q = list(p)
    q[8] = None  # dy
    assert call(q) == c.SS_ERR_NULL
    assert call(N=3) == c.SS_ERR_UNSUPPORTED
    assert call(D=20) == c.SS_ERR_ALIGN
    assert call(w=None) == c.SS_ERR_WORKSPACE
    assert call(wsz=ws - 1) == c.SS_ERR_WORKSPACE
    assert call(w=_fake(0x90008)) == c.SS_ERR_ALIGN


def test_layer_fwd_validation(lib):
    from mamba_selective_ssm_gb300 import _capi as c
    p = [_fake(0x10000 + 256 * i) for i in range(4)]
    conv = lambda ptrs=p, B=2, L=10, D=16, K=4, silu=1, dt=c.SS_BF16: lib.conv1d_causal_fwd(*ptrs, B, L, D, K, silu, dt, None)
    q = list(p)
    q[0] = None
    assert conv(q) == c.SS_ERR_NULL
    assert conv(K=5) == c.SS_ERR_UNSUPPORTED
    assert conv(K=0) == c.SS_ERR_DIM
    assert conv(D=12) == c.SS_ERR_ALIGN
    assert conv(dt=3) == c.SS_ERR_UNSUPPORTED
    q = list(p)
    q[3] = _fake(0x10008)
    assert conv(q) == c.SS_ERR_ALIGN
    r = [_fake(0x20000 + 256 * i) for i in range(4)]
    rms = lambda eps=1e-5, rows=4, dim=64, dt=c.SS_F32, x=r[0]: lib.rmsnorm_fwd(x, r[1], eps, r[2], r[3], rows, dim, dt, None)
    assert rms(x=None) == c.SS_ERR_NULL
    assert rms(eps=-1.0) == c.SS_ERR_DIM
    assert rms(eps=float("nan")) == c.SS_ERR_DIM
    assert rms(dim=12) == c.SS_ERR_ALIGN
    assert rms(dim=32776) == c.SS_ERR_DIM
    assert rms(rows=0) == c.SS_ERR_DIM
    assert rms(dt=2) == c.SS_ERR_UNSUPPORTED


def test_decode_step_validation(lib):
    from mamba_selective_ssm_gb300 import _capi as c
    p = [_fake(0x30000 + 256 * i) for i in range(9)]
    step = lambda ptrs=p, B=2, D=16, N=16, dt=c.SS_F32: lib.ss_scan_step(*ptrs, B, D, N, dt, None)
    q = list(p)
    q[7] = None
    assert step(q) == c.SS_ERR_NULL
    assert step(N=5) == c.SS_ERR_UNSUPPORTED
    assert step(B=0) == c.SS_ERR_DIM
    assert step(dt=9) == c.SS_ERR_UNSUPPORTED
    q = list(p)
    q[7] = _fake(0x30004)  # h
    assert step(q) == c.SS_ERR_ALIGN
    r = [_fake(0x40000 + 256 * i) for i in range(5)]
    conv = lambda ptrs=r, B=2, D=16, K=4, dt=c.SS_BF16: lib.conv1d_causal_step(*ptrs, B, D, K, 1, dt, None)
    q = list(r)
    q[1] = None
    assert conv(q) == c.SS_ERR_NULL
    assert conv(K=5) == c.SS_ERR_UNSUPPORTED
    assert conv(D=0) == c.SS_ERR_DIM


def test_conv_and_rms_validation(lib):
    from mamba_selective_ssm_gb300 import _capi as c
    assert lib.conv1d_causal_bwd_workspace_size(4, 2048, 4096, 4) > 0
    assert lib.conv1d_causal_bwd_workspace_size(4, 2048, 4096, 5) == 0
    p = [_fake(0x10000 + 256 * i) for i in range(6)]
    ws = lib.conv1d_causal_bwd_workspace_size(2, 10, 16, 4)
    assert lib.conv1d_causal_bwd(*p, 2, 10, 16, 5, c.SS_F32, _fake(0x90000), ws, None) == c.SS_ERR_UNSUPPORTED
    assert lib.conv1d_causal_bwd(*p, 2, 10, 16, 4, 3, _fake(0x90000), ws, None) == c.SS_ERR_UNSUPPORTED
    assert lib.conv1d_causal_bwd(*p, 2, 10, 12, 4, c.SS_F32, _fake(0x90000), ws, None) == c.SS_ERR_ALIGN
    assert lib.conv1d_causal_bwd(*p, 2, 10, 16, 4, c.SS_F32, None, ws, None) == c.SS_ERR_WORKSPACE
    assert lib.conv1d_causal_bwd(None, *p[1:], 2, 10, 16, 4, c.SS_F32, _fake(0x90000), ws, None) == c.SS_ERR_NULL
    wr = lib.rmsnorm_bwd_workspace_size(100, 768)
    assert wr == 100 * 768 * 4
    assert lib.rmsnorm_bwd_workspace_size(10, 65536) == 0
    assert lib.rmsnorm_bwd(*p, 100, 770, c.SS_F32, _fake(0x90000), wr, None) == c.SS_ERR_ALIGN
    assert lib.rmsnorm_bwd(*p, 0, 768, c.SS_F32, _fake(0x90000), wr, None) == c.SS_ERR_DIM
    assert lib.rmsnorm_bwd(*p, 100, 768, c.SS_F32, _fake(0x90000), wr - 4, None) == c.SS_ERR_WORKSPACE


def test_num_chunks(lib):
    assert lib.ss_scan_num_chunks(64, 64) == 1
    assert lib.ss_scan_num_chunks(65, 64) == 2
    assert lib.ss_scan_num_chunks(16384, 256) == 64
    assert lib.ss_scan_num_chunks(0, 16) == 0


def test_wrapper_rejects_strided_and_cpu_tensors():
    torch = pytest.importorskip("torch")
    from mamba_selective_ssm_gb300 import ops
    t = torch.zeros(4, 4)
    with pytest.raises(ValueError, match="CUDA"):
        ops._req(t, "x")


def test_count_nonfinite_validation(lib):
    from mamba_selective_ssm_gb300 import _capi as c
    wsz = lib.ss_count_nonfinite_workspace_size()
    assert wsz >= 4096
    f = lambda p=_fake(0x50000), n=100, dt=c.SS_F32, cnt=_fake(0x60000), w=_fake(0x70000), ws=wsz: \
        lib.ss_count_nonfinite(p, n, dt, cnt, w, ws, None)
    assert f(cnt=None) == c.SS_ERR_NULL
    assert f(p=None) == c.SS_ERR_NULL
    assert f(dt=7) == c.SS_ERR_UNSUPPORTED
    assert f(w=None) == c.SS_ERR_WORKSPACE
    assert f(ws=wsz - 4) == c.SS_ERR_WORKSPACE
    assert f(p=_fake(0x50004)) == c.SS_ERR_ALIGN
    assert f(cnt=_fake(0x60004)) == c.SS_ERR_ALIGN


def test_abi_is_usable_from_plain_c(lib, tmp_path):
    """tests/abi_from_c.c includes include/ssscan.h and links libssscan.so with gcc: no Python or torch types
    cross the boundary."""
    import subprocess
    from mamba_selective_ssm_gb300 import _build
    gcc = shutil.which("gcc") or shutil.which("cc")
    if gcc is None:
        pytest.skip("no C compiler")
    libdir = os.path.dirname(_build.LIB_PATH)
    exe = tmp_path / "abi_from_c"
    src = os.path.join(ROOT, "tests", "abi_from_c.c")
    r = subprocess.run([gcc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), src, "-o", str(exe),
                        "-L", libdir, "-lssscan", f"-Wl,-rpath,{libdir}"], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr


def test_shard_entry_points_validation(lib):
    """The sequence-sharding calls reject bad arguments on the host before any launch."""
    from mamba_selective_ssm_gb300 import _capi as c
    p = [_fake(0x50000 + 256 * i) for i in range(7)]
    fs = lambda ptrs=p[:6], B=2, L=64, D=16, N=4, dt=c.SS_F32: lib.ss_scan_fwd_summary(*ptrs, B, L, D, N, dt, None, 0, None)
    q = list(p[:6])
    q[4] = None  # h_end
    assert fs(q) == c.SS_ERR_NULL
    assert fs(N=5) == c.SS_ERR_UNSUPPORTED
    assert fs(dt=4) == c.SS_ERR_UNSUPPORTED
    assert fs(B=0) == c.SS_ERR_DIM
    assert fs(D=12) == c.SS_ERR_ALIGN
    q = list(p[:6])
    q[1] = _fake(0x50004)
    assert fs(q) == c.SS_ERR_ALIGN
    bs = lambda ptrs=p, B=2, L=64, D=16, N=16, dt=c.SS_BF16: lib.ss_scan_bwd_summary(*ptrs, B, L, D, N, dt, None, 1, None)
    q = list(p)
    q[4] = None  # dy
    assert bs(q) == c.SS_ERR_NULL
    assert bs(N=2) == c.SS_ERR_UNSUPPORTED
    assert bs(L=-3) == c.SS_ERR_DIM
    assert bs(D=20) == c.SS_ERR_ALIGN
    q = list(p)
    q[5] = _fake(0x50008)  # g_start
    assert bs(q) == c.SS_ERR_ALIGN
    r = [_fake(0x60000 + 256 * i) for i in range(5)]
    car = lambda ptrs=r, P=4, B=2, D=16, N=16: lib.ss_scan_carries(*ptrs, P, B, D, N, 0, None)
    q = list(r)
    q[0] = None  # A
    assert car(q) == c.SS_ERR_NULL
    q = list(r)
    q[4] = None  # carry
    assert car(q) == c.SS_ERR_NULL
    assert car(P=0) == c.SS_ERR_DIM
    assert car(B=0) == c.SS_ERR_DIM
    assert car(P=65) == c.SS_ERR_UNSUPPORTED
