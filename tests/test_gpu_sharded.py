"""Sequence sharding on the GPU: the piece summaries and the carry composition
through the C ABI against the float64 oracle, the pieces of one sequence run one
after another in one process, and two gloo ranks that share the GPU, each
holding half of the time axis, against the oracle over the whole sequence.

The ranks exchange only on the host (gloo, through host memory): no kernel of
one rank waits on the other's."""

import os
import socket
import sys

import numpy as np
import pytest

from oracle import scan_bwd_ref, scan_fwd_ref
from oracle.scan import delta_softplus_ref, scan_bwd_fused_ref, scan_fwd_fused_ref
from tests._util import TOL, assert_close
from tests.gpu_util import dev, host, scan_inputs_on_device, ss_module
from workloads import CONFIGS, make_scan_inputs

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def ss():
    return ss_module()


def _wl(B, L, D, N, dtype):
    return CONFIGS["tiny"].with_(B=B, L=L, D=D, N=N, dtype=dtype, chunk=16)


SUMMARY_CASES = [
    # B, L, D, N, dtype, fused
    (2, 64, 16, 4, "f32", False),
    (3, 203, 40, 16, "f32", True),    # ragged last tile and channel tile
    (2, 100, 72, 8, "bf16", False),
    (1, 333, 136, 16, "bf16", True),
    (2, 1, 8, 16, "f32", False),      # one step
]


@pytest.mark.parametrize("B,L,D,N,dtype,fused", SUMMARY_CASES)
def test_fwd_summary(ss, B, L, D, N, dtype, fused):
    inp = make_scan_inputs(_wl(B, L, D, N, dtype), seed=L + 3)
    d = scan_inputs_on_device(inp, dtype)
    if fused:
        raw = dev(inp["delta_raw"], dtype)
        h_end, dsum = ss.ss_scan_fwd_summary(d["x"], raw, d["A"], d["Bm"], dt_bias=dev(inp["dt_bias"]),
                                             delta_softplus=True)
        delta = delta_softplus_ref(inp["delta_raw"], inp["dt_bias"], True)
    else:
        h_end, dsum = ss.ss_scan_fwd_summary(d["x"], d["delta"], d["A"], d["Bm"])
        delta = inp["delta"]
    zeros = np.zeros_like(inp["Cm"])
    _, h_ref, _ = scan_fwd_ref(inp["x"], delta, inp["A"], inp["Bm"], zeros, inp["Dv"], inp["z"])
    tol = TOL[dtype]
    assert_close(host(h_end), h_ref, tol, "h_end")
    assert_close(host(dsum), delta.sum(1), tol, "delta_sum")
    assert ss.device_status() == 0


@pytest.mark.parametrize("B,L,D,N,dtype,fused", SUMMARY_CASES)
def test_bwd_summary(ss, B, L, D, N, dtype, fused):
    inp = make_scan_inputs(_wl(B, L, D, N, dtype), seed=L + 4)
    d = scan_inputs_on_device(inp, dtype)
    if fused:
        raw = dev(inp["delta_raw"], dtype)
        g_start, dsum = ss.ss_scan_bwd_summary(raw, d["A"], d["Cm"], d["z"], d["dy"], dt_bias=dev(inp["dt_bias"]),
                                               delta_softplus=True)
        delta = delta_softplus_ref(inp["delta_raw"], inp["dt_bias"], True)
    else:
        g_start, dsum = ss.ss_scan_bwd_summary(d["delta"], d["A"], d["Cm"], d["z"], d["dy"])
        delta = inp["delta"]
    g = scan_bwd_ref(inp["x"], delta, inp["A"], inp["Bm"], inp["Cm"], inp["Dv"], inp["z"], inp["dy"])
    tol = TOL[dtype]
    assert_close(host(g_start), g["dh0"], tol, "g_start")
    assert_close(host(dsum), delta.sum(1), tol, "delta_sum")
    assert ss.device_status() == 0


def _compose(A, S, H, init, reverse):
    """The carries by their definition: a plain loop over the pieces in float64."""
    P = H.shape[0]
    c = np.zeros_like(H)
    cur = np.zeros_like(H[0]) if init is None else init.copy()
    for p in (range(P - 1, -1, -1) if reverse else range(P)):
        c[p] = cur
        cur = np.exp(A[None] * S[p][..., None]) * cur + H[p]
    return c


@pytest.mark.parametrize("P,B,D,N,reverse,with_init", [
    (1, 2, 8, 4, False, True), (2, 3, 40, 16, True, True), (7, 2, 24, 8, False, False),
    (33, 1, 16, 16, True, False), (64, 2, 8, 16, False, True), (64, 1, 16, 4, True, True),
])
def test_carries(ss, P, B, D, N, reverse, with_init):
    rng = np.random.default_rng(P * 100 + D)
    f32 = lambda a: a.astype(np.float32).astype(np.float64)
    A = f32(-np.broadcast_to(np.arange(1, N + 1), (D, N)) * 0.05)
    S = f32(rng.uniform(0.0, 4.0, (P, B, D)))
    H = f32(rng.standard_normal((P, B, D, N)))
    init = f32(rng.standard_normal((B, D, N))) if with_init else None
    got = ss.ss_scan_carries(dev(A), dev(S), dev(H), None if init is None else dev(init), reverse=reverse)
    assert_close(host(got), _compose(A, S, H, init, reverse), TOL["f32"], "carry")


PIECE_CASES = [
    # dtype, N, pieces, fused, chunk
    ("f32", 16, (48, 80, 17, 64, 1), False, 16),
    ("bf16", 16, (100, 37, 200), True, 8),
    ("bf16", 8, (64, 64, 64, 64), False, 32),
    ("f32", 4, (30, 2, 70), True, 16),   # a two-step piece, N = 4 (one warp spans 32 channels)
]


@pytest.mark.parametrize("dtype,N,pieces,fused,chunk", PIECE_CASES)
def test_pieces_in_sequence_match_the_whole(ss, dtype, N, pieces, fused, chunk):
    """The sharded scan with its ranks run one after another: summaries of every piece, one
    composition per direction, then every piece from its carry."""
    import torch
    B, D = 2, 48
    L = sum(pieces)
    inp = make_scan_inputs(_wl(B, L, D, N, dtype), seed=len(pieces))
    d = scan_inputs_on_device(inp, dtype)
    rng = np.random.default_rng(1)
    h0 = rng.standard_normal((B, D, N)).astype(np.float32).astype(np.float64)
    dhl = rng.standard_normal((B, D, N)).astype(np.float32).astype(np.float64)
    delta_key = "delta_raw" if fused else "delta"
    kw = dict(dt_bias=dev(inp["dt_bias"]), delta_softplus=True) if fused else {}
    draw = dev(inp["delta_raw"], dtype) if fused else d["delta"]
    cuts = np.cumsum((0,) + pieces)
    sl = [slice(int(cuts[i]), int(cuts[i + 1])) for i in range(len(pieces))]
    piece = lambda t, s: t[:, s].contiguous()
    fs = [ss.ss_scan_fwd_summary(piece(d["x"], s), piece(draw, s), d["A"], piece(d["Bm"], s), **kw) for s in sl]
    carry = ss.ss_scan_carries(d["A"], torch.stack([f[1] for f in fs]), torch.stack([f[0] for f in fs]), init=dev(h0))
    outs = [ss.ss_scan_fwd(piece(d["x"], s), piece(draw, s), d["A"], piece(d["Bm"], s), piece(d["Cm"], s), d["Dv"],
                           piece(d["z"], s), h0=carry[i], chunk=chunk, **kw) for i, s in enumerate(sl)]
    bs = [ss.ss_scan_bwd_summary(piece(draw, s), d["A"], piece(d["Cm"], s), piece(d["z"], s), piece(d["dy"], s), **kw)
          for s in sl]
    gcarry = ss.ss_scan_carries(d["A"], torch.stack([b[1] for b in bs]), torch.stack([b[0] for b in bs]),
                                init=dev(dhl), reverse=True)
    grads = [ss.ss_scan_bwd(piece(d["x"], s), piece(draw, s), d["A"], piece(d["Bm"], s), piece(d["Cm"], s), d["Dv"],
                            piece(d["z"], s), outs[i][1], piece(d["dy"], s), dh_last=gcarry[i], chunk=chunk, **kw)
             for i, s in enumerate(sl)]
    a = (inp["x"], inp[delta_key], inp["A"], inp["Bm"], inp["Cm"], inp["Dv"], inp["z"])
    if fused:
        y, hl, _ = scan_fwd_fused_ref(*a, dt_bias=inp["dt_bias"], softplus=True, h0=h0)
        g = scan_bwd_fused_ref(*a, inp["dy"], dt_bias=inp["dt_bias"], softplus=True, h0=h0, dh_last=dhl)
    else:
        y, hl, _ = scan_fwd_ref(*a, h0=h0)
        g = scan_bwd_ref(*a, inp["dy"], h0=h0, dh_last=dhl)
    tol = TOL[dtype]
    assert_close(host(torch.cat([o[0] for o in outs], 1)), y, tol, "y")
    assert_close(host(outs[-1][2]), hl, tol, "h_last")
    for k in ("dx", "ddelta", "dz", "dB", "dC"):
        assert_close(host(torch.cat([gr[k] for gr in grads], 1)), g[k], tol, k)
    for k in ("dA", "dD") + (("d_dt_bias",) if fused else ()):
        assert_close(sum(host(gr[k]) for gr in grads), g[k], tol, k)
    assert_close(host(grads[0]["dh0"]), g["dh0"], tol, "dh0")
    assert ss.device_status() == 0


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


RANK_CASE = dict(B=2, D=64, N=16, dtype="bf16", pieces=(150, 170), chunk=8)


def _rank_worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    from mamba_selective_ssm_gb300 import sharded
    from tests.gpu_util import dev as dev_, host as host_
    c = RANK_CASE
    torch.cuda.set_device(0)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        inp = make_scan_inputs(_wl(c["B"], sum(c["pieces"]), c["D"], c["N"], c["dtype"]), seed=77)
        t0 = sum(c["pieces"][:rank])
        s = slice(t0, t0 + c["pieces"][rank])
        p = {k: dev_(np.ascontiguousarray(inp[k][:, s]), c["dtype"]) for k in ("x", "delta_raw", "z", "Bm", "Cm", "dy")}
        A, Dv, bias = dev_(inp["A"]), dev_(inp["Dv"]), dev_(inp["dt_bias"])
        rng = np.random.default_rng(2)
        h0 = dev_(rng.standard_normal((c["B"], c["D"], c["N"])))
        dhl = dev_(rng.standard_normal((c["B"], c["D"], c["N"])))
        kw = dict(dt_bias=bias, delta_softplus=True)
        y, ck, hl, _ = sharded.ss_scan_fwd_sharded(p["x"], p["delta_raw"], A, p["Bm"], p["Cm"], Dv, p["z"], h0=h0,
                                                   chunk=c["chunk"], **kw)
        g = sharded.ss_scan_bwd_sharded(p["x"], p["delta_raw"], A, p["Bm"], p["Cm"], Dv, p["z"], ck, p["dy"],
                                         dh_last=dhl, chunk=c["chunk"], **kw)
        torch.cuda.synchronize()
        q.put((rank, {"y": host_(y), "h_last": host_(hl), "h0": host_(h0), "dhl": host_(dhl),
                      **{k: host_(v) for k, v in g.items() if v is not None}}))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_on_one_gpu_match_the_whole_sequence(ss):
    import torch.multiprocessing as mp
    c = RANK_CASE
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=600) for _ in range(2))
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    inp = make_scan_inputs(_wl(c["B"], sum(c["pieces"]), c["D"], c["N"], c["dtype"]), seed=77)
    h0, dhl = got[0]["h0"], got[0]["dhl"]
    a = (inp["x"], inp["delta_raw"], inp["A"], inp["Bm"], inp["Cm"], inp["Dv"], inp["z"])
    y, hl, _ = scan_fwd_fused_ref(*a, dt_bias=inp["dt_bias"], softplus=True, h0=h0)
    g = scan_bwd_fused_ref(*a, inp["dy"], dt_bias=inp["dt_bias"], softplus=True, h0=h0, dh_last=dhl)
    tol = TOL[c["dtype"]]
    assert_close(np.concatenate([got[0]["y"], got[1]["y"]], 1), y, tol, "y")
    assert_close(got[1]["h_last"], hl, tol, "h_last")
    for k in ("dx", "ddelta", "dz", "dB", "dC"):
        assert_close(np.concatenate([got[0][k], got[1][k]], 1), g[k], tol, k)
    for r in range(2):
        for k in ("dA", "dD", "d_dt_bias"):
            assert_close(got[r][k], g[k], tol, f"{k} rank {r}")
    assert_close(got[0]["dh0"], g["dh0"], tol, "dh0")


def _nccl_one_rank_worker(port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), NCCL_NVLS_ENABLE="0")
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    from mamba_selective_ssm_gb300 import ops, sharded
    from tests.gpu_util import dev as dev_, host as host_
    torch.cuda.set_device(0)
    dist.init_process_group("nccl", rank=0, world_size=1, device_id=torch.device("cuda", 0))
    try:
        rng = np.random.default_rng(5)
        t = dev_(rng.standard_normal((2, 24, 16)))
        u = dev_(rng.standard_normal((24,)))
        g = sharded.all_gather_pieces(t)
        u0 = u.clone()
        sharded.all_reduce_sum_(u)
        c = RANK_CASE
        inp = make_scan_inputs(_wl(c["B"], sum(c["pieces"]), c["D"], c["N"], c["dtype"]), seed=78)
        p = {k: dev_(inp[k], c["dtype"]) for k in ("x", "delta_raw", "z", "Bm", "Cm", "dy")}
        A, Dv, bias = dev_(inp["A"]), dev_(inp["Dv"]), dev_(inp["dt_bias"])
        kw = dict(dt_bias=bias, delta_softplus=True)
        a = (p["x"], p["delta_raw"], A, p["Bm"], p["Cm"], Dv, p["z"])
        y, ck, hl, _ = sharded.ss_scan_fwd_sharded(*a, chunk=c["chunk"], **kw)
        gs = sharded.ss_scan_bwd_sharded(*a, ck, p["dy"], chunk=c["chunk"], **kw)
        # the exchange the ranks of a larger group run, through the device collectives: one piece composes to h0
        h0 = dev_(rng.standard_normal((c["B"], c["D"], c["N"])))
        h_end, dsum = ops.ss_scan_fwd_summary(p["x"], p["delta_raw"], A, p["Bm"], **kw)
        carry = ops.ss_scan_carries(A, sharded.all_gather_pieces(dsum), sharded.all_gather_pieces(h_end), init=h0)
        y1, ck1, hl1 = ops.ss_scan_fwd(*a, chunk=c["chunk"], **kw)
        g1 = ops.ss_scan_bwd(*a, ck1, p["dy"], chunk=c["chunk"], **kw)
        torch.cuda.synchronize()
        q.put({"backend": dist.get_backend(), "gather_shape": tuple(g.shape), "gather_same": bool(torch.equal(g[0], t)),
               "carry_shape": tuple(carry.shape), "carry_err": float((carry[0] - h0).abs().max() / h0.abs().max()),
               "reduce_same": bool(torch.equal(u, u0)), "y_same": bool(torch.equal(y, y1)),
               "h_last_same": bool(torch.equal(hl, hl1)),
               "grads_same": {k: bool(torch.equal(v, g1[k])) for k, v in gs.items() if v is not None and k in g1}})
    finally:
        dist.destroy_process_group()


def test_one_nccl_rank_runs_the_device_exchange(ss):
    """The NCCL branch of the exchange (all-gather into one device tensor, device all-reduce) with a single rank:
    no peer to wait on, so it runs on this one GPU; the whole sequence as one piece equals the unsharded calls."""
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    proc = ctx.Process(target=_nccl_one_rank_worker, args=(_free_port(), q))
    proc.start()
    got = q.get(timeout=600)
    proc.join(timeout=120)
    assert proc.exitcode == 0
    assert got["backend"] == "nccl"
    assert got["gather_shape"] == (1, 2, 24, 16) and got["gather_same"]
    assert got["reduce_same"]
    assert got["carry_shape"] == (1, RANK_CASE["B"], RANK_CASE["D"], RANK_CASE["N"]) and got["carry_err"] <= 1e-6
    assert got["y_same"] and got["h_last_same"]
    assert got["grads_same"] and all(got["grads_same"].values()), got["grads_same"]
