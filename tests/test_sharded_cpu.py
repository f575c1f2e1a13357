"""The sequence-sharded scan's exchange on the CPU: three gloo ranks.

Each rank holds a piece of the time axis (pieces of different lengths).  The
library calls of ``mamba_selective_ssm_gb300.sharded`` are replaced, in the
ranks only, by float64 stand-ins built on the oracle (the forward / backward of
a piece from a given start, its zero-start summary, and the composition of the
pieces' affine maps written as a plain loop), so this checks on the CPU what the
module itself does: which rank gets which carry, the direction of the
backward's exchange, the all-reduce of dA / dD / d_dt_bias and the accumulation
convention, against the oracle run over the whole sequence."""

import os
import socket
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PIECES = (5, 9, 7)
B, D, N = 2, 6, 4


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _inputs():
    sys.path.insert(0, ROOT)
    from workloads import CONFIGS, make_scan_inputs
    wl = CONFIGS["tiny"].with_(B=B, L=sum(PIECES), D=D, N=N, dtype="f32", chunk=4)
    inp = make_scan_inputs(wl, seed=21)
    rng = np.random.default_rng(5)
    extra = {k: rng.standard_normal(s) for k, s in (("h0", (B, D, N)), ("dhl", (B, D, N)), ("dA0", (D, N)),
                                                       ("dD0", (D,)), ("db0", (D,)))}
    return inp, extra


class _OracleOps:
    """float64 stand-ins for the library calls the sharded module makes (torch in, torch out)."""

    def __init__(self):
        import torch
        self.t = torch

    def _np(self, v):
        return None if v is None else v.detach().numpy()

    def _delta(self, delta, dt_bias, softplus):
        from oracle.scan import delta_softplus_ref
        d = self._np(delta)
        return delta_softplus_ref(d, self._np(dt_bias), softplus) if (dt_bias is not None or softplus) else d

    def ss_scan_fwd_summary(self, x, delta, A, Bm, dt_bias=None, delta_softplus=False):
        from oracle import scan_fwd_ref
        d = self._delta(delta, dt_bias, delta_softplus)
        Bsz, L, Dd = d.shape
        zeros = np.zeros((Bsz, L, A.shape[1]))
        _, h_end, _ = scan_fwd_ref(self._np(x), d, self._np(A), self._np(Bm), zeros, np.zeros(Dd), np.zeros_like(d))
        return self.t.from_numpy(h_end), self.t.from_numpy(d.sum(1))

    def ss_scan_bwd_summary(self, delta, A, Cm, z, dy, dt_bias=None, delta_softplus=False):
        from oracle import scan_bwd_ref
        d = self._delta(delta, dt_bias, delta_softplus)
        g = scan_bwd_ref(np.zeros_like(d), d, self._np(A), np.zeros_like(self._np(Cm)), self._np(Cm),
                         np.zeros(d.shape[2]), self._np(z), self._np(dy))
        return self.t.from_numpy(g["dh0"]), self.t.from_numpy(d.sum(1))

    def ss_scan_carries(self, A, delta_sum, summ, init=None, reverse=False):
        A, S, H = self._np(A), self._np(delta_sum), self._np(summ)
        P = H.shape[0]
        c = np.zeros_like(H)
        cur = np.zeros_like(H[0]) if init is None else self._np(init).copy()
        order = range(P - 1, -1, -1) if reverse else range(P)
        for p in order:
            c[p] = cur
            cur = np.exp(A[None] * S[p][..., None]) * cur + H[p]
        return self.t.from_numpy(c)

    def ss_scan_fwd(self, x, delta, A, Bm, Cm, Dv, z, h0=None, chunk=64, want_h_last=True, dt_bias=None,
                    delta_softplus=False):
        from oracle import scan_fwd_ref
        d = self._delta(delta, dt_bias, delta_softplus)
        y, hl, ck = scan_fwd_ref(self._np(x), d, self._np(A), self._np(Bm), self._np(Cm), self._np(Dv), self._np(z),
                                 h0=self._np(h0), chunk=chunk)
        return self.t.from_numpy(y), self.t.from_numpy(ck), self.t.from_numpy(hl)

    def ss_scan_bwd(self, x, delta, A, Bm, Cm, Dv, z, ckpt, dy, dh_last=None, chunk=64, dA=None, dD=None,
                    dt_bias=None, delta_softplus=False, d_dt_bias=None):
        from oracle.scan import scan_bwd_fused_ref
        from oracle import scan_bwd_ref
        a = [self._np(v) for v in (x, delta, A, Bm, Cm, Dv, z)]
        h0 = self._np(ckpt)[:, 0]  # the piece's start state, as the library reads it from its checkpoints
        if dt_bias is not None or delta_softplus:
            g = scan_bwd_fused_ref(*a, self._np(dy), dt_bias=self._np(dt_bias), softplus=delta_softplus, h0=h0,
                                   dh_last=self._np(dh_last))
        else:
            g = scan_bwd_ref(*a, self._np(dy), h0=h0, dh_last=self._np(dh_last))
        out = {k: self.t.from_numpy(np.ascontiguousarray(v)) for k, v in g.items()}
        for k, acc in (("dA", dA), ("dD", dD), ("d_dt_bias", d_dt_bias)):
            if acc is not None and k in out:
                acc += out[k]
                out[k] = acc
        return out


def _worker(rank, world, port, fused, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    from mamba_selective_ssm_gb300 import sharded
    sharded.ops = _OracleOps()
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        inp, ex = _inputs()
        t0 = sum(PIECES[:rank])
        sl = slice(t0, t0 + PIECES[rank])
        T = lambda a: torch.from_numpy(np.ascontiguousarray(a))
        seq = {k: T(inp[k][:, sl]) for k in ("x", "z", "Bm", "Cm", "dy")}
        delta = T(inp["delta_raw"][:, sl] if fused else inp["delta"][:, sl])
        kw = dict(dt_bias=T(inp["dt_bias"]), delta_softplus=True) if fused else {}
        A, Dv = T(inp["A"]), T(inp["Dv"])
        y, ck, hl, h_in = sharded.ss_scan_fwd_sharded(seq["x"], delta, A, seq["Bm"], seq["Cm"], Dv, seq["z"],
                                                      h0=T(ex["h0"]), chunk=4, **kw)
        g = sharded.ss_scan_bwd_sharded(seq["x"], delta, A, seq["Bm"], seq["Cm"], Dv, seq["z"], ck, seq["dy"],
                                        dh_last=T(ex["dhl"]), chunk=4, dA=T(ex["dA0"].copy()), dD=T(ex["dD0"].copy()),
                                        d_dt_bias=T(ex["db0"].copy()) if fused else None, **kw)
        q.put((rank, {"y": y.numpy(), "h_last": hl.numpy(), **{k: v.numpy() for k, v in g.items() if v is not None}}))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("fused", [False, True])
def test_sharded_scan_three_gloo_ranks_match_the_whole_sequence(fused):
    import torch.multiprocessing as mp
    from oracle import scan_bwd_ref, scan_fwd_ref
    from oracle.scan import scan_bwd_fused_ref, scan_fwd_fused_ref
    world = len(PIECES)
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, fused, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=300) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    inp, ex = _inputs()
    a = (inp["x"], inp["delta_raw"] if fused else inp["delta"], inp["A"], inp["Bm"], inp["Cm"], inp["Dv"], inp["z"])
    if fused:
        y, hl, _ = scan_fwd_fused_ref(*a, dt_bias=inp["dt_bias"], softplus=True, h0=ex["h0"])
        g = scan_bwd_fused_ref(*a, inp["dy"], dt_bias=inp["dt_bias"], softplus=True, h0=ex["h0"], dh_last=ex["dhl"])
    else:
        y, hl, _ = scan_fwd_ref(*a, h0=ex["h0"])
        g = scan_bwd_ref(*a, inp["dy"], h0=ex["h0"], dh_last=ex["dhl"])
    cat = lambda k: np.concatenate([got[r][k] for r in range(world)], axis=1)
    close = lambda u, v: np.testing.assert_allclose(u, v, rtol=1e-10, atol=1e-10)
    close(cat("y"), y)
    close(got[world - 1]["h_last"], hl)
    for k in ("dx", "ddelta", "dz", "dB", "dC"):
        close(cat(k), g[k])
    close(got[0]["dh0"], g["dh0"])
    close(got[world - 1]["g_in"], ex["dhl"])
    for r in range(world):  # replicated, accumulated parameter gradients
        close(got[r]["dA"], ex["dA0"] + g["dA"])
        close(got[r]["dD"], ex["dD0"] + g["dD"])
        if fused:
            close(got[r]["d_dt_bias"], ex["db0"] + g["d_dt_bias"])
