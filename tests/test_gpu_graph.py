"""The library's calls inside a CUDA graph: a decode loop (SSM step + conv step for
several tokens) and a training step's scan forward + backward are captured once with
torch.cuda.graph, replayed on new inputs copied into the captured buffers, and compared
with the same calls run eagerly (bitwise: the same kernels on the same data)."""

import numpy as np
import pytest

from tests.gpu_util import ss_module

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ss():
    return ss_module()


def test_decode_loop_in_a_graph(ss):
    import torch
    dev = torch.device("cuda", 0)
    g = torch.Generator(device=dev).manual_seed(3)
    B, D, N, K, T = 64, 256, 16, 4, 5
    bf = torch.bfloat16
    A = -(torch.rand(D, N, device=dev, generator=g) + 0.5)
    Dv, w, bias = torch.randn(D, device=dev, generator=g), torch.randn(D, K, device=dev, generator=g) * 0.5, \
        torch.randn(D, device=dev, generator=g) * 0.1
    def draw():
        return {"x": torch.randn(T, B, D, device=dev, generator=g).to(bf),
                "delta": (0.001 + 0.1 * torch.rand(T, B, D, device=dev, generator=g)).to(bf),
                "z": torch.randn(T, B, D, device=dev, generator=g).to(bf),
                "Bm": torch.randn(T, B, N, device=dev, generator=g).to(bf),
                "Cm": torch.randn(T, B, N, device=dev, generator=g).to(bf)}
    static = draw()
    h = torch.zeros(B, D, N, device=dev)
    cs = torch.zeros(B, D, K, device=dev)
    ys = torch.empty(T, B, D, device=dev, dtype=bf)

    def loop(h, cs, ys, inp):
        for t in range(T):
            u = ss.conv1d_causal_step(inp["x"][t], cs, w, bias, silu=True)
            ys[t] = ss.ss_scan_step(u, inp["delta"][t], A, inp["Bm"][t], inp["Cm"][t], Dv, inp["z"][t], h)

    s = torch.cuda.Stream(dev)
    s.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(s):  # warm-up outside the graph (attributes, occupancy queries, first-use setup)
        loop(h, cs, ys, static)
    torch.cuda.current_stream(dev).wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        loop(h, cs, ys, static)
    for _ in range(2):
        new = draw()
        for k in static:
            static[k].copy_(new[k])
        h0, c0 = h.clone(), cs.clone()
        graph.replay()
        torch.cuda.synchronize(dev)
        he, ce = h0.clone(), c0.clone()
        ye = torch.empty_like(ys)
        loop(he, ce, ye, new)
        torch.cuda.synchronize(dev)
        assert torch.equal(ys, ye) and torch.equal(h, he) and torch.equal(cs, ce)
    assert ss.device_status() == 0


def test_scan_forward_backward_in_a_graph(ss):
    import torch
    dev = torch.device("cuda", 0)
    g = torch.Generator(device=dev).manual_seed(4)
    B, L, D, N, chunk = 2, 256, 128, 16, 8
    bf = torch.bfloat16
    A = -(torch.rand(D, N, device=dev, generator=g) + 0.5)
    Dv = torch.randn(D, device=dev, generator=g)
    def draw():
        return {"x": torch.randn(B, L, D, device=dev, generator=g).to(bf),
                "delta": (0.001 + 0.1 * torch.rand(B, L, D, device=dev, generator=g)).to(bf),
                "z": torch.randn(B, L, D, device=dev, generator=g).to(bf),
                "dy": torch.randn(B, L, D, device=dev, generator=g).to(bf),
                "Bm": torch.randn(B, L, N, device=dev, generator=g).to(bf),
                "Cm": torch.randn(B, L, N, device=dev, generator=g).to(bf)}
    static = draw()

    def step(inp):
        y, ck, hl = ss.ss_scan_fwd(inp["x"], inp["delta"], A, inp["Bm"], inp["Cm"], Dv, inp["z"], chunk=chunk)
        gr = ss.ss_scan_bwd(inp["x"], inp["delta"], A, inp["Bm"], inp["Cm"], Dv, inp["z"], ck, inp["dy"], chunk=chunk)
        return y, hl, gr

    s = torch.cuda.Stream(dev)
    s.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(s):
        step(static)
    torch.cuda.current_stream(dev).wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        y, hl, gr = step(static)
    new = draw()
    for k in static:
        static[k].copy_(new[k])
    graph.replay()
    torch.cuda.synchronize(dev)
    ye, hle, gre = step(new)
    torch.cuda.synchronize(dev)
    assert torch.equal(y, ye) and torch.equal(hl, hle)
    for k in ("dx", "ddelta", "dz", "dB", "dC", "dA", "dD", "dh0"):
        assert torch.equal(gr[k], gre[k]), k
    assert ss.device_status() == 0
