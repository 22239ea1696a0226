"""Runtime properties of the layer call: it records into a CUDA graph (no host
synchronisation, allocation or device-to-host copy inside), and calls on
different streams with their own workspaces run concurrently without sharing
state.  Both must give the same bits as plain sequential calls."""
import pytest
import torch

import moe_expert_layer_router_gb300 as m
import workload as wl
from parity import Layer

pytestmark = pytest.mark.gpu

LC = wl.DSV3.with_(name="dsv3_shape_T64", T=64, E=32, k=4, I=256, I_shared=256)


def weights_of(L, cfg):
    return m.ExpertWeights(cfg, [w[0] for w in L.W], [w[1] for w in L.W], [w[2] for w in L.W],
                           shared=L.S)


def test_forward_replays_from_a_cuda_graph():
    dev = torch.device("cuda")
    L = Layer(LC, dev)
    cfg = m.config_from(LC)
    W = weights_of(L, cfg)
    ws = m.Workspace(cfg, "forward")
    ref = m.moe_forward(cfg, W, L.x, L.wr, L.bias, ws=ws)
    torch.cuda.synchronize()
    x = L.x.clone()
    out = torch.empty_like(ref)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        m.moe_forward(cfg, W, x, L.wr, L.bias, out=out, ws=ws, stream=torch.cuda.current_stream())
    for _ in range(3):
        out.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, ref)
    # the recorded graph reads x from its buffer when it runs
    x.copy_(Layer(LC.with_(seed=5), dev).x)
    graph.replay()
    ref2 = m.moe_forward(cfg, W, x, L.wr, L.bias, ws=ws)
    torch.cuda.synchronize()
    assert torch.equal(out, ref2) and not torch.equal(ref2, ref)
    assert m.moe_get_device_error(ws) == 0


def test_concurrent_streams_with_separate_workspaces():
    dev = torch.device("cuda")
    layers = [Layer(LC.with_(seed=s), dev) for s in (0, 1)]
    cfg = m.config_from(LC)
    Ws = [weights_of(L, cfg) for L in layers]
    refs = [m.moe_forward(cfg, W, L.x, L.wr, L.bias) for W, L in zip(Ws, layers)]
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    wss = [m.Workspace(cfg, "forward") for _ in range(2)]
    outs = [torch.empty_like(r) for r in refs]
    torch.cuda.synchronize()
    for _ in range(4):
        for i in (0, 1):
            with torch.cuda.stream(streams[i]):
                m.moe_forward(cfg, Ws[i], layers[i].x, layers[i].wr, layers[i].bias, out=outs[i],
                              ws=wss[i], stream=streams[i])
    torch.cuda.synchronize()
    for i in (0, 1):
        assert torch.equal(outs[i], refs[i])
        assert m.moe_get_device_error(wss[i]) == 0
