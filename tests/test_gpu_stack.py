"""Layer stacks: L layers behind one layer-oblivious descriptor table, the layer
index read on the device when the kernels run.  Every layer of a stack must
match the oracle's layer for that layer's weights and logit bias (routing
bit-exact off measured near ties, output within the layer tolerance), and give
the same bits as that layer run on its own through moe_forward (same kernels,
same arithmetic), through direct calls and through one CUDA graph recorded once
and replayed for every layer."""
import pytest
import torch

import moe_expert_layer_router_gb300 as m
import workload as wl
from oracle import fp8 as of8
from oracle import moe as om
from parity import FP8_MAX_OVER_RMS, Layer, Routing, assert_close_layer, f64, with_flips
from test_gpu_fp8 import Fp8Layer

pytestmark = pytest.mark.gpu

NUM_LAYERS = 3


def bf16_stack(lc, dev, with_bias):
    """NUM_LAYERS seeded layers of one shape, their per-layer references on a
    common input, and the stack.  With bias, layer 0 has none and the others a
    seeded fp32 logit bias (a NULL entry in the stack's bias table)."""
    layers = [Layer(lc.with_(seed=s), dev) for s in range(NUM_LAYERS)]
    x = layers[0].x
    cfg = m.config_from(lc)
    W = [m.ExpertWeights(cfg, [w[0] for w in L.W], [w[1] for w in L.W], [w[2] for w in L.W],
                         shared=L.S) for L in layers]
    bias = None
    if with_bias:
        g = torch.Generator().manual_seed(7)
        bias = [None] + [torch.randn(lc.E, generator=g).mul_(0.5).to(dev)
                         for _ in range(NUM_LAYERS - 1)]
    refs, oracle = [], []
    for l in range(NUM_LAYERS):
        b = None if bias is None else bias[l]
        out, ids, _ = m.moe_forward(cfg, W[l], x, layers[l].wr, b, return_routing=True)
        torch.cuda.synchronize()
        refs.append(out)
        oracle.append(oracle_bf16_layer(f"stack_layer{l}", lc, cfg, layers[l], x, b,
                                        ids.cpu().numpy()))
    stack = m.LayerStack(cfg, W, [L.wr for L in layers], bias)
    torch.cuda.synchronize()
    return cfg, x, refs, stack, oracle


def oracle_bf16_layer(name, lc, cfg, L, x, bias, ids_gpu):
    """The oracle's output of layer L (its weights and logit bias) on input x,
    flipped near-tie tokens evaluated on the GPU's ids."""
    r = Routing(name, lc, cfg, x, L.wr, bias, ids_gpu, m)
    b = None if bias is None else f64(bias)
    ref = om.moe_layer(f64(x), f64(L.wr), b, L.experts_cpu, L.shared_cpu(), lc.k, lc.score,
                       lc.renormalize, lc.route_scale)
    return with_flips(r, ref["out"], lambda t, i, w_: om.moe_tokens(
        f64(x)[t], i, w_, L.experts_cpu, L.shared_cpu()))


SHAPES = [
    wl.TINY.with_(name="tiny_shared_sigmoid", T=200, I_shared=256, score="sigmoid",
                  route_scale=2.5),
    wl.DSV3.with_(name="dsv3_shape_T64", T=64, E=32, k=4, I=256, I_shared=256),
    # 79 token tiles: the router runs on CTA pairs (K unsplit) with the stack's table
    wl.TINY.with_(name="pair_router_T10000", T=10000, H=256, E=32, k=4, I=128, I_shared=128,
                  score="sigmoid", route_scale=2.5),
]


@pytest.mark.parametrize("lc", SHAPES, ids=lambda c: c.name)
def test_stack_layers_match_single_layer_calls(lc):
    dev = torch.device("cuda")
    cfg, x, refs, stack, oracle = bf16_stack(lc, dev, with_bias=True)
    layer = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = m.Workspace(cfg, "forward")
    for l in (2, 0, 1, 2):
        layer.fill_(l)
        out = m.moe_forward_stack(cfg, stack, layer, x, ws=ws)
        torch.cuda.synchronize()
        assert m.moe_get_device_error(ws) == 0
        assert_close_layer(out, oracle[l], what=f"{lc.name} stack layer {l}")
        assert torch.equal(out, refs[l]), f"layer {l}"


def test_one_graph_serves_every_layer():
    """Record moe_forward_stack once; writing the layer index and replaying runs any
    layer, with no host work between layers."""
    dev = torch.device("cuda")
    lc = SHAPES[1]
    cfg, x, refs, stack, oracle = bf16_stack(lc, dev, with_bias=True)
    layer = torch.zeros(1, dtype=torch.int32, device=dev)
    out = torch.empty(lc.T, lc.H, dtype=torch.bfloat16, device=dev)
    ws = m.Workspace(cfg, "forward")
    m.moe_forward_stack(cfg, stack, layer, x, out=out, ws=ws)  # first use outside capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        m.moe_forward_stack(cfg, stack, layer, x, out=out, ws=ws,
                            stream=torch.cuda.current_stream())
    for l in (1, 2, 0, 2, 1):
        layer.fill_(l)
        out.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert_close_layer(out, oracle[l], what=f"graph, stack layer {l}")
        assert torch.equal(out, refs[l]), f"layer {l}"
    assert m.moe_get_device_error(ws) == 0


def test_layer_index_out_of_range_is_reported():
    dev = torch.device("cuda")
    lc = SHAPES[0]
    cfg, x, refs, stack, oracle = bf16_stack(lc, dev, with_bias=False)
    layer = torch.full((1,), NUM_LAYERS, dtype=torch.int32, device=dev)
    ws = m.Workspace(cfg, "forward")
    out = m.moe_forward_stack(cfg, stack, layer, x, ws=ws)   # runs layer 0, flags the index
    torch.cuda.synchronize()
    with pytest.raises(m.MoeError):
        m.moe_get_device_error(ws)
    assert torch.equal(out, refs[0])
    assert_close_layer(out, oracle[0], what="out-of-range index runs layer 0")
    layer.fill_(1)
    out = m.moe_forward_stack(cfg, stack, layer, x, ws=ws)
    torch.cuda.synchronize()
    assert m.moe_get_device_error(ws) == 0
    assert torch.equal(out, refs[1])
    assert_close_layer(out, oracle[1], what="stack layer 1")


def test_fp8_stack_layers_match_single_layer_calls():
    dev = torch.device("cuda")
    lc = wl.DSV3_FP8.with_(name="fp8_stack", T=96, H=512, E=8, k=2, I=384, I_shared=256)
    layers = [Fp8Layer(lc.with_(seed=s), dev) for s in range(2)]
    x = layers[0].x
    cfg = layers[0].cfg
    refs, oracle = [], []
    for l, L in enumerate(layers):
        out, ids, _ = m.moe_forward(cfg, L.weights, x, L.wr, return_routing=True)
        torch.cuda.synchronize()
        refs.append(out)
        r = Routing(f"fp8_stack_layer{l}", lc, cfg, x, L.wr, None, ids.cpu().numpy(), m)
        ref = of8.moe_layer_fp8(f64(x), f64(L.wr), None, L.oracle_expert, L.oracle_shared(),
                                lc.k, lc.score, lc.renormalize, lc.route_scale)
        oracle.append(with_flips(r, ref["out"], lambda t, i, w_, L=L: of8.moe_tokens_fp8(
            f64(x)[t], i, w_, L.oracle_expert, L.oracle_shared())))
    stack = m.LayerStack(cfg, [L.weights for L in layers], [L.wr for L in layers])
    layer = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = m.Workspace(cfg, "forward")
    for l in (1, 0, 1):
        layer.fill_(l)
        out = m.moe_forward_stack(cfg, stack, layer, x, ws=ws)
        torch.cuda.synchronize()
        assert m.moe_get_device_error(ws) == 0
        assert_close_layer(out, oracle[l], max_over_rms=FP8_MAX_OVER_RMS, mean_rel=1.0,
                           what=f"fp8 stack layer {l}")
        assert torch.equal(out, refs[l]), f"layer {l}"
