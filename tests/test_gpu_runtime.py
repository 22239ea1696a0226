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


def test_a_wait_that_runs_out_is_reported_and_the_next_call_recovers():
    """Failure detection on the GPU without a fault: the test hook makes the first
    CTA pair of GEMM1 wait on a barrier that nothing signals.  The bounded wait
    gives up (2 s), the pair abandons its tiles, drains its loads and frees its
    tensor memory, and the status word reports the timeout; the next call on the
    same workspace matches the oracle."""
    from moe_expert_layer_router_gb300 import _native as N
    from oracle import moe as om
    from parity import Routing, assert_close_layer, f64, with_flips

    dev = torch.device("cuda")
    lc = LC.with_(name="stall", T=600)
    L = Layer(lc, dev)
    cfg = m.config_from(lc)
    W = weights_of(L, cfg)
    ws = m.Workspace(cfg, "forward")
    N.check(N.lib().moe_test_stall_gemm1(1), "moe_test_stall_gemm1")
    try:
        m.moe_forward(cfg, W, L.x, L.wr, L.bias, ws=ws)
        torch.cuda.synchronize()
        with pytest.raises(m.MoeError) as ei:
            m.moe_get_device_error(ws)
        assert ei.value.status == N.MOE_ERR_DEVICE_TIMEOUT
    finally:
        N.lib().moe_test_stall_gemm1(0)
    out, ids, _ = m.moe_forward(cfg, W, L.x, L.wr, L.bias, ws=ws, return_routing=True)
    torch.cuda.synchronize()
    assert m.moe_get_device_error(ws) == 0
    r = Routing(lc.name, lc, cfg, L.x, L.wr, L.bias, ids.cpu().numpy(), m)
    ref = om.moe_layer(f64(L.x), f64(L.wr), None, L.experts_cpu, L.shared_cpu(), lc.k, lc.score,
                       lc.renormalize, lc.route_scale)
    ref_out = with_flips(r, ref["out"], lambda t, i, w_: om.moe_tokens(
        f64(L.x)[t], i, w_, L.experts_cpu, L.shared_cpu()))
    assert_close_layer(out, ref_out, what="after the stalled call")


def _trace(n, mask):
    from moe_expert_layer_router_gb300 import _native as N
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    for e in evs:
        e.record()
    torch.cuda.synchronize()
    arr = (N.C.c_void_p * n)(*[e.cuda_event for e in evs])
    kid = (N.C.c_int32 * n)()
    t = N.MoeTrace(N.C.cast(arr, N.C.POINTER(N.C.c_void_p)),
                   N.C.cast(kid, N.C.POINTER(N.C.c_int32)), n, 0, mask)
    return t, kid, evs


def test_trace_marks_every_kernel_or_the_masked_ones():
    """The trace hook: without a mask an event before each of the layer's 8
    kernels and one after the last; with the GEMM1 and GEMM2 bits, exactly the
    two events that bracket GEMM1, and the output is unchanged."""
    from moe_expert_layer_router_gb300 import _native as N
    dev = torch.device("cuda")
    L = Layer(LC, dev)
    cfg = m.config_from(LC)
    W = weights_of(L, cfg)
    ws = m.Workspace(cfg, "forward")
    ref = m.moe_forward(cfg, W, L.x, L.wr, L.bias, ws=ws)
    torch.cuda.synchronize()
    g1, g2 = N.KERNEL_NAMES.index("gemm1_gate_up_swiglu"), N.KERNEL_NAMES.index("gemm2_down")
    for mask, want in ((0, [0, 1, 2, 3, 4, g1, g2, 7, -1]), ((1 << g1) | (1 << g2), [g1, g2])):
        t, kid, evs = _trace(16, mask)
        N.check(N.lib().moe_set_trace(N.C.byref(t)), "moe_set_trace")
        try:
            out = m.moe_forward(cfg, W, L.x, L.wr, L.bias, ws=ws)
        finally:
            N.lib().moe_set_trace(None)
        torch.cuda.synchronize()
        assert [kid[i] for i in range(t.count)] == want
        assert torch.equal(out, ref)
        assert evs[0].elapsed_time(evs[1]) >= 0.0
