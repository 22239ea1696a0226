"""moe_grouped_ffn (tcgen05 grouped GEMMs) on the GPU against the oracle's
grouped evaluation, on permuted rows prepared by the oracle."""
import numpy as np
import pytest
import torch

import moe_expert_layer_router_gb300 as m
import workload as wl
from oracle import moe as om
from parity import Layer, assert_close_layer, f64

pytestmark = pytest.mark.gpu


def run_ffn(lc, L, x_perm, offsets, row_weight, with_shared=True):
    dev = L.dev
    cfg = m.config_from(lc)
    W = m.ExpertWeights(cfg, [w[0] for w in L.W], [w[1] for w in L.W], [w[2] for w in L.W],
                        shared=L.S)
    ws = m.Workspace(cfg, "grouped_ffn")
    y, s = m.moe_grouped_ffn(cfg, W, x_perm, torch.from_numpy(offsets.astype(np.int32)).to(dev),
                             None if row_weight is None else
                             torch.from_numpy(row_weight.astype(np.float32)).to(dev),
                             x_shared=L.x if (with_shared and L.S is not None) else None, ws=ws)
    torch.cuda.synchronize()
    m.moe_get_device_error(ws)
    return y, s


@pytest.mark.parametrize("lc", [
    wl.TINY,                                                                  # 4 k-steps x 8 n-tiles
    wl.TINY.with_(name="shared", T=300, E=8, k=2, H=640, I=256, I_shared=384,
                  score="sigmoid", route_scale=2.5),                          # H % 256 != 0, Is != I
    wl.TINY.with_(name="wide", T=150, E=16, k=4, H=1024, I=512),
], ids=lambda c: c.name)
def test_grouped_ffn_matches_oracle(lc):
    dev = torch.device("cuda")
    L = Layer(lc, dev)
    lg = om.router_logits(f64(L.x), f64(L.wr))
    ids = om.select_topk(lg, lc.k)
    w = om.routing_weights(lg, ids, lc.score, lc.renormalize, lc.route_scale)
    counts, offsets = om.expert_histogram(ids, lc.E)
    perm, slot, _ = om.permutation(ids, lc.E)
    rw = w[perm, slot].astype(np.float32)
    x_perm = L.x[torch.from_numpy(perm).to(dev)].contiguous()
    y, s = run_ffn(lc, L, x_perm, offsets, rw)
    ref = om.grouped_ffn(f64(x_perm), offsets, L.experts_cpu, rw.astype(np.float64))
    assert_close_layer(y, ref, what="y_perm")
    if L.S is not None:
        assert_close_layer(s, om.swiglu_ffn(f64(L.x), *L.shared_cpu()), what="shared_out")


def test_grouped_ffn_ragged_segments():
    """Hand-made expert segments: empty, 1, 127, 128, 129, 300 rows; no row weights."""
    dev = torch.device("cuda")
    sizes = [0, 1, 127, 128, 129, 0, 300, 5]
    R = sum(sizes)
    lc = wl.TINY.with_(T=R, E=len(sizes), k=1, H=256, I=384)
    L = Layer(lc, dev)
    offsets = np.concatenate([[0], np.cumsum(sizes)])
    y, _ = run_ffn(lc, L, L.x, offsets, None)
    ref = om.grouped_ffn(f64(L.x), offsets, L.experts_cpu)
    assert_close_layer(y, ref, what="ragged")


def test_grouped_ffn_tile_boundaries():
    """Segments on every side of the GEMM1 tile boundaries: a group's last 1..128
    rows join the 256-row tile before them (a big tile of 257..384 rows), 129..256
    rows make a tile of their own; with and without the shared expert."""
    dev = torch.device("cuda")
    sizes = [256, 257, 300, 383, 384, 385, 511, 512, 513, 640, 641, 767, 768, 769, 1, 200]
    R = sum(sizes)
    for I_shared in (0, 256):
        lc = wl.TINY.with_(name=f"bounds_s{I_shared}", T=R, E=len(sizes), k=1, H=256, I=256,
                           I_shared=I_shared)
        L = Layer(lc, dev)
        offsets = np.concatenate([[0], np.cumsum(sizes)])
        rw = np.linspace(0.5, 1.5, R).astype(np.float32)
        y, s = run_ffn(lc, L, L.x, offsets, rw)
        ref = om.grouped_ffn(f64(L.x), offsets, L.experts_cpu, rw.astype(np.float64))
        assert_close_layer(y, ref, what=lc.name)
        if I_shared:
            assert_close_layer(s, om.swiglu_ffn(f64(L.x), *L.shared_cpu()), what="shared_out")


def test_grouped_ffn_single_expert_is_dense_swiglu():
    """E = 1: one group holding every row; output = the dense SwiGLU FFN."""
    dev = torch.device("cuda")
    lc = wl.TINY.with_(T=513, E=1, k=1, H=512, I=512)
    L = Layer(lc, dev)
    y, _ = run_ffn(lc, L, L.x, np.array([0, lc.T]), None)
    ref = om.swiglu_ffn(f64(L.x), *L.experts_cpu(0))
    assert_close_layer(y, ref, what="dense")


def test_grouped_ffn_row_weights_scale_rows():
    dev = torch.device("cuda")
    lc = wl.TINY.with_(T=200, E=4, k=1, H=256, I=256)
    L = Layer(lc, dev)
    offsets = np.array([0, 50, 100, 150, 200])
    rw = np.linspace(-2, 3, 200).astype(np.float32)
    y, _ = run_ffn(lc, L, L.x, offsets, rw)
    ref = om.grouped_ffn(f64(L.x), offsets, L.experts_cpu, rw.astype(np.float64))
    assert_close_layer(y, ref, what="row weights")
