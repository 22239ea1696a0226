"""fp8 e4m3 path on the GPU: the block quantisers bit-exact against the oracle's
codec, and the grouped FFN / whole layer against the oracle's fp8 layer
(within the fp8 tolerance, max |err| <= 6e-2 x RMS)."""
import numpy as np
import pytest
import torch

import moe_expert_layer_router_gb300 as m
import workload as wl
from oracle import fp8 as of8
from oracle import moe as om
from parity import (FP8_MAX_OVER_RMS, Case, Routing, assert_close_layer, f64, family_parity,
                    with_flips)

pytestmark = pytest.mark.gpu


def test_weight_quantiser_bit_exact():
    dev = torch.device("cuda")
    w = wl.rng.normal_f32(0, 77, (384, 640), 0.02, dev)
    w[:128, :128] = 0.0
    q, s = m.moe_quantize_weight_fp8(w)
    rq, rs = of8.quantize_weight_blocks(w.cpu().numpy())
    assert (q.cpu().numpy() == rq).all()
    assert (s.cpu().numpy() == rs).all()


def test_activation_quantiser_bit_exact():
    dev = torch.device("cuda")
    x = wl.rng.normal_bf16(0, 78, (300, 1024), 1.0, dev)
    x[3] = 0
    q, s = m.moe_quantize_act_fp8(x)
    rq, rs = of8.quantize_act_groups(f64(x).astype(np.float32))
    assert (q.cpu().numpy() == rq).all()
    assert (s.cpu().numpy() == rs).all()


class Fp8Layer:
    """Seeded fp8 layer: fp32 weights on the device, quantised by the library for
    the GPU path; the oracle quantises its own copy (same codec, decided in fp32)."""

    def __init__(self, lc, dev):
        self.lc, self.dev = lc, dev
        self.x = wl.gen_x(lc, dev)
        self.wr = wl.gen_router(lc, dev)
        self.Wf = [tuple(wl.gen_expert(lc, e, w, dev) for w in ("gate", "up", "down"))
                   for e in range(lc.E)]
        self.Sf = (tuple(wl.gen_shared(lc, w, dev) for w in ("gate", "up", "down"))
                   if lc.I_shared else None)
        self.Q = [tuple(m.moe_quantize_weight_fp8(t) for t in w3) for w3 in self.Wf]
        self.SQ = tuple(m.moe_quantize_weight_fp8(t) for t in self.Sf) if self.Sf else None
        self.cfg = m.config_from(lc)
        self.weights = m.ExpertWeights(
            self.cfg, [w[0][0] for w in self.Q], [w[1][0] for w in self.Q],
            [w[2][0] for w in self.Q],
            shared=tuple(t[0] for t in self.SQ) if self.SQ else None,
            scales=([w[0][1] for w in self.Q], [w[1][1] for w in self.Q], [w[2][1] for w in self.Q]),
            shared_scales=tuple(t[1] for t in self.SQ) if self.SQ else None)

    def oracle_expert(self, e):
        return tuple(of8.dequant_weight(*of8.quantize_weight_blocks(t.cpu().numpy()))
                     for t in self.Wf[e])

    def oracle_shared(self):
        if self.Sf is None:
            return None
        return tuple(of8.dequant_weight(*of8.quantize_weight_blocks(t.cpu().numpy()))
                     for t in self.Sf)


@pytest.mark.parametrize("lc", [
    wl.DSV3_FP8.with_(name="fp8_small", T=96, H=512, E=8, k=2, I=384, I_shared=256),
    wl.DSV3_FP8.with_(name="fp8_ragged", T=150, H=1024, E=4, k=2, I=256, I_shared=0,
                      score="softmax", route_scale=1.0),
    # H = 3 x 128: GEMM2's last 256-column tile has only its first weight block
    wl.DSV3_FP8.with_(name="fp8_h384", T=80, H=384, E=4, k=2, I=256, I_shared=128),
], ids=lambda c: c.name)
def test_fp8_grouped_ffn_matches_oracle(lc):
    dev = torch.device("cuda")
    L = Fp8Layer(lc, dev)
    lg = om.router_logits(f64(L.x), f64(L.wr))
    ids = om.select_topk(lg, lc.k)
    w = om.routing_weights(lg, ids, lc.score, lc.renormalize, lc.route_scale)
    counts, offsets = om.expert_histogram(ids, lc.E)
    perm, slot, _ = om.permutation(ids, lc.E)
    xq, xs = of8.quantize_act_groups(f64(L.x).astype(np.float32))
    rw = w[perm, slot]
    ws = m.Workspace(L.cfg, "grouped_ffn")
    x_shared = torch.from_numpy(xq).to(dev) if lc.I_shared else None
    y, s = m.moe_grouped_ffn(
        L.cfg, L.weights, torch.from_numpy(xq[perm]).to(dev),
        torch.from_numpy(offsets.astype(np.int32)).to(dev),
        torch.from_numpy(rw.astype(np.float32)).to(dev), x_shared,
        x_perm_scales=torch.from_numpy(xs[perm]).to(dev),
        x_shared_scales=torch.from_numpy(xs).to(dev) if lc.I_shared else None, ws=ws)
    torch.cuda.synchronize()
    m.moe_get_device_error(ws)
    xd = of8.dequant_act(xq, xs)
    ref = np.zeros((lc.R, lc.H))
    for e in range(lc.E):
        a, b = offsets[e], offsets[e + 1]
        if b > a:
            ref[a:b] = of8.swiglu_ffn_fp8(xd[perm[a:b]], *L.oracle_expert(e))
    ref *= rw[:, None].astype(np.float32).astype(np.float64)
    assert_close_layer(y, ref, max_over_rms=FP8_MAX_OVER_RMS, mean_rel=1.0, what="fp8 y_perm")
    if lc.I_shared:
        assert_close_layer(s, of8.swiglu_ffn_fp8(xd, *L.oracle_shared()),
                           max_over_rms=FP8_MAX_OVER_RMS, mean_rel=1.0, what="fp8 shared")


def test_fp8_forward_small_matches_oracle():
    """A small fp8 layer, every output row against the oracle's fp8 layer."""
    dev = torch.device("cuda")
    lc = wl.DSV3_FP8.with_(name="fp8_layer_small", T=200, H=1024, E=16, k=4, I=256, I_shared=256)
    L = Fp8Layer(lc, dev)
    ws = m.Workspace(L.cfg, "forward")
    out, ids, w = m.moe_forward(L.cfg, L.weights, L.x, L.wr, return_routing=True, ws=ws)
    torch.cuda.synchronize()
    m.moe_get_device_error(ws)
    r = Routing(lc.name, lc, L.cfg, L.x, L.wr, None, ids.cpu().numpy(), m)
    ref = of8.moe_layer_fp8(f64(L.x), f64(L.wr), None, L.oracle_expert, L.oracle_shared(), lc.k,
                            lc.score, lc.renormalize, lc.route_scale)
    ref_out = with_flips(r, ref["out"], lambda t, i, w_: of8.moe_tokens_fp8(
        f64(L.x)[t], i, w_, L.oracle_expert, L.oracle_shared()))
    assert_close_layer(out, ref_out, max_over_rms=FP8_MAX_OVER_RMS, mean_rel=1.0, what=lc.name)


FP8_FAMILY = [wl.DSV3_FP8, *wl.DSV3_FP8_DECODE]


@pytest.fixture(scope="module")
def fp8_family():
    """The fp8 workload (DeepSeek-V3 shapes, T = 512) and its decode-sized batches,
    which share one set of fp8 expert weights: each runs on the GPU, its routing
    is checked, and every output row of all of them (each token through all of
    its experts) goes through one oracle pass."""
    dev = torch.device("cuda")
    L = Fp8Layer(wl.DSV3_FP8.with_(T=max(lc.T for lc in FP8_FAMILY)), dev)
    cases, failed = [], {}
    for lc in FP8_FAMILY:
        x = L.x[:lc.T]
        cfg = m.config_from(lc)
        ws = m.Workspace(cfg, "forward")
        out, ids, _ = m.moe_forward(cfg, L.weights, x, L.wr, return_routing=True, ws=ws)
        torch.cuda.synchronize()
        try:
            m.moe_get_device_error(ws)
            r = Routing(lc.name, lc, cfg, x, L.wr, None, ids.cpu().numpy(), m)
            cases.append(Case(lc.name, lc, r, x, out, FP8_MAX_OVER_RMS, 1.0))
        except (AssertionError, m.MoeError) as e:
            failed[lc.name] = str(e)
    res = family_parity(cases)
    res.update(failed)
    return res


@pytest.mark.parametrize("lc", FP8_FAMILY, ids=lambda c: c.name)
def test_fp8_forward_full_size(fp8_family, lc):
    rec = fp8_family[lc.name]
    assert isinstance(rec, dict), rec
    assert rec["rows_compared"] == lc.T and rec["experts_covered"] == rec["experts_with_rows"]
