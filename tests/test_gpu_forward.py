"""moe_forward (route -> permute -> grouped FFN -> combine, one call) on the GPU
against the oracle: whole outputs on small layers; at the workloads' full
sizes, routing over every token (bit-exact off near ties measured from the
GPU's own logits) and a stratified sample of at least 512 output rows that
reaches every expert's first and last row, evaluated by the oracle one
expert at a time."""
import numpy as np
import pytest
import torch

import moe_expert_layer_router_gb300 as m
import workload as wl
from oracle import moe as om
from parity import (BF16_MAX_OVER_RMS, BF16_MEAN_REL, Case, Layer, Routing, assert_close_layer,
                    check_sampled, f64, family_parity, with_flips)

pytestmark = pytest.mark.gpu


def forward(L, lc, fused=False):
    cfg = m.config_from(lc)
    W = m.ExpertWeights(cfg, [w[0] for w in L.W], [w[1] for w in L.W], [w[2] for w in L.W],
                        shared=L.S)
    ws = m.Workspace(cfg, "forward")
    out, ids, w = m.moe_forward(cfg, W, L.x, L.wr, L.bias, return_routing=True,
                                fused_dispatch=fused, ws=ws)
    torch.cuda.synchronize()
    m.moe_get_device_error(ws)
    return out, ids.cpu().numpy(), w.cpu().numpy()


SMALL = [
    wl.TINY,
    wl.TINY.with_(name="tiny_sigmoid_shared", T=200, I_shared=256, score="sigmoid", route_scale=2.5),
    wl.DSV3.with_(name="dsv3_shape_T64", T=64, E=32, k=4, I=256, I_shared=256),
    wl.TINY.with_(name="skewish", T=700, E=16, k=3, H=384, I=128, zipf_bias=False),
    wl.TINY.with_(name="one_token_k1", T=1, k=1),
    wl.TINY.with_(name="e40_k5", T=300, E=40, k=5, H=512, I=256, I_shared=128),
    # about 350 rows per expert: every expert ends in a big tile (256 + tail)
    wl.DSV3.with_(name="big_tiles", T=700, E=4, k=2, H=512, I=256, I_shared=256),
]


@pytest.mark.parametrize("fused", [False, True], ids=["x_perm", "fused_dispatch"])
@pytest.mark.parametrize("lc", SMALL, ids=lambda c: c.name)
def test_forward_small_matches_oracle(lc, fused):
    dev = torch.device("cuda")
    L = Layer(lc, dev)
    out, ids, w = forward(L, lc, fused)
    r = Routing(lc.name, lc, m.config_from(lc), L.x, L.wr, L.bias, ids, m)
    ref = om.moe_layer(f64(L.x), f64(L.wr), None, L.experts_cpu, L.shared_cpu(), lc.k, lc.score,
                       lc.renormalize, lc.route_scale)
    ref_out = with_flips(r, ref["out"], lambda t, i, w_: om.moe_tokens(
        f64(L.x)[t], i, w_, L.experts_cpu, L.shared_cpu()))
    assert_close_layer(out.float().cpu().numpy(), ref_out, what=lc.name)


def test_forward_empty_batch_is_a_noop():
    """T = 0: the call succeeds, launches nothing and leaves the status word clear."""
    dev = torch.device("cuda")
    L = Layer(wl.TINY, dev)
    lc0 = wl.TINY.with_(name="empty", T=0)
    cfg = m.config_from(lc0)
    W = m.ExpertWeights(cfg, [w[0] for w in L.W], [w[1] for w in L.W], [w[2] for w in L.W])
    ws = m.Workspace(cfg, "forward")
    out = m.moe_forward(cfg, W, L.x[:0], L.wr, L.bias, ws=ws)
    torch.cuda.synchronize()
    assert tuple(out.shape) == (0, lc0.H)
    assert m.moe_get_device_error(ws) == 0


# Full-size layers that share the DeepSeek-V3 expert weights (same seed and
# shapes): the prefill batch with and without the fused dispatch, the skewed
# batch, and the small and decode-sized batches.  x[t] depends on t alone, so
# every batch is a prefix of one generated x.
DSV3_FAMILY = [("dsv3", wl.DSV3, False), ("dsv3_fused", wl.DSV3, True),
               ("dsv3_skewed", wl.DSV3_SKEW, False), ("dsv3_bf16_t512", wl.DSV3_T512, False),
               *[(c.name, c, False) for c in wl.DSV3_DECODE]]


@pytest.fixture(scope="module")
def dsv3_family():
    """Runs every DeepSeek-V3-shaped full-size layer on the GPU, checks its routing,
    and compares the stratified samples of all of them with one oracle pass.
    Returns, per layer, its parity record or the failure message."""
    dev = torch.device("cuda")
    base = wl.DSV3
    x_all = wl.gen_x(base.with_(T=max(lc.T for _, lc, _ in DSV3_FAMILY)), dev)
    wr = wl.gen_router(base, dev)
    W = [tuple(wl.gen_expert(base, e, w, dev) for w in ("gate", "up", "down"))
         for e in range(base.E)]
    S = tuple(wl.gen_shared(base, w, dev) for w in ("gate", "up", "down"))
    cases, failed = [], {}
    for name, lc, fused in DSV3_FAMILY:
        x = x_all[:lc.T]
        b = wl.gen_bias(lc)
        bias = b.to(dev) if b is not None else None
        cfg = m.config_from(lc)
        weights = m.ExpertWeights(cfg, [w[0] for w in W], [w[1] for w in W], [w[2] for w in W],
                                  shared=S)
        ws = m.Workspace(cfg, "forward")
        out, ids, _ = m.moe_forward(cfg, weights, x, wr, bias, return_routing=True,
                                    fused_dispatch=fused, ws=ws)
        torch.cuda.synchronize()
        try:
            m.moe_get_device_error(ws)
            r = Routing(name, lc, cfg, x, wr, bias, ids.cpu().numpy(), m)
            if lc.zipf_bias:                           # the workload's defining skew
                counts = np.bincount(r.ref_ids.reshape(-1), minlength=lc.E)
                assert 8.5 <= counts.max() / counts.mean() <= 11.5 and (counts == 0).sum() >= 4
            cases.append(Case(name, lc, r, x, out, BF16_MAX_OVER_RMS, BF16_MEAN_REL))
        except (AssertionError, m.MoeError) as e:
            failed[name] = str(e)
    res = family_parity(cases)
    res.update(failed)
    return res


@pytest.mark.parametrize("name", [n for n, _, _ in DSV3_FAMILY])
def test_forward_full_size_dsv3_family(dsv3_family, name):
    rec = dsv3_family[name]
    assert isinstance(rec, dict), rec
    assert rec["experts_covered"] == rec["experts_with_rows"]


def test_forward_full_size_qwen3():
    dev = torch.device("cuda")
    lc = wl.QWEN3
    L = Layer(lc, dev)
    out, ids, w = forward(L, lc)
    r = Routing(lc.name, lc, m.config_from(lc), L.x, L.wr, L.bias, ids, m)
    rec = check_sampled(lc.name, lc, r, L.x, out, BF16_MAX_OVER_RMS, BF16_MEAN_REL)
    assert rec["experts_covered"] == rec["experts_with_rows"]


@pytest.mark.parametrize("lc", SMALL[:3], ids=lambda c: c.name)
def test_forward_matches_the_four_calls(lc):
    """moe_forward keeps the expert outputs as fp16 with a power-of-two scale per
    32 columns; the four public calls keep them fp32.  On the same routing the two
    outputs differ by that rounding alone.  Each fp16 value is within 2^-12 of its
    fp32 value (relative), so the two fp32 sums differ by at most 2^-12 of the
    summed magnitudes; the two bf16 roundings of the sums then differ by at most
    one bf16 ulp (<= 2^-7 of the output) more.  The test allows 2^-11."""
    dev = torch.device("cuda")
    L = Layer(lc, dev)
    cfg = m.config_from(lc)
    W = m.ExpertWeights(cfg, [w[0] for w in L.W], [w[1] for w in L.W], [w[2] for w in L.W],
                        shared=L.S)
    out, ids, w = m.moe_forward(cfg, W, L.x, L.wr, L.bias, return_routing=True)
    ids2, w2, _ = m.moe_route(cfg, L.x, L.wr, L.bias)
    assert torch.equal(ids, ids2) and torch.equal(w, w2)
    p = m.moe_permute(cfg, ids2, w2, L.x)
    y, s = m.moe_grouped_ffn(cfg, W, p["x_perm"], p["expert_offsets"], p["row_weight"],
                             x_shared=L.x if L.S is not None else None)
    out4 = m.moe_combine(cfg, y, p["inv_row"], s)
    torch.cuda.synchronize()
    a, b = out.float(), out4.float()
    # magnitude of everything summed into each output element
    mag = y.abs()[p["inv_row"].long()].sum(dim=1)
    if s is not None:
        mag = mag + s.abs()
    bound = 2.0 ** -7 * b.abs() + 2.0 ** -11 * mag + 1e-30
    assert ((a - b).abs() <= bound).all(), float(((a - b).abs() / bound).max())
