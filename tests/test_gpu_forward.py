"""moe_forward (route -> permute -> grouped FFN -> combine, one call) on the GPU
against the oracle: whole outputs on small layers, and at the five workloads'
full sizes, routing over every token plus sampled output rows computed one
token at a time by the oracle."""
import numpy as np
import pytest
import torch

import moe_expert_layer_router_gb300 as m
import workload as wl
from oracle import moe as om
from parity import Layer, assert_close_layer, f64, logit_tolerance, near_tie_tokens

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
]


@pytest.mark.parametrize("fused", [False, True], ids=["x_perm", "fused_dispatch"])
@pytest.mark.parametrize("lc", SMALL, ids=lambda c: c.name)
def test_forward_small_matches_oracle(lc, fused):
    dev = torch.device("cuda")
    L = Layer(lc, dev)
    out, ids, w = forward(L, lc, fused)
    ref = om.moe_layer(f64(L.x), f64(L.wr), None, L.experts_cpu, L.shared_cpu(), lc.k, lc.score,
                       lc.renormalize, lc.route_scale)
    tie = near_tie_tokens(ref["logits"], lc.k, logit_tolerance(L.x, L.wr))
    assert (ids[~tie] == ref["ids"][~tie]).all()
    keep = ~tie & (ids == ref["ids"]).all(axis=1)
    assert_close_layer(out.float().cpu().numpy()[keep], ref["out"][keep], what=lc.name)


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


FULL = [(wl.QWEN3, False), (wl.DSV3, False), (wl.DSV3_SKEW, False), (wl.DSV3, True),
        (wl.DSV3_T512, False)]


@pytest.mark.parametrize("lc,fused", FULL,
                         ids=lambda c: c.name if hasattr(c, "name") else ("fused" if c else ""))
def test_forward_full_size_sampled(lc, fused):
    dev = torch.device("cuda")
    L = Layer(lc, dev)
    out, ids, w = forward(L, lc, fused)
    b = None if L.bias is None else f64(L.bias)
    ref_lg = om.router_logits(f64(L.x), f64(L.wr), b)
    ref_ids = om.select_topk(ref_lg, lc.k)
    tie = near_tie_tokens(ref_lg, lc.k, logit_tolerance(L.x, L.wr))
    assert (ids[~tie] == ref_ids[~tie]).all()
    counts, _ = om.expert_histogram(ref_ids, lc.E)
    if lc.zipf_bias:                                   # the workload's defining skew
        assert 8.5 <= counts.max() / counts.mean() <= 11.5 and (counts == 0).sum() >= 4
    g = np.random.default_rng(0)
    cand = np.flatnonzero(~tie)
    sample = np.sort(g.choice(cand, size=6, replace=False))
    ref_w = om.routing_weights(ref_lg[sample], ref_ids[sample], lc.score, lc.renormalize,
                               lc.route_scale)
    ref = om.moe_tokens(f64(L.x[torch.from_numpy(sample).to(dev)]), ref_ids[sample], ref_w,
                        L.experts_cpu, L.shared_cpu())
    assert_close_layer(out[torch.from_numpy(sample).to(dev)], ref, what=f"{lc.name} sampled")
    assert torch.isfinite(out.float()).all()
    print(f"{lc.name}: T={lc.T} near-tie tokens {int(tie.sum())}, max/mean rows "
          f"{counts.max() / counts.mean():.2f}")


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
