"""moe_permute on the GPU: histogram, offsets, permutation maps, row weights and
the gathered rows bit-exact against the oracle, fed the oracle's routing."""
import numpy as np
import pytest
import torch

import moe_expert_layer_router_gb300 as m
import workload as wl
from oracle import fp8 as of8
from oracle import moe as om
from parity import f64

pytestmark = pytest.mark.gpu


def oracle_routing(lc, x, wr, b=None):
    lg = om.router_logits(f64(x), f64(wr), None if b is None else f64(b))
    ids = om.select_topk(lg, lc.k)
    w = om.routing_weights(lg, ids, lc.score, lc.renormalize, lc.route_scale)
    return ids, w


def run_permute(lc, ids, w, x, dev):
    cfg = m.config_from(lc)
    ws = m.Workspace(cfg, "permute")
    o = m.moe_permute(cfg, torch.from_numpy(ids.astype(np.int32)).to(dev),
                      torch.from_numpy(w.astype(np.float32)).to(dev), x, ws=ws)
    torch.cuda.synchronize()
    m.moe_get_device_error(ws)
    return o


def check_against_oracle(lc, ids, w32, x, o):
    counts, offsets = om.expert_histogram(ids, lc.E)
    perm, slot, inv = om.permutation(ids, lc.E)
    assert (o["expert_counts"].cpu().numpy() == counts).all()
    assert (o["expert_offsets"].cpu().numpy() == offsets).all()
    assert (o["perm_token"].cpu().numpy() == perm).all()
    assert (o["inv_row"].cpu().numpy() == inv).all()
    assert (o["row_weight"].cpu().numpy() == w32[perm, slot]).all()
    if o["x_perm"] is not None and lc.wtype == "bf16":
        xp = o["x_perm"].cpu()
        assert torch.equal(xp, x.cpu()[torch.from_numpy(perm)])


@pytest.mark.parametrize("lc", [
    wl.TINY,
    wl.TINY.with_(name="t1", T=1),
    wl.TINY.with_(name="t65", T=65, E=16, k=4, H=256),
    wl.TINY.with_(name="e1", E=1, k=1, T=100),
    wl.TINY.with_(name="k16", E=32, k=16, T=190, H=128),
    wl.DSV3.with_(name="dsv3_1000", T=1000),
], ids=lambda c: c.name)
def test_permute_matches_oracle(lc):
    dev = torch.device("cuda")
    x = wl.gen_x(lc, dev)
    ids, w = oracle_routing(lc, x, wl.gen_router(lc, dev))
    w32 = w.astype(np.float32)
    o = run_permute(lc, ids, w32, x, dev)
    check_against_oracle(lc, ids, w32, x, o)


def test_permute_skewed_and_empty_experts():
    """Every token picks experts 0..k-1: the other experts get no rows."""
    dev = torch.device("cuda")
    lc = wl.TINY.with_(T=300, E=64, k=4, H=256)
    x = wl.gen_x(lc, dev)
    ids = np.tile(np.array([3, 0, 2, 1]), (lc.T, 1))
    w = np.full((lc.T, 4), 0.25, np.float32)
    o = run_permute(lc, ids, w, x, dev)
    check_against_oracle(lc, ids, w, x, o)
    assert (o["expert_counts"].cpu().numpy()[4:] == 0).all()


def test_permute_full_size_dsv3_random_ids():
    """Full DeepSeek-V3 batch (T=16384, k=8, E=256): random distinct ids per token."""
    dev = torch.device("cuda")
    lc = wl.DSV3
    g = np.random.default_rng(7)
    ids = np.argsort(g.random((lc.T, lc.E)), axis=1)[:, :lc.k].astype(np.int64)
    w = g.random((lc.T, lc.k)).astype(np.float32)
    x = wl.gen_x(lc, dev)
    o = run_permute(lc, ids, w, x, dev)
    check_against_oracle(lc, ids, w, x, o)


def test_permute_fp8_codes_and_scales():
    """fp8 layers: each token quantised once (1x128 groups) and gathered; codes and
    scales bit-exact against the oracle's codec (decisions in fp32 on both sides)."""
    dev = torch.device("cuda")
    lc = wl.DSV3_FP8.with_(T=200)
    x = wl.gen_x(lc, dev)
    ids, w = oracle_routing(lc, x, wl.gen_router(lc, dev))
    o = run_permute(lc, ids, w.astype(np.float32), x, dev)
    perm, _, _ = om.permutation(ids, lc.E)
    q, s = of8.quantize_act_groups(f64(x).astype(np.float32))
    assert (o["x_perm"].cpu().numpy() == q[perm]).all()
    assert (o["x_perm_scales"].cpu().numpy() == s[perm]).all()


def test_permute_reports_bad_ids():
    """An id outside [0, E) is skipped and flagged in the status word, not trapped."""
    dev = torch.device("cuda")
    lc = wl.TINY.with_(T=64, E=8, k=2, H=128)
    cfg = m.config_from(lc)
    ids = np.tile(np.array([0, 1]), (64, 1)).astype(np.int32)
    ids[5, 1] = 99
    ws = m.Workspace(cfg, "permute")
    m.moe_permute(cfg, torch.from_numpy(ids).to(dev), ws=ws)
    torch.cuda.synchronize()
    with pytest.raises(m.MoeError, match="out-of-range"):
        m.moe_get_device_error(ws)
    assert m.moe_get_device_error(ws) == 0          # cleared after reading


def test_permute_reports_repeated_ids():
    """A token that lists one expert in two slots is flagged (status bit 3):
    every row index stays in range, but one row of that expert is not written."""
    dev = torch.device("cuda")
    lc = wl.TINY.with_(T=130, E=8, k=3, H=128)
    cfg = m.config_from(lc)
    ids = np.tile(np.array([0, 1, 2]), (130, 1)).astype(np.int32)
    ids[77, 2] = 0
    ws = m.Workspace(cfg, "permute")
    m.moe_permute(cfg, torch.from_numpy(ids).to(dev), ws=ws)
    torch.cuda.synchronize()
    with pytest.raises(m.MoeError, match="same expert twice"):
        m.moe_get_device_error(ws)
    assert m.moe_get_device_error(ws) == 0
