"""moe_route on the GPU against the oracle: fp32 logits within the accumulation
bound, ids bit-exact except on near-tie tokens (reported), gate weights within
the bound their logits imply."""
import numpy as np
import pytest
import torch

import moe_expert_layer_router_gb300 as m
import workload as wl
from oracle import moe as om
from parity import (check_selection_valid, f64, logit_tolerance, near_tie_tokens, record,
                    routing_tau)

pytestmark = pytest.mark.gpu

CASES = [
    wl.TINY,                                                             # E=8, k=2, softmax
    wl.TINY.with_(name="t1", T=1),
    wl.TINY.with_(name="ragged", T=333, E=16, k=4, H=1024),
    wl.DSV3.with_(name="dsv3_router_small", T=517),                      # E=256, k=8, sigmoid x2.5
    wl.DSV3_SKEW.with_(name="skew_router_small", T=300),                 # + Zipf bias
    wl.QWEN3.with_(name="qwen_router_small", T=200),                     # E=128, k=8
    wl.TINY.with_(name="k1", E=32, k=1, T=130, score="sigmoid", renormalize=False),
    wl.TINY.with_(name="softmax_full", E=64, k=6, T=200, renormalize=False),
    wl.TINY.with_(name="k16", E=48, k=16, T=140, H=256),
    wl.TINY.with_(name="e40", E=40, k=5, T=300, H=512),                   # E_pad = 48: 8 padded columns
    # more than one 128-token tile per SM pair: unsplit K; E_pad = 48 keeps single
    # CTAs, E_pad = 64 runs CTA pairs (79 tiles, the last pair half past T)
    wl.TINY.with_(name="unsplit_e40", E=40, k=5, T=10000, H=512),
    wl.TINY.with_(name="pairs_softmax_full", E=64, k=6, T=10000, H=256, renormalize=False),
    wl.TINY.with_(name="pairs_k16", E=64, k=16, T=10000, H=256, score="sigmoid"),
]


def run_route(lc, dev):
    x = wl.gen_x(lc, dev)
    wr = wl.gen_router(lc, dev)
    b = wl.gen_bias(lc)
    b = b.to(dev) if b is not None else None
    cfg = m.config_from(lc)
    ws = m.Workspace(cfg, "route")
    ids, w, lg = m.moe_route(cfg, x, wr, b, return_logits=True, ws=ws)
    torch.cuda.synchronize()
    m.moe_get_device_error(ws)
    return x, wr, b, ids.cpu().numpy(), w.cpu().numpy().astype(np.float64), lg.cpu().numpy()


@pytest.mark.parametrize("lc", CASES, ids=lambda c: c.name)
def test_route_matches_oracle(lc):
    dev = torch.device("cuda")
    x, wr, b, ids, w, lg = run_route(lc, dev)
    ref_lg = om.router_logits(f64(x), f64(wr), None if b is None else f64(b))
    tol = logit_tolerance(x, wr)
    err = np.abs(lg.astype(np.float64) - ref_lg)
    assert (err <= tol).all(), f"logit error {err.max():.3e} above bound"
    ref_ids = om.select_topk(ref_lg, lc.k)
    ref_w = om.routing_weights(ref_lg, ref_ids, lc.score, lc.renormalize, lc.route_scale)
    tie = near_tie_tokens(ref_lg, lc.k, routing_tau(lg, ref_lg))
    ok = ~tie
    assert (ids[ok] == ref_ids[ok]).all(), "routing differs on a token that is not a near tie"
    check_selection_valid(ids, lg, lc.k)
    # weights: |d log w| <= 2 max|d logit| for softmax / normalised sigmoid, plus fp32 rounding
    dl = err.max(axis=1, keepdims=True)
    rel = np.abs(w[ok] - ref_w[ok]) / np.abs(ref_w[ok])
    assert (rel <= 2 * dl[ok] + 2e-6).all(), f"weight rel error {rel.max():.3e}"
    print(f"{lc.name}: near-tie tokens {int(tie.sum())}/{lc.T}, max logit err {err.max():.2e}")


def test_route_all_equal_logits_pick_lowest_experts():
    """Zero router weights: every logit is 0 (+ bias 0); selection must be 0..k-1."""
    dev = torch.device("cuda")
    lc = wl.TINY.with_(T=129, E=16, k=4, score="sigmoid", route_scale=2.5)
    cfg = m.config_from(lc)
    x = wl.gen_x(lc, dev)
    wr = torch.zeros(lc.E, lc.H, dtype=torch.bfloat16, device=dev)
    ids, w, _ = m.moe_route(cfg, x, wr)
    assert (ids.cpu().numpy() == np.arange(4)[None, :]).all()
    np.testing.assert_allclose(w.cpu().numpy(), 2.5 / 4, rtol=1e-6)


def test_route_bias_decides_ties():
    """Equal logits broken by the bias: larger bias wins regardless of index."""
    dev = torch.device("cuda")
    lc = wl.TINY.with_(T=64, E=8, k=3)
    cfg = m.config_from(lc)
    x = wl.gen_x(lc, dev)
    wr = torch.zeros(lc.E, lc.H, dtype=torch.bfloat16, device=dev)
    b = torch.tensor([0, 1, 0, 3, 0, 2, 0, 0], dtype=torch.float32, device=dev)
    ids, w, _ = m.moe_route(cfg, x, wr, b)
    assert (ids.cpu().numpy() == np.array([3, 5, 1])[None, :]).all()
    e = np.exp([3.0, 2.0, 1.0])
    np.testing.assert_allclose(w.cpu().numpy(), (e / e.sum())[None, :].repeat(64, 0), rtol=1e-6)


# T = 64, 2000, 5000, 10000 give K splits S = 8, 4, 2, 1 on a 152-SM GPU, so the
# selection runs with Q = 4 S = 32, 16, 8, 4 finishing threads per token.
@pytest.mark.parametrize("T", [64, 2000, 5000, 10000])
@pytest.mark.parametrize("pattern", ["one_owner", "tied_boundary"])
def test_route_exact_logits_selection(T, pattern):
    """Logits set exactly (x[:, 0] = 1, router column 0 = the logit, every other
    router column 0), so the selection has one right answer, taken from the
    oracle's stable top-k.  one_owner: the k best are experts 0..k-1, which the
    same finishing thread owns; tied_boundary: six experts share the k-th largest
    value, and the lowest-indexed of them must be taken."""
    dev = torch.device("cuda")
    E, k, H = 64, 4, 256
    lc = wl.TINY.with_(T=T, E=E, k=k, H=H, score="softmax", renormalize=True, I_shared=0)
    cfg = m.config_from(lc)
    x = wl.gen_x(lc, dev)
    x[:, 0] = 1.0
    # distinct values in [-4, 0) on a 1/16 grid: exact in bf16 and in fp32 sums
    v = np.random.default_rng(5).permutation(np.arange(E)) / 16.0 - 4.0
    if pattern == "one_owner":
        v[:k] = 4.0 + np.arange(k)[::-1]
    else:
        v[[50, 20, 7]] = [3.0, 2.5, 2.25]
        v[[5, 9, 17, 33, 40, 63]] = 2.0
    wr = torch.zeros(E, H, dtype=torch.bfloat16, device=dev)
    wr[:, 0] = torch.tensor(v, dtype=torch.bfloat16, device=dev)
    ids, w, lg = m.moe_route(cfg, x, wr, return_logits=True)
    exact = np.broadcast_to(v, (T, E))
    np.testing.assert_array_equal(lg.cpu().numpy().astype(np.float64), exact)
    ref = om.select_topk(exact, k)
    np.testing.assert_array_equal(ids.cpu().numpy(), ref)
    if pattern == "tied_boundary":
        assert (ref[:, 3] == 5).all()


def test_route_full_size_dsv3():
    """Full DeepSeek-V3 router shape (T=16384, H=7168, E=256, k=8)."""
    dev = torch.device("cuda")
    lc = wl.DSV3
    x, wr, b, ids, w, lg = run_route(lc, dev)
    ref_lg = om.router_logits(f64(x), f64(wr))
    err = np.abs(lg.astype(np.float64) - ref_lg)
    assert (err <= logit_tolerance(x, wr)).all()
    ref_ids = om.select_topk(ref_lg, lc.k)
    tau = routing_tau(lg, ref_lg)
    tie = near_tie_tokens(ref_lg, lc.k, tau)
    assert (ids[~tie] == ref_ids[~tie]).all()
    assert tie.sum() <= 0.01 * lc.T
    check_selection_valid(ids, lg, lc.k)
    record(dict(config="dsv3_route", T=lc.T, near_ties=int(tie.sum()),
                flipped=int((ids != ref_ids).any(1).sum()), tau_max=float(tau.max()),
                max_logit_err=float(err.max())))
