"""Host logic of the GPU parity harness, checked on the CPU: the oracle's view of
each expert's weights (regenerated and dequantised 128 rows at a time) equals
the oracle's codec applied to the whole matrix, the stratified token sample
reaches every expert's first and last token, the near-tie rule flags exactly
the tokens whose order a logit error of the given size can change, and the
weight-family comparison passes a correct output and reports a wrong one."""
import numpy as np
import pytest
import torch

import workload as wl
from oracle import fp8 as of8
from oracle import moe as om
from oracle import nvfp4 as onv
from parity import (BF16_MAX_OVER_RMS, BF16_MEAN_REL, Case, expert_matrices, f64, family_parity,
                    near_tie_tokens, routing_tau, stratified_tokens)

SMALL = wl.TINY.with_(name="harness", T=96, H=256, E=6, k=2, I=384, I_shared=256)


def _whole(lc, e):
    mats = ([wl.gen_expert(lc, e, w) for w in ("gate", "up", "down")] if e >= 0 else
            [wl.gen_shared(lc, w) for w in ("gate", "up", "down")])
    if lc.wtype == "fp8_e4m3":
        return [of8.dequant_weight(*of8.quantize_weight_blocks(t.numpy())) for t in mats]
    if lc.wtype == "nvfp4":
        return list(onv.dequantize_expert(*onv.quantize_expert(*(f64(t) for t in mats))))
    return [f64(t) for t in mats]


@pytest.mark.parametrize("wtype", ["bf16", "fp8_e4m3", "nvfp4"])
def test_expert_matrices_equal_the_whole_matrix_codec(wtype):
    lc = SMALL.with_(wtype=wtype)
    for e in (0, 5, -1):
        for a, b in zip(expert_matrices(lc, e), _whole(lc, e)):
            assert a.shape == b.shape and (a == b).all()


def test_stratified_tokens_reach_every_expert():
    g = np.random.default_rng(1)
    T, E, k = 3000, 40, 4
    ids = np.argsort(g.random((T, E - 1)), axis=1)[:, :k]   # expert 39 receives no token
    tok = stratified_tokens(ids, E, n_min=512, n_random=64)
    assert len(tok) >= 512 and len(set(tok.tolist())) == len(tok) and T - 1 in tok
    for e in range(E):
        t = np.flatnonzero((ids == e).any(axis=1))
        if len(t):
            assert t[0] in tok and t[-1] in tok
    small = stratified_tokens(ids[:300], E, n_min=512)
    assert (small == np.arange(300)).all()


def test_near_ties_follow_the_measured_logit_error():
    ref = np.array([[5.0, 4.0, 3.0, 2.0],          # gaps 1: no tie at tau 1e-3
                    [5.0, 4.9995, 3.0, 2.0],       # gap 5e-4 among the top 2
                    [5.0, 4.0, 3.0, 2.9995],       # gap 5e-4 below the top k+1 = 3: no tie
                    [5.0, 4.0005, 4.0, 2.0]])      # gap 5e-4 between k-th and (k+1)-th
    gpu = ref + np.array([[1e-4, 0, 0, 0]] * 4) / 2    # |dl| max 5e-5 -> tau = 1e-4
    tau = routing_tau(gpu, ref)
    assert np.allclose(tau, 1e-4)
    assert near_tie_tokens(ref, 2, tau).tolist() == [False, False, False, False]
    tie = near_tie_tokens(ref, 2, np.full(4, 1e-3))
    assert tie.tolist() == [False, True, False, True]
    assert routing_tau(ref, ref).min() == 1e-6      # never below 1e-6


class _Routing:
    """The slice of parity.Routing that family_parity reads, from the oracle."""

    def __init__(self, lc, x, wr):
        self.lc = lc
        self.ref_logits = om.router_logits(f64(x), f64(wr))
        self.ids = om.select_topk(self.ref_logits, lc.k)
        self.rec = dict(config=lc.name, T=lc.T)

    def weights(self, tokens):
        lc = self.lc
        return om.routing_weights(self.ref_logits[tokens], self.ids[tokens], lc.score,
                                  lc.renormalize, lc.route_scale)


def test_family_parity_passes_the_oracle_and_reports_a_wrong_row():
    lc = SMALL.with_(score="sigmoid", route_scale=2.5)
    x, wr = wl.gen_x(lc), wl.gen_router(lc)
    W = [_whole(lc, e) for e in range(lc.E)]
    S = _whole(lc, -1)
    r = _Routing(lc, x, wr)
    exact = om.moe_tokens(f64(x), r.ids, r.weights(np.arange(lc.T)), lambda e: W[e], S)
    good = torch.from_numpy(exact)
    bad = good.clone()
    bad[7, 3] += 0.5 * float(np.sqrt(np.mean(exact ** 2)))
    res = family_parity([Case("good", lc, r, x, good, BF16_MAX_OVER_RMS, BF16_MEAN_REL),
                         Case("bad", lc.with_(name="bad"), r, x, bad, BF16_MAX_OVER_RMS,
                              BF16_MEAN_REL)])
    assert isinstance(res["good"], dict) and res["good"]["rows_compared"] == lc.T
    assert res["good"]["max_err_over_rms"] < 1e-12
    assert isinstance(res["bad"], str) and "max|err|/rms" in res["bad"]
