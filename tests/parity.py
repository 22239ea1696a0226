"""Helpers of the GPU parity tests: tolerances derived from the arithmetic,
near-tie handling for routing, and seeded layer inputs on the device."""
from __future__ import annotations

import atexit
import concurrent.futures as cf
import functools
import json
import multiprocessing as mp
import os

import numpy as np
import torch

import workload as wl
from oracle import fp8 as of8
from oracle import moe as om
from oracle import nvfp4 as onv

# bf16 layer output: max |err| <= 2e-2 * RMS(ref), mean relative (L1 ratio) <= 5e-3;
# fp8 layer output: max |err| <= 6e-2 * RMS(ref)
BF16_MAX_OVER_RMS = 2e-2
BF16_MEAN_REL = 5e-3
FP8_MAX_OVER_RMS = 6e-2
# NVFP4 (no bound on the pages): the GPU and the oracle quantise the same values
# with the same float32 steps, so they differ by fp32 accumulation, the fp16 /
# bf16 output roundings, and the rare E2M1 or e4m3 decision on h that fp32 and
# fp64 take on different sides of a rounding threshold; one such decision moves
# a row by a few percent of RMS at the test sizes, hence the quantised-path bound
# of the fp8 layer, with the bf16 mean bound.
NVFP4_MAX_OVER_RMS = 6e-2
NVFP4_MEAN_REL = 5e-3


def f64(t) -> np.ndarray:
    if isinstance(t, np.ndarray):
        return t.astype(np.float64)
    return t.detach().float().cpu().numpy().astype(np.float64) if t.dtype != torch.float64 \
        else t.detach().cpu().numpy()


def assert_close_layer(got, ref, max_over_rms=BF16_MAX_OVER_RMS, mean_rel=BF16_MEAN_REL, what=""):
    got = f64(got)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    if ref.size == 0:
        return 0.0, 0.0
    rms = float(np.sqrt(np.mean(ref ** 2)))
    err = np.abs(got - ref)
    m = float(err.max()) / rms if rms > 0 else float(err.max())
    r = float(err.sum() / max(np.abs(ref).sum(), 1e-300))
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    assert m <= max_over_rms, f"{what}: max|err|/rms = {m:.3e} > {max_over_rms}"
    assert r <= mean_rel, f"{what}: mean rel = {r:.3e} > {mean_rel}"
    return m, r


def logit_tolerance(x, w_router) -> np.ndarray:
    """Bound on |fp32 logit - exact logit| per (token, expert): the sum runs in
    16-term MMA blocks whose partial sums are accumulated H/16 times in fp32;
    the classic bound gamma_n * sum|x_h W_eh| with n = H/16 + 16 and unit
    roundoff 2^-23 (truncating accumulation), doubled."""
    xa = np.abs(f64(x))
    wa = np.abs(f64(w_router))
    H = xa.shape[1]
    n = H / 16 + 16
    return 2.0 * n * 2.0 ** -23 * (xa @ wa.T) + 1e-30


def routing_tau(logits_gpu, ref_logits) -> np.ndarray:
    """Per-token near-tie threshold from the measured logit error:
    tau_t = max(1e-6, 2 * max_e |l_gpu[t, e] - l_exact[t, e]|).  Two logits whose
    exact gap is above tau_t keep their order in the GPU's fp32 logits."""
    err = np.abs(np.asarray(logits_gpu, dtype=np.float64) - ref_logits)
    return np.maximum(1e-6, 2.0 * err.max(axis=1)) if err.size else np.zeros(len(err))


def near_tie_tokens(ref_logits, k, tau) -> np.ndarray:
    """Tokens whose selection or order can flip under the given per-token (or
    per-element) threshold: some pair of adjacent entries among the exact
    top-(k+1) logits is no further apart than tau.  A flip of any two logits
    that matters for the top-k (or its order) implies such an adjacent pair."""
    E = ref_logits.shape[1]
    srt = -np.sort(-ref_logits, axis=1)[:, :min(k + 1, E)]
    gaps = srt[:, :-1] - srt[:, 1:]
    tau = np.asarray(tau, dtype=np.float64)
    tau = tau.max(axis=1, keepdims=True) if tau.ndim == 2 else tau.reshape(-1, 1)
    return (gaps <= tau).any(axis=1) if gaps.shape[1] else np.zeros(len(srt), bool)


def with_flips(routing, ref_out, tokens_fn):
    """A whole-layer oracle output with every flipped token replaced by
    ``tokens_fn(token_indices, gpu_ids, weights)``, the oracle's per-token sum on
    the GPU's ids (either selection is correct at a near tie)."""
    out = np.array(ref_out, dtype=np.float64, copy=True)
    fl = np.flatnonzero(routing.flipped)
    if len(fl):
        out[fl] = tokens_fn(fl, routing.ids[fl], routing.weights(fl))
    return out


def check_selection_valid(ids, logits_gpu, k):
    """The GPU's ids are the k largest of its own fp32 logits, in descending
    order, equal values in ascending index order (checked without the oracle)."""
    ids = np.asarray(ids)
    lg = np.asarray(logits_gpu, dtype=np.float64)
    T, E = lg.shape
    sel = np.take_along_axis(lg, ids, axis=1)
    assert (np.diff(sel, axis=1) <= 0).all(), "selected logits not descending"
    eq = np.diff(sel, axis=1) == 0
    assert (~eq | (np.diff(ids, axis=1) > 0)).all(), "equal logits not in index order"
    mask = np.ones_like(lg, dtype=bool)
    np.put_along_axis(mask, ids, False, axis=1)
    rest = np.where(mask, lg, -np.inf).max(axis=1)
    assert (sel[:, -1] >= rest).all(), "an unselected logit exceeds a selected one"
    for t in range(T):
        assert len(set(ids[t].tolist())) == k


class Layer:
    """Seeded inputs of one layer config on a device (weights per expert)."""

    def __init__(self, lc: wl.LayerConfig, device):
        self.lc = lc
        self.dev = device
        self.x = wl.gen_x(lc, device)
        self.wr = wl.gen_router(lc, device)
        b = wl.gen_bias(lc)
        self.bias = b.to(device) if b is not None else None
        self.W = [tuple(wl.gen_expert(lc, e, w, device) for w in ("gate", "up", "down"))
                  for e in range(lc.E)]
        self.S = (tuple(wl.gen_shared(lc, w, device) for w in ("gate", "up", "down"))
                  if lc.I_shared else None)

    def experts_cpu(self, e):
        return tuple(f64(t) for t in self.W[e])

    def shared_cpu(self):
        return tuple(f64(t) for t in self.S) if self.S is not None else None


# ---------------------------------------------------------------- reports
REPORT: list[dict] = []


def record(rec: dict) -> None:
    """Keep one parity record for the session summary, and append it as a JSON
    line to the file named by MOE_PARITY_REPORT when that is set."""
    REPORT.append(rec)
    path = os.environ.get("MOE_PARITY_REPORT")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps(rec, sort_keys=True) + "\n")


# ---------------------------------------------------------------- routing
class Routing:
    """Routing of one layer on the GPU checked against the oracle.

    The GPU's fp32 logits come from ``moe_route(..., return_logits=True)`` on the
    layer's inputs; its ids must equal the ids of the call under test (same
    kernel, same inputs).  A token is a near tie when an adjacent pair of its
    exact top-(k+1) logits is within tau_t = max(1e-6, 2 max_e |dl|); on every
    other token the ids must be bit-exact.  Near ties must stay below 1% of the
    tokens (at least 2 are allowed on small batches).  Tokens whose ids differ
    ("flipped", necessarily near ties) are evaluated by the oracle with the
    GPU's ids."""

    def __init__(self, name, lc, cfg, x, wr, bias, ids_gpu, m):
        ids_r, _, lg = m.moe_route(cfg, x, wr, bias, return_logits=True)
        torch.cuda.synchronize()
        self.ids = np.asarray(ids_gpu)
        assert (ids_r.cpu().numpy() == self.ids).all(), "moe_route and the call under test differ"
        lg = lg.cpu().numpy().astype(np.float64)
        b = None if bias is None else f64(bias)
        self.ref_logits = om.router_logits(f64(x), f64(wr), b)
        err = np.abs(lg - self.ref_logits)
        assert (err <= logit_tolerance(x, wr)).all(), f"{name}: logit error {err.max():.3e}"
        self.ref_ids = om.select_topk(self.ref_logits, lc.k)
        tau = routing_tau(lg, self.ref_logits)
        self.tie = near_tie_tokens(self.ref_logits, lc.k, tau)
        self.flipped = (self.ids != self.ref_ids).any(axis=1)
        bad = ~self.tie & self.flipped
        assert not bad.any(), f"{name}: routing differs on {int(bad.sum())} tokens that are not near ties"
        T = len(self.ids)
        assert self.tie.sum() <= max(2, 0.01 * T), f"{name}: {int(self.tie.sum())} near ties of {T}"
        self.lc = lc
        self.rec = dict(config=name, T=int(T), near_ties=int(self.tie.sum()),
                        flipped=int(self.flipped.sum()),
                        tau_max=float(tau.max()) if T else 0.0,
                        max_logit_err=float(err.max()) if T else 0.0)

    def weights(self, tokens):
        """Oracle gate weights of the GPU's ids on the given tokens."""
        lc = self.lc
        return om.routing_weights(self.ref_logits[tokens], self.ids[tokens], lc.score,
                                  lc.renormalize, lc.route_scale)


def stratified_tokens(ids, E, n_min=512, n_random=64, seed=0) -> np.ndarray:
    """Tokens to evaluate at full size: the first and the last token routed to
    every expert with rows (the last lands in that expert's tail tile), the last
    token (the shared expert's last tile), n_random random tokens, and more
    random tokens up to n_min; every token when there are no more than n_min."""
    ids = np.asarray(ids)
    T = len(ids)
    if T <= n_min:
        return np.arange(T)
    pick = {T - 1}
    for e in range(E):
        t = np.flatnonzero((ids == e).any(axis=1))
        if len(t):
            pick.update((int(t[0]), int(t[-1])))
    g = np.random.default_rng(seed)
    rest = np.setdiff1d(np.arange(T), np.fromiter(pick, int))
    extra = max(n_random, n_min - len(pick))
    pick.update(g.choice(rest, size=min(extra, len(rest)), replace=False).tolist())
    return np.array(sorted(pick))


# ---------------------------------------------------------------- oracle pool
CHUNK_ROWS = 128


def _gen_rows(lc, e, which, dtype):
    """Routed expert e's (e = -1: the shared expert's) matrix ``which`` regenerated
    on the host, 128 rows at a time (each slice equals those rows of the matrix)."""
    I = lc.I if e >= 0 else lc.I_shared
    n = I if which in ("gate", "up") else lc.H
    gen = (lambda r0, r: wl.gen_expert(lc, e, which, "cpu", r0, r)) if e >= 0 else \
          (lambda r0, r: wl.gen_shared(lc, which, "cpu", r0, r))
    return np.concatenate([gen(r0, min(CHUNK_ROWS, n - r0)).to(dtype).numpy()
                           for r0 in range(0, n, CHUNK_ROWS)])


def _by_row_chunks(w, fn):
    """fn applied to 128-row slices of w, stacked.  Used only where fn's blocks
    lie within rows (fp8 128 x 128 weight blocks, NVFP4 1 x 16 blocks), so the
    result equals fn(w); the slices keep the temporaries small."""
    return np.concatenate([fn(w[r0:r0 + CHUNK_ROWS]) for r0 in range(0, len(w), CHUNK_ROWS)])


def expert_matrices(lc, e):
    """Routed expert e (e = -1: the shared expert) in the form the oracle's row
    function takes: fp64 (W_gate, W_up, W_down), dequantised through the oracle's
    own codec for fp8 and NVFP4 layers."""
    if lc.wtype == "fp8_e4m3":
        return [_by_row_chunks(_gen_rows(lc, e, w, torch.float32),
                               lambda c: of8.dequant_weight(*of8.quantize_weight_blocks(c)))
                for w in ("gate", "up", "down")]
    if lc.wtype == "nvfp4":
        # gate and up stacked into one matrix with one tensor scale, down on its own
        out = []
        for mats in ((("gate", "up")), ("down",)):
            w = np.concatenate([_gen_rows(lc, e, x, torch.float32) for x in mats])
            g = onv.tensor_scale(w)
            out.append(_by_row_chunks(w, lambda c: onv.dequantize(*onv.quantize_blocks(c, g), g)))
        n = lc.I if e >= 0 else lc.I_shared
        return [out[0][:n], out[0][n:], out[1]]
    return [_gen_rows(lc, e, w, torch.float64) for w in ("gate", "up", "down")]


def expert_job(lc, e, rows):
    """One expert's oracle outputs for the given input rows (runs in a worker)."""
    W = expert_matrices(lc, e)
    if lc.wtype == "fp8_e4m3":
        return of8.expert_rows_fp8(rows, *W)
    if lc.wtype == "nvfp4":
        gx, gh = wl.nvfp4_act_scales(lc)
        return onv.expert_rows_nvfp4(rows, *W, gx, gh)
    return om.swiglu_ffn(rows, *W)


_POOL = None


def oracle_pool():
    """A process pool for the oracle's per-expert work, started with spawn (the
    test process already holds a CUDA context), one BLAS thread per worker."""
    global _POOL
    if _POOL is None:
        for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
            os.environ[v] = "1"
        n = max(1, min(16, (os.cpu_count() or 2) - 1))
        _POOL = cf.ProcessPoolExecutor(max_workers=n, mp_context=mp.get_context("spawn"))
        atexit.register(_POOL.shutdown, wait=False, cancel_futures=True)
    return _POOL


def same_weights(a, b) -> bool:
    """Two layer configs whose seeded expert weights are the same tensors."""
    return all(getattr(a, f) == getattr(b, f)
               for f in ("seed", "H", "E", "I", "I_shared", "wtype", "w_std"))


def oracle_tokens(lc, x_rows, ids, w) -> np.ndarray:
    """The oracle's layer output on the given tokens (rows of x, their ids and
    gate weights), one expert's weights at a time, spread over the pool."""
    pool = oracle_pool()
    x_rows = f64(x_rows)
    shared = pool.submit(expert_job, lc, -1, x_rows) if lc.I_shared else None
    return om.moe_tokens_by_expert(
        x_rows, ids, w, functools.partial(expert_job, lc),
        (lambda xr: shared.result()) if shared is not None else None,
        map_fn=lambda f, a, b: pool.map(f, a, b))


class Case:
    """One full-size layer run on the GPU, waiting for its oracle comparison."""

    def __init__(self, name, lc, routing, x, out, tol_max, tol_mean, n_min=512, seed=0):
        self.name, self.lc, self.routing = name, lc, routing
        self.tol_max, self.tol_mean = tol_max, tol_mean
        self.tokens = stratified_tokens(routing.ids, lc.E, n_min=n_min, seed=seed)
        idx = torch.from_numpy(self.tokens).to(out.device)
        self.x_rows = f64(x[idx])
        self.got = f64(out[idx])
        self.finite = bool(torch.isfinite(out.float()).all())


def family_parity(cases) -> dict:
    """Stratified full-size float parity for layers that share one set of expert
    weights: the sampled tokens of every case go through one oracle pass (each
    expert's weights regenerated and evaluated once), and each case's rows are
    compared element by element with its GPU output.  Returns, per case name,
    the record (also written by ``record``) or the assertion message."""
    base = cases[0].lc
    assert all(same_weights(base, c.lc) for c in cases)
    ids = np.concatenate([c.routing.ids[c.tokens] for c in cases])
    w = np.concatenate([c.routing.weights(c.tokens) for c in cases])
    ref = oracle_tokens(base, np.concatenate([c.x_rows for c in cases]), ids, w)
    res, at = {}, 0
    for c in cases:
        r = ref[at:at + len(c.tokens)]
        at += len(c.tokens)
        try:
            assert c.finite, f"{c.name}: non-finite output"
            mx, mr = assert_close_layer(c.got, r, c.tol_max, c.tol_mean, what=f"{c.name} sampled")
        except AssertionError as e:
            res[c.name] = str(e)
            continue
        rec = dict(c.routing.rec, rows_compared=int(len(c.tokens)),
                   experts_covered=int(len(np.unique(c.routing.ids[c.tokens]))),
                   experts_with_rows=int(len(np.unique(c.routing.ids))),
                   max_err_over_rms=mx, mean_rel=mr)
        record(rec)
        res[c.name] = rec
    return res


def check_sampled(name, lc, routing, x, out_gpu, tol_max, tol_mean, n_min=512, seed=0):
    """Stratified full-size float parity of one layer (see ``family_parity``)."""
    res = family_parity([Case(name, lc, routing, x, out_gpu, tol_max, tol_mean, n_min, seed)])
    assert isinstance(res[name], dict), res[name]
    return res[name]


