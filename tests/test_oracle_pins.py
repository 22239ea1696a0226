"""Pins of the CPU oracle against facts that do not come from the oracle itself:
hand-worked fixtures (tests/golden/), closed forms, invariants, brute force on
tiny inputs and library routines.  CPU only."""
import itertools

import numpy as np
import pytest
import torch
from scipy.special import expit

from golden_io import lines, matrix, vector
from oracle import fp8, moe

rng = np.random.default_rng(1234)


# ------------------------------------------------------------- selection
def test_topk_golden_ties():
    n = 0
    for _, rest in lines("topk_ties.txt"):
        head, lg, want = [p.strip() for p in rest.split("|")]
        E, k = (int(v) for v in head.split())
        logits = vector(lg)[None, :]
        assert logits.shape[1] == E
        got = moe.select_topk(logits, k)[0]
        assert got.tolist() == vector(want, int).tolist(), rest
        n += 1
    assert n == 5


def _argmax_rounds(row, k):
    """Independent brute force: k rounds of 'take the largest remaining logit,
    the first index among equals'."""
    left = list(range(len(row)))
    out = []
    for _ in range(k):
        best = left[0]
        for e in left[1:]:
            if row[e] > row[best]:
                best = e
        out.append(best)
        left.remove(best)
    return out


@pytest.mark.parametrize("E,k", [(8, 2), (16, 4), (5, 5), (32, 8), (7, 1)])
def test_topk_bruteforce(E, k):
    # quantised logits so exact ties are common
    lg = np.round(rng.normal(size=(64, E)) * 2) / 2
    ids = moe.select_topk(lg, k)
    for t in range(lg.shape[0]):
        assert ids[t].tolist() == _argmax_rounds(lg[t], k)
        assert len(set(ids[t].tolist())) == k


def test_topk_all_equal_logits_pick_first_experts():
    lg = np.zeros((4, 9))
    assert moe.select_topk(lg, 3).tolist() == [[0, 1, 2]] * 4


def test_topk_set_is_maximal():
    """Every selected logit >= every unselected logit (checked over all subsets on tiny E)."""
    lg = rng.normal(size=(10, 6))
    for t in range(10):
        sel = set(moe.select_topk(lg[t:t + 1], 3)[0].tolist())
        best = max(itertools.combinations(range(6), 3), key=lambda s: sum(lg[t, list(s)]))
        assert sel == set(best)


# ------------------------------------------------------------- weights
def test_routing_weights_golden():
    n = 0
    for _, rest in lines("routing_weights.txt"):
        head, lg, want = [p.strip() for p in rest.split("|")]
        score, scale = head.split()
        sel = vector(lg)[None, :]
        ids = np.arange(sel.shape[1])[None, :]
        w = moe.routing_weights(sel, ids, score, True, float(scale))[0]
        np.testing.assert_allclose(w, vector(want), rtol=1e-14, atol=1e-15)
        n += 1
    assert n == 5


def test_softmax_renorm_two_forms_agree():
    lg = rng.normal(size=(50, 16)) * 3
    ids = moe.select_topk(lg, 4)
    a = moe.routing_weights(lg, ids, "softmax", True, 1.0)
    b = moe.softmax_all_then_renormalize(lg, ids)
    np.testing.assert_allclose(a, b, rtol=1e-13)


def test_softmax_two_experts_closed_form():
    lg = rng.normal(size=(20, 8))
    ids = moe.select_topk(lg, 2)
    w = moe.routing_weights(lg, ids, "softmax", True, 1.0)
    l0 = np.take_along_axis(lg, ids[:, :1], 1)[:, 0]
    l1 = np.take_along_axis(lg, ids[:, 1:], 1)[:, 0]
    np.testing.assert_allclose(w[:, 0], expit(l0 - l1), rtol=1e-13)


@pytest.mark.parametrize("score,scale", [("softmax", 1.0), ("sigmoid", 2.5), ("sigmoid", 1.0)])
def test_weights_sum_to_scale(score, scale):
    lg = rng.normal(size=(40, 12)) * 2
    ids = moe.select_topk(lg, 5)
    w = moe.routing_weights(lg, ids, score, True, scale)
    np.testing.assert_allclose(w.sum(1), scale, rtol=1e-13)
    assert (w > 0).all()
    # weights follow the selection order (descending logits)
    assert (np.diff(w, axis=1) <= 1e-15).all()


def test_weights_uniform_when_logits_equal():
    lg = np.zeros((3, 10))
    ids = moe.select_topk(lg, 4)
    np.testing.assert_allclose(moe.routing_weights(lg, ids, "softmax", True, 1.0), 0.25)
    np.testing.assert_allclose(moe.routing_weights(lg, ids, "sigmoid", True, 2.5), 2.5 / 4)


def test_sigmoid_without_renorm_is_expit():
    lg = rng.normal(size=(7, 9))
    ids = moe.select_topk(lg, 3)
    w = moe.routing_weights(lg, ids, "sigmoid", False, 1.0)
    np.testing.assert_allclose(w, expit(np.take_along_axis(lg, ids, 1)), rtol=1e-14)


def test_softmax_without_renorm_is_full_softmax():
    lg = rng.normal(size=(7, 9))
    ids = moe.select_topk(lg, 3)
    w = moe.routing_weights(lg, ids, "softmax", False, 1.0)
    p = torch.softmax(torch.from_numpy(lg), dim=1).numpy()
    np.testing.assert_allclose(w, np.take_along_axis(p, ids, 1), rtol=1e-13)


def test_logits_bias_and_library_matmul():
    x = rng.normal(size=(5, 7))
    wr = rng.normal(size=(4, 7))
    b = rng.normal(size=4)
    lg = moe.router_logits(x, wr, b)
    ref = np.array([[sum(x[t, h] * wr[e, h] for h in range(7)) + b[e] for e in range(4)]
                    for t in range(5)])
    np.testing.assert_allclose(lg, ref, rtol=1e-13)


# ------------------------------------------------------------- histogram / permutation
def test_permutation_golden():
    d = dict(lines("permutation_3tok.txt"))
    ids = matrix(d["ids"], int)
    counts, offsets = moe.expert_histogram(ids, 3)
    perm, slot, inv = moe.permutation(ids, 3)
    assert counts.tolist() == vector(d["counts"], int).tolist()
    assert offsets.tolist() == vector(d["offsets"], int).tolist()
    assert perm.tolist() == vector(d["perm_token"], int).tolist()
    assert inv.tolist() == matrix(d["inv_row"], int).tolist()


def _random_ids(T, E, k):
    lg = rng.normal(size=(T, E))
    return moe.select_topk(lg, k)


@pytest.mark.parametrize("T,E,k", [(1, 1, 1), (37, 8, 2), (100, 16, 4), (64, 64, 8), (5, 3, 3)])
def test_histogram_and_permutation_invariants(T, E, k):
    ids = _random_ids(T, E, k)
    counts, offsets = moe.expert_histogram(ids, E)
    assert counts.tolist() == np.bincount(ids.ravel(), minlength=E).tolist()
    assert counts.sum() == T * k and offsets[-1] == T * k and offsets[0] == 0
    perm, slot, inv = moe.permutation(ids, E)
    R = T * k
    assert sorted(perm.tolist()) == sorted(np.repeat(np.arange(T), k).tolist())
    assert sorted(inv.ravel().tolist()) == list(range(R))           # bijection
    for t in range(T):
        for j in range(k):
            r = inv[t, j]
            assert perm[r] == t and slot[r] == j                     # inverse
            e = ids[t, j]
            assert offsets[e] <= r < offsets[e + 1]                  # right segment
    for e in range(E):
        seg = perm[offsets[e]:offsets[e + 1]]
        assert (np.diff(seg) > 0).all()                              # ascending tokens
        assert set(seg.tolist()) == {t for t in range(T) if e in ids[t]}


# ------------------------------------------------------------- experts / layer
def test_silu_matches_library():
    z = np.linspace(-30, 30, 601)
    np.testing.assert_allclose(moe.silu(z), z * expit(z), rtol=1e-14, atol=1e-300)


def test_swiglu_golden():
    d = dict(lines("swiglu_2x2.txt"))
    x = vector(d["x"])[None, :]
    wg, wu, wd = matrix(d["w_gate"]), matrix(d["w_up"]), matrix(d["w_down"])
    h = moe.silu(x @ wg.T) * (x @ wu.T)
    np.testing.assert_allclose(h[0], vector(d["h"]), rtol=1e-15)
    np.testing.assert_allclose(moe.swiglu_ffn(x, wg, wu, wd)[0], vector(d["y"]), rtol=1e-15)


def _layer_inputs(T, H, E, k, I, Is):
    x = rng.normal(size=(T, H))
    wr = rng.normal(size=(E, H)) * 0.3
    W = [(rng.normal(size=(I, H)) * 0.2, rng.normal(size=(I, H)) * 0.2,
          rng.normal(size=(H, I)) * 0.2) for _ in range(E)]
    sh = None
    if Is:
        sh = (rng.normal(size=(Is, H)) * 0.2, rng.normal(size=(Is, H)) * 0.2,
              rng.normal(size=(H, Is)) * 0.2)
    return x, wr, W, sh


@pytest.mark.parametrize("score,scale,Is", [("softmax", 1.0, 0), ("sigmoid", 2.5, 6)])
def test_grouped_equals_bruteforce(score, scale, Is):
    T, H, E, k, I = 23, 8, 6, 3, 5
    x, wr, W, sh = _layer_inputs(T, H, E, k, I, Is)
    r = moe.moe_layer(x, wr, None, lambda e: W[e], sh, k, score, True, scale)
    bf = moe.moe_tokens(x, r["ids"], r["weights"], lambda e: W[e], sh)
    np.testing.assert_allclose(r["out"], bf, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("score,scale,Is", [("softmax", 1.0, 0), ("sigmoid", 2.5, 6)])
def test_by_expert_equals_bruteforce(score, scale, Is):
    """The expert-by-expert evaluation (one expert's weights at a time) gives the
    per-token sum, on all tokens and on a subset of them, whatever order the
    per-expert calls run in."""
    T, H, E, k, I = 31, 8, 7, 3, 5
    x, wr, W, sh = _layer_inputs(T, H, E, k, I, Is)
    r = moe.moe_layer(x, wr, None, lambda e: W[e], sh, k, score, True, scale)
    rows = lambda e, xr: moe.swiglu_ffn(xr, *W[e])
    shared = (lambda xr: moe.swiglu_ffn(xr, *sh)) if sh else None
    be = moe.moe_tokens_by_expert(x, r["ids"], r["weights"], rows, shared)
    np.testing.assert_allclose(be, r["out"], rtol=1e-12, atol=1e-12)
    sub = np.array([0, 4, 5, 17, 30])
    rev = lambda f, a, b: reversed([f(*z) for z in reversed(list(zip(a, b)))])
    be2 = moe.moe_tokens_by_expert(x[sub], r["ids"][sub], r["weights"][sub], rows, shared, rev)
    bf = moe.moe_tokens(x[sub], r["ids"][sub], r["weights"][sub], lambda e: W[e], sh)
    np.testing.assert_allclose(be2, bf, rtol=1e-12, atol=1e-12)
    # a wrong weight or a dropped shared expert is visible
    assert not np.allclose(moe.moe_tokens_by_expert(x, r["ids"], r["weights"][:, ::-1], rows,
                                                    shared), r["out"])


def test_single_expert_is_dense_swiglu():
    T, H, I = 9, 6, 4
    x, wr, W, _ = _layer_inputs(T, H, 1, 1, I, 0)
    r = moe.moe_layer(x, wr, None, lambda e: W[e], None, 1, "softmax", True, 1.0)
    assert (r["ids"] == 0).all()
    np.testing.assert_allclose(r["weights"], 1.0)
    g = x @ W[0][0].T
    dense = (g * expit(g)) * (x @ W[0][1].T) @ W[0][2].T
    np.testing.assert_allclose(r["out"], dense, rtol=1e-12, atol=1e-12)


def test_zero_down_projection_leaves_shared_expert():
    T, H, E, k, I, Is = 11, 6, 4, 2, 5, 3
    x, wr, W, sh = _layer_inputs(T, H, E, k, I, Is)
    W0 = [(a, b, np.zeros_like(c)) for a, b, c in W]
    r = moe.moe_layer(x, wr, None, lambda e: W0[e], sh, k, "sigmoid", True, 2.5)
    g = x @ sh[0].T
    np.testing.assert_allclose(r["out"], (g * expit(g)) * (x @ sh[1].T) @ sh[2].T,
                               rtol=1e-12, atol=1e-12)


def test_relabelling_experts_changes_nothing():
    T, H, E, k, I = 17, 6, 7, 3, 4
    x, wr, W, _ = _layer_inputs(T, H, E, k, I, 0)
    r = moe.moe_layer(x, wr, None, lambda e: W[e], None, k, "softmax", True, 1.0)
    p = rng.permutation(E)                      # new expert i is old expert p[i]
    r2 = moe.moe_layer(x, wr[p], None, lambda e: W[p[e]], None, k, "softmax", True, 1.0)
    np.testing.assert_allclose(r2["out"], r["out"], rtol=1e-12, atol=1e-12)
    assert (p[r2["ids"]] == r["ids"]).all()


def test_down_projection_linearity():
    T, H, E, k, I = 13, 6, 5, 2, 4
    x, wr, W, _ = _layer_inputs(T, H, E, k, I, 0)
    W2 = [(a, b, 2.0 * c) for a, b, c in W]
    r = moe.moe_layer(x, wr, None, lambda e: W[e], None, k, "sigmoid", True, 2.5)
    r2 = moe.moe_layer(x, wr, None, lambda e: W2[e], None, k, "sigmoid", True, 2.5)
    np.testing.assert_allclose(r2["out"], 2.0 * r["out"], rtol=1e-12, atol=1e-12)


def test_combine_by_hand():
    y = np.arange(12.0).reshape(6, 2)
    inv = np.array([[2, 0], [1, 4], [3, 5]])
    s = np.ones((3, 2))
    out = moe.combine(y, inv, s)
    assert out.tolist() == [[1 + 4 + 0, 1 + 5 + 1], [1 + 2 + 8, 1 + 3 + 9], [1 + 6 + 10, 1 + 7 + 11]]


# ------------------------------------------------------------- e4m3 codec
def test_e4m3_golden_points():
    n = 0
    for _, rest in lines("e4m3_points.txt"):
        v, code = rest.split()
        assert int(fp8.encode(np.array([float(v)]))[0]) == int(code, 16), rest
        n += 1
    assert n == 15


def test_e4m3_decode_matches_torch_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = fp8.decode(codes)
    nan = np.isnan(ref)
    assert (np.isnan(got) == nan).all() and nan.sum() == 2
    assert (got[~nan] == ref[~nan]).all()
    assert np.nanmax(got) == 448.0


def test_e4m3_roundtrip_all_finite_codes():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    assert (fp8.encode(fp8.decode(codes)) == codes).all()


def test_e4m3_encode_matches_torch_rne():
    # random values over the whole range plus all midpoints between neighbours
    mags = fp8.decode(np.arange(127, dtype=np.uint8))
    mids = (mags[1:] + mags[:-1]) / 2
    v = np.concatenate([rng.normal(size=20000) * 50, rng.normal(size=5000) * 1e-2,
                        mids, -mids, mags, rng.uniform(-447, 447, 5000)]).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = fp8.encode(v)
    assert (got == ref).all()


def test_e4m3_saturates():
    assert fp8.encode(np.array([1e30, -1e30, 449.0, 463.9]))[:].tolist() == [0x7E, 0xFE, 0x7E, 0x7E]


def test_block_quantisation_error_bound_and_scales():
    w = (rng.normal(size=(256, 384)) * 0.02).astype(np.float32)
    w[:128, :128] = 0.0                                            # an all-zero block
    q, s = fp8.quantize_weight_blocks(w)
    assert s.shape == (2, 3) and s[0, 0] == 1.0
    deq = fp8.dequant_weight(q, s)
    for bi in range(2):
        for bk in range(3):
            blk = w[bi * 128:(bi + 1) * 128, bk * 128:(bk + 1) * 128].astype(np.float64)
            d = deq[bi * 128:(bi + 1) * 128, bk * 128:(bk + 1) * 128]
            amax = np.abs(blk).max()
            if amax == 0:
                assert (d == 0).all()
                continue
            assert np.abs(d).max() == pytest.approx(amax, rel=1e-6)   # amax -> code 448
            # e4m3 half-ulp: 2^-4 relative for normals, 2^-10 * s absolute near 0
            err = np.abs(d - blk)
            bound = np.maximum(np.abs(blk) * 2.0 ** -4, 2.0 ** -10 * s[bi, bk]) * (1 + 1e-6)
            assert (err <= bound).all()


def test_activation_groups_match_per_row_blocks():
    x = (rng.normal(size=(5, 256))).astype(np.float32)
    q, s = fp8.quantize_act_groups(x)
    assert s.shape == (5, 2)
    for t in range(5):
        for g in range(2):
            seg = x[t, g * 128:(g + 1) * 128]
            assert s[t, g] == np.float32(np.abs(seg).max()) / np.float32(448.0)
            assert (q[t, g * 128:(g + 1) * 128] == fp8.encode((seg / s[t, g]).astype(np.float32))).all()


def test_fp8_layer_without_quantisation_equals_bf16_layer():
    T, H, E, k, I = 9, 128, 4, 2, 128
    x, wr, W, sh = _layer_inputs(T, H, E, k, I, 128)
    a = fp8.moe_layer_fp8(x, wr, None, lambda e: W[e], sh, k, "sigmoid", True, 2.5,
                          quantize_activations=False)
    b = moe.moe_layer(x, wr, None, lambda e: W[e], sh, k, "sigmoid", True, 2.5)
    np.testing.assert_allclose(a["out"], b["out"], rtol=1e-12, atol=1e-12)
    c = fp8.moe_layer_fp8(x, wr, None, lambda e: W[e], sh, k, "sigmoid", True, 2.5)
    rel = np.abs(c["out"] - b["out"]).mean() / np.abs(b["out"]).mean()
    assert 1e-4 < rel < 0.1                                       # quantisation noise, bounded


def test_fp8_bruteforce_equals_grouped_fp8_layer():
    T, H, E, k, I = 11, 256, 4, 2, 128
    x, wr, W, sh = _layer_inputs(T, H, E, k, I, 128)
    Wd = [tuple(fp8.dequant_weight(*fp8.quantize_weight_blocks(m_.astype(np.float32))) for m_ in w3)
          for w3 in W]
    shd = tuple(fp8.dequant_weight(*fp8.quantize_weight_blocks(m_.astype(np.float32))) for m_ in sh)
    r = fp8.moe_layer_fp8(x, wr, None, lambda e: Wd[e], shd, k, "sigmoid", True, 2.5)
    bf = fp8.moe_tokens_fp8(x, r["ids"], r["weights"], lambda e: Wd[e], shd)
    np.testing.assert_allclose(bf, r["out"], rtol=1e-12, atol=1e-12)


def test_fp8_by_expert_equals_bruteforce():
    T, H, E, k, I = 13, 256, 5, 2, 128
    x, wr, W, sh = _layer_inputs(T, H, E, k, I, 128)
    Wd = [tuple(fp8.dequant_weight(*fp8.quantize_weight_blocks(m_.astype(np.float32))) for m_ in w3)
          for w3 in W]
    shd = tuple(fp8.dequant_weight(*fp8.quantize_weight_blocks(m_.astype(np.float32))) for m_ in sh)
    r = fp8.moe_layer_fp8(x, wr, None, lambda e: Wd[e], shd, k, "sigmoid", True, 2.5)
    be = moe.moe_tokens_by_expert(x, r["ids"], r["weights"],
                                  lambda e, xr: fp8.expert_rows_fp8(xr, *Wd[e]),
                                  lambda xr: fp8.expert_rows_fp8(xr, *shd))
    np.testing.assert_allclose(be, r["out"], rtol=1e-12, atol=1e-12)
    bf = fp8.moe_tokens_fp8(x, r["ids"], r["weights"], lambda e: Wd[e], shd)
    np.testing.assert_allclose(be, bf, rtol=1e-12, atol=1e-12)


def test_e4m3_table_encoder_equals_bitfield_encoder():
    mags = fp8.decode(np.arange(127, dtype=np.uint8))
    mids = (mags[1:] + mags[:-1]) / 2
    v = np.concatenate([rng.normal(size=50000) * 30, rng.normal(size=20000) * 1e-2,
                        rng.normal(size=5000) * 1e-3, mids, -mids, mags, -mags,
                        np.nextafter(mids, 0), np.nextafter(mids, 1e9), [0.0, -0.0, 448.0, 449.0,
                        1e9, -1e9, 2.0 ** -6, 2.0 ** -10, 2.0 ** -11]])
    assert (fp8.encode(v) == fp8.encode_bitfield(v)).all()
