"""Pins of the NVFP4 part of the CPU oracle: hand-worked fixtures
(tests/golden/nvfp4_points.txt), the E2M1 bit fields, a second encoder written
from the rounding intervals, invariants of the two-level quantiser and brute
force on tiny layers.  CPU only."""
import numpy as np
import pytest

from golden_io import lines
from oracle import fp8, moe, nvfp4

rng = np.random.default_rng(4321)


def test_e2m1_decode_from_bit_fields():
    """Every code from its fields: exponent e (2 bits, bias 1), mantissa m:
    e = 0 gives m * 0.5 (subnormal), otherwise (1 + m/2) * 2^(e-1)."""
    for c in range(16):
        e, m = (c >> 1) & 3, c & 1
        mag = m * 0.5 if e == 0 else (1 + m / 2) * 2.0 ** (e - 1)
        assert nvfp4.decode(np.array([c]))[0] == (-mag if c & 8 else mag)


def test_e2m1_golden_points():
    n = 0
    for key, rest in lines("nvfp4_points.txt"):
        if key != "point":
            continue
        v, code = rest.split()
        assert int(nvfp4.encode(np.array([float(v)]))[0]) == int(code, 16), rest
        n += 1
    assert n == 20


def test_e2m1_roundtrip_all_codes():
    codes = np.array([c for c in range(16) if c != 8], dtype=np.uint8)
    assert (nvfp4.encode(nvfp4.decode(codes)) == codes).all()
    assert nvfp4.encode(nvfp4.decode(np.array([8])))[0] == 0      # -0 is written as +0


def test_e2m1_encoder_equals_interval_encoder():
    mags = nvfp4.E2M1_MAG
    mids = (mags[1:] + mags[:-1]) / 2
    v = np.concatenate([rng.normal(size=40000) * 3, rng.uniform(-8, 8, size=40000),
                        mids, -mids, mags, -mags, np.nextafter(mids, 0), np.nextafter(mids, 9),
                        [0.0, -0.0, 6.0, 7.0, 1e9, -1e9, 1e-30]])
    assert (nvfp4.encode(v) == nvfp4.encode_intervals(v)).all()


def test_e2m1_is_nearest_value():
    """The decoded code is a nearest representable value (brute force over all
    eight magnitudes), and never further than the saturation point."""
    v = rng.uniform(-6, 6, size=20000)
    got = nvfp4.decode(nvfp4.encode(v))
    best = np.abs(np.abs(v)[:, None] - nvfp4.E2M1_MAG[None, :]).min(axis=1)
    assert np.allclose(np.abs(np.abs(v) - np.abs(got)), best)
    assert (np.sign(got) * np.sign(v) >= 0).all()


def test_golden_blocks():
    n = 0
    for key, rest in lines("nvfp4_points.txt"):
        if key != "block":
            continue
        g, xs, sc, cs = (p.strip() for p in rest.split("|"))
        x = np.array([[float(v) for v in xs.split()]], dtype=np.float32)
        q, s = nvfp4.quantize_blocks(x, np.float32(g))
        assert int(s[0, 0]) == int(sc, 16), rest
        assert [int(c) for c in q[0]] == [int(c, 16) for c in cs.split()], rest
        n += 1
    assert n == 4


def test_tensor_scale_maps_amax_to_the_top_code():
    """g = amax / 2688: the largest element's block scale is 448 and the
    element itself encodes to +-6."""
    w = (rng.normal(size=(64, 256)) * 0.02).astype(np.float32)
    i, j = np.unravel_index(np.abs(w).argmax(), w.shape)
    q, s, g = nvfp4.quantize_weight(w)
    assert g == np.float32(np.float32(np.abs(w).max()) / np.float32(2688.0))
    assert fp8.decode(s[i, j // 16]) == 448.0
    assert nvfp4.decode(q[i, j]) == np.sign(w[i, j]) * 6.0


def test_quantisation_error_bound():
    """Within a block of scale s: |x - deq| <= s*g (half the widest spacing,
    2, of E2M1, and the saturation of the top code when s rounded down)."""
    w = (rng.normal(size=(32, 512)) * 0.05).astype(np.float32)
    w[3, 16:32] = 0.0
    q, s, g = nvfp4.quantize_weight(w)
    deq = nvfp4.dequantize(q, s, g)
    bound = np.repeat(fp8.decode(s), 16, axis=1) * np.float64(g)
    assert (np.abs(deq - w) <= bound * (1 + 1e-6)).all()
    assert (q[3, 16:32] == 0).all() and s[3, 1] == 0
    # the block amax lands on a top code (4 or 6) unless its scale underflows
    blk = np.abs(w).reshape(32, 32, 16)
    top = nvfp4.E2M1_MAG[q.reshape(32, 32, 16)[np.arange(32)[:, None], np.arange(32)[None, :],
                                               blk.argmax(axis=2)] & 7]
    assert (top[s != 0] >= 4).all()


def test_power_of_two_rescaling_is_exact():
    """Scaling a matrix by 2^k scales its tensor scale by 2^k and leaves every
    code and block scale unchanged."""
    w = (rng.normal(size=(16, 128)) * 0.02).astype(np.float32)
    q0, s0, g0 = nvfp4.quantize_weight(w)
    q1, s1, g1 = nvfp4.quantize_weight(w * np.float32(8.0))
    assert g1 == g0 * 8 and (q0 == q1).all() and (s0 == s1).all()


def test_all_zero_matrix():
    q, s, g = nvfp4.quantize_weight(np.zeros((4, 32), np.float32))
    assert g == 1.0 and (q == 0).all() and (s == 0).all()


def test_block_scale_saturates_with_a_small_static_scale():
    """An activation block beyond 6 * 448 * g saturates its scale at 448 and its
    top elements at 6: the static scale bounds the range."""
    x = np.zeros((1, 16), np.float32)
    x[0, 0], x[0, 1] = 5000.0, -1.0
    q, s = nvfp4.quantize_blocks(x, np.float32(1.0))
    assert fp8.decode(s[0, 0]) == 448.0 and nvfp4.decode(q[0, 0]) == 6.0
    assert nvfp4.decode(q[0, 1]) == 0.0                         # 1/448 rounds to zero


def test_stacked_gate_up_equals_separate_rows():
    """Block scales are per row: quantising [W_g; W_u] as one matrix gives each
    row the codes it gets alone under the shared tensor scale."""
    wg = (rng.normal(size=(32, 128)) * 0.02).astype(np.float32)
    wu = (rng.normal(size=(32, 128)) * 0.03).astype(np.float32)
    (qgu, sgu, g), _ = nvfp4.quantize_expert(wg, wu, np.zeros((128, 32), np.float32))
    assert g == nvfp4.tensor_scale(np.concatenate([wg, wu]))
    qg, sg = nvfp4.quantize_blocks(wg, g)
    qu, su = nvfp4.quantize_blocks(wu, g)
    assert (qgu[:32] == qg).all() and (qgu[32:] == qu).all()
    assert (sgu[:32] == sg).all() and (sgu[32:] == su).all()


def _layer_inputs(T, H, E, k, I):
    x = rng.normal(size=(T, H)).astype(np.float32)
    wr = (rng.normal(size=(E, H)) * 0.02).astype(np.float32)
    W = [tuple((rng.normal(size=s) * 0.02).astype(np.float32) for s in ((I, H), (I, H), (H, I)))
         for _ in range(E)]
    sh = tuple((rng.normal(size=s) * 0.02).astype(np.float32) for s in ((I, H), (I, H), (H, I)))
    return x, wr, W, sh


def _grid_weights(shape):
    """Weights exactly representable in NVFP4 under the weight rule: E2M1
    values times an e4m3 scale per 16-element block times g = 2^-9, every
    block holding one +-6 (so its amax / (6 g) is its scale) and one block
    scaled by 448 (so amax / 2688 is g)."""
    codes = rng.integers(0, 16, size=shape)
    codes[:, ::16] = rng.choice([7, 15], size=codes[:, ::16].shape)
    s = fp8.decode(rng.integers(0x30, 0x70, size=(shape[0], shape[1] // 16)))
    s[0, 0] = 448.0
    return (nvfp4.decode(codes) * np.repeat(s, 16, axis=1) * 2.0 ** -9).astype(np.float32)


def test_layer_on_representable_weights_equals_bf16_layer():
    """With weights already on the NVFP4 grid and activations left unquantised,
    quantise-dequantise is the identity and the NVFP4 layer is the plain layer."""
    T, H, E, k, I = 7, 64, 4, 2, 32
    x = rng.normal(size=(T, H)).astype(np.float32)
    wr = (rng.normal(size=(E, H)) * 0.02).astype(np.float32)
    W = [(_grid_weights((I, H)), _grid_weights((I, H)), _grid_weights((H, I))) for _ in range(E)]
    Wq = [nvfp4.dequantize_expert(*nvfp4.quantize_expert(*w)) for w in W]
    for a, b in zip(W, Wq):
        for m_a, m_b in zip(a, b):
            assert (m_a.astype(np.float64) == m_b).all()
    r = nvfp4.moe_layer_nvfp4(x, wr, None, lambda e: Wq[e], None, k, "softmax", True, 1.0,
                              quantize_activations=False)
    ref = moe.moe_layer(x, wr, None, lambda e: W[e], None, k, "softmax", True, 1.0)
    np.testing.assert_allclose(r["out"], ref["out"], rtol=1e-12, atol=1e-12)


def test_bruteforce_equals_grouped_nvfp4_layer():
    T, H, E, k, I = 11, 128, 4, 2, 64
    x, wr, W, sh = _layer_inputs(T, H, E, k, I)
    Wd = [nvfp4.dequantize_expert(*nvfp4.quantize_expert(*w)) for w in W]
    shd = nvfp4.dequantize_expert(*nvfp4.quantize_expert(*sh))
    gx, gh = 2.0 ** -8, 2.0 ** -4
    r = nvfp4.moe_layer_nvfp4(x, wr, None, lambda e: Wd[e], shd, k, "sigmoid", True, 2.5, gx, gh)
    bf = nvfp4.moe_tokens_nvfp4(x, r["ids"], r["weights"], lambda e: Wd[e], shd, gx, gh)
    np.testing.assert_allclose(bf, r["out"], rtol=1e-12, atol=1e-12)
    # the quantised layer stays close to the unquantised one (NVFP4 noise, bounded)
    ref = moe.moe_layer(x, wr, None, lambda e: W[e], sh, k, "sigmoid", True, 2.5)
    rel = np.abs(r["out"] - ref["out"]).mean() / np.abs(ref["out"]).mean()
    assert 1e-3 < rel < 0.3


def test_by_expert_equals_bruteforce_nvfp4():
    T, H, E, k, I = 13, 128, 5, 2, 64
    x, wr, W, sh = _layer_inputs(T, H, E, k, I)
    Wd = [nvfp4.dequantize_expert(*nvfp4.quantize_expert(*w)) for w in W]
    shd = nvfp4.dequantize_expert(*nvfp4.quantize_expert(*sh))
    gx, gh = 2.0 ** -8, 2.0 ** -4
    r = nvfp4.moe_layer_nvfp4(x, wr, None, lambda e: Wd[e], shd, k, "sigmoid", True, 2.5, gx, gh)
    be = moe.moe_tokens_by_expert(x, r["ids"], r["weights"],
                                  lambda e, xr: nvfp4.expert_rows_nvfp4(xr, *Wd[e], gx, gh),
                                  lambda xr: nvfp4.expert_rows_nvfp4(xr, *shd, gx, gh))
    np.testing.assert_allclose(be, r["out"], rtol=1e-12, atol=1e-12)
    bf = nvfp4.moe_tokens_nvfp4(x, r["ids"], r["weights"], lambda e: Wd[e], shd, gx, gh)
    np.testing.assert_allclose(be, bf, rtol=1e-12, atol=1e-12)


def test_activation_quantisation_is_per_row():
    """Each token is quantised on its own: quantising a stack of rows equals
    quantising each row alone (so quantise-then-gather equals gather-then-quantise)."""
    x = rng.normal(size=(6, 64)).astype(np.float32)
    q, s = nvfp4.quantize_blocks(x, np.float32(2.0 ** -8))
    for t in range(6):
        qt, st = nvfp4.quantize_blocks(x[t:t + 1], np.float32(2.0 ** -8))
        assert (qt[0] == q[t]).all() and (st[0] == s[t]).all()
