"""NVFP4 codec, two-level block quantisation and the NVFP4 layer (test
infrastructure only).

The pages name the format and nothing more: the DWDP write-up's experimental
setup (section A4, hardware, software and model) runs DeepSeek-R1 from an
NVFP4 checkpoint whose MoE weights are NVFP4.  What follows is the format as NVIDIA publishes it, plus the readings
the pages leave open.

Element: E2M1 (OCP Microscaling Formats (MX) v1.0, FP4): 1 sign bit, 2 exponent
bits (bias 1), 1 mantissa bit, no infinities or NaN.  The eight magnitudes are
0, 0.5, 1, 1.5, 2, 3, 4, 6.  Encoding rounds to the nearest magnitude, ties to
the even code, saturates beyond 6, and writes a value that rounds to zero as
code 0 (never the negative zero 0x8).

Scaling: each run of 16 consecutive elements along the contraction dimension
shares one E4M3 scale (the fp8 codec in ``fp8.py``), and a float32 tensor scale
g widens the range: value = e2m1 * e4m3 * g.

Quantising a tensor with tensor scale g (every step in float32, round to
nearest):
    d    = 6 * g
    s    = e4m3(amax_block / d)              (round to nearest even, saturating at 448)
    q    = e2m1(x / (decode(s) * g))         (q = 0 for the whole block if decode(s) == 0)
Readings (the pages are silent; "parity unpinned" beyond the published format):
  * weights: g = amax(W) / (6 * 448) over the whole matrix (g = 1 for an
    all-zero matrix), so the largest element maps to exactly 6 * 448 * g.  The
    gate and up projections of one expert share one tensor scale (they are
    quantised as one stacked matrix).
  * activations: the tensor scale is a static per-layer constant supplied with
    the weights, as NVFP4 checkpoints carry one ("input scale"): g_x for the
    expert inputs (each token quantised once, before dispatch) and g_h for the
    intermediate h, quantised per row after the SwiGLU, rounded to float32
    first.  The 16-element block scales are computed at run time.
"""
from __future__ import annotations

import numpy as np

from . import fp8, moe

BLOCK = 16
E2M1_MAX = 6.0
E4M3_MAX = 448.0

# magnitude of the 3-bit code (exponent field << 1 | mantissa bit)
E2M1_MAG = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def decode(codes) -> np.ndarray:
    """4-bit codes (0..15) -> float64."""
    c = np.asarray(codes).astype(np.int64)
    mag = E2M1_MAG[c & 7]
    return np.where(c & 8, -mag, mag)


def encode(v) -> np.ndarray:
    """float -> 4-bit code: nearest of the eight magnitudes, ties to the even
    code, saturating at 6; zero magnitude always code 0."""
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    lo = np.clip(np.searchsorted(E2M1_MAG, a, side="right") - 1, 0, 7)
    hi = np.minimum(lo + 1, 7)
    dlo = a - E2M1_MAG[lo]
    dhi = E2M1_MAG[hi] - a
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (hi != lo) & ((lo & 1) == 1))
    mag = np.where(pick_hi, hi, lo)
    mag = np.where(a >= E2M1_MAX, 7, mag)
    code = mag | np.where((v < 0) & (mag != 0), 8, 0)
    return code.astype(np.uint8)


def encode_intervals(v) -> np.ndarray:
    """Second, independent encoder (used to pin ``encode``): the rounding
    intervals written out from the magnitudes and the ties-to-even rule.  A
    tie goes to the even code: 0.25 -> 0, 0.75 -> 1.0, 1.25 -> 1.0,
    1.75 -> 2.0, 2.5 -> 2.0, 3.5 -> 4.0, 5 -> 4.0."""
    a = np.abs(np.asarray(v, dtype=np.float64))
    mag = np.select(
        [a <= 0.25, a < 0.75, a <= 1.25, a < 1.75, a <= 2.5, a < 3.5, a <= 5.0],
        [0, 1, 2, 3, 4, 5, 6], default=7)
    neg = (np.asarray(v, dtype=np.float64) < 0) & (mag != 0)
    return (mag | np.where(neg, 8, 0)).astype(np.uint8)


def tensor_scale(w) -> np.float32:
    """Weight tensor scale g = amax / (6 * 448) in float32 (1 for all zeros)."""
    a = np.float32(np.abs(np.asarray(w, dtype=np.float32)).max()) if np.size(w) else np.float32(0)
    return np.float32(1.0) if a == 0 else np.float32(a / np.float32(E2M1_MAX * E4M3_MAX))


def quantize_blocks(x, g):
    """[M, K] values (K a multiple of 16) with tensor scale g -> (codes uint8
    [M, K] in 0..15, block scales as e4m3 codes uint8 [M, K/16])."""
    x = np.asarray(moe._f64(x), dtype=np.float32)
    g = np.float32(g)
    M, K = x.shape
    if K % BLOCK:
        raise ValueError("the contraction dimension must be a multiple of 16")
    blk = x.reshape(M, K // BLOCK, BLOCK)
    amax = np.abs(blk).max(axis=2) if M else np.zeros((0, K // BLOCK), np.float32)
    d = np.float32(np.float32(E2M1_MAX) * g)
    s_code = fp8.encode((amax / d).astype(np.float32))
    s = fp8.decode(s_code).astype(np.float32)
    denom = (s * g).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = (blk / denom[:, :, None]).astype(np.float32)
    q = np.where(denom[:, :, None] == 0, 0, encode(r))
    return q.reshape(M, K).astype(np.uint8), s_code


def dequantize(codes, s_codes, g) -> np.ndarray:
    """value = e2m1(code) * e4m3(scale) * g, in float64 (exact)."""
    codes = np.asarray(codes)
    s = np.repeat(fp8.decode(s_codes), BLOCK, axis=1)[:, :codes.shape[1]]
    return decode(codes) * s * np.float64(np.float32(g))


def quantize_weight(w):
    """[N, K] weights -> (codes [N, K], e4m3 block scales [N, K/16], tensor scale g)."""
    w = np.asarray(moe._f64(w), dtype=np.float32)
    g = tensor_scale(w)
    q, s = quantize_blocks(w, g)
    return q, s, g


def quantize_expert(w_gate, w_up, w_down):
    """One expert's three matrices as NVFP4: gate and up stacked into one
    [2I, H] matrix with one tensor scale, down on its own.  Returns
    ((gu codes, gu scales, g_gu), (down codes, down scales, g_down))."""
    gu = np.concatenate([np.asarray(moe._f64(w_gate), np.float32),
                         np.asarray(moe._f64(w_up), np.float32)], axis=0)
    return quantize_weight(gu), quantize_weight(w_down)


def dequantize_expert(q_gu, q_down):
    """Inverse of ``quantize_expert``: the dequantised (W_g, W_u, W_d)."""
    gu = dequantize(*q_gu)
    I = gu.shape[0] // 2
    return gu[:I], gu[I:], dequantize(*q_down)


def quantize_act(x, g):
    """Activations [M, K] -> dequantised float64 values after NVFP4 quantisation
    with the static tensor scale g (codes and scales are returned too)."""
    q, s = quantize_blocks(np.asarray(moe._f64(x), dtype=np.float32), g)
    return dequantize(q, s, g), q, s


def swiglu_ffn_nvfp4(x_deq, w_gate, w_up, w_down, g_h, quantize_h=True) -> np.ndarray:
    """One NVFP4 expert on dequantised input rows: GEMM1 and the SwiGLU in
    float64, h rounded to float32 and quantised per row with tensor scale g_h
    (the input of the second GEMM is NVFP4 too), then GEMM2.  The weights are
    already dequantised."""
    h = moe.silu(x_deq @ w_gate.T) * (x_deq @ w_up.T)
    if quantize_h:
        h = quantize_act(h.astype(np.float32), g_h)[0]
    return h @ w_down.T


def moe_layer_nvfp4(x, w_router, bias, experts, shared, k, score, renormalize=True,
                    route_scale=1.0, g_x=1.0, g_h=1.0, quantize_activations=True):
    """NVFP4 layer: routing as the bf16 layer (bf16 router, fp64 logits), each
    token quantised once with the static tensor scale g_x, expert weights
    NVFP4 (``experts(e)`` returns the three dequantised matrices), h quantised
    per row with g_h, all products in float64.  ``quantize_activations=False``
    keeps the activations unquantised (diagnostic)."""
    x64 = moe._f64(x)
    E = moe._f64(w_router).shape[0]
    lg, ids, w = moe.route(x64, w_router, bias, k, score, renormalize, route_scale)
    counts, offsets = moe.expert_histogram(ids, E)
    perm_token, perm_slot, inv_row = moe.permutation(ids, E)
    if quantize_activations:
        x_deq, xq, xs = quantize_act(x64.astype(np.float32), g_x)
    else:
        x_deq, xq, xs = x64, None, None
    x_perm = x_deq[perm_token]
    row_weight = w[perm_token, perm_slot]
    y = np.zeros(x_perm.shape, dtype=np.float64)
    for e in range(E):
        a, b = int(offsets[e]), int(offsets[e + 1])
        if b > a:
            y[a:b] = swiglu_ffn_nvfp4(x_perm[a:b], *experts(e), g_h,
                                      quantize_h=quantize_activations)
    y_perm = y * row_weight[:, None]
    s = (swiglu_ffn_nvfp4(x_deq, *shared, g_h, quantize_h=quantize_activations)
         if shared is not None else None)
    out = moe.combine(y_perm, inv_row, s)
    return dict(logits=lg, ids=ids, weights=w, counts=counts, offsets=offsets,
                perm_token=perm_token, inv_row=inv_row, x_codes=xq, x_scales=xs,
                y_perm=y_perm, shared_out=s, out=out)


def moe_tokens_nvfp4(x_rows, ids, w, experts, shared, g_x, g_h):
    """Brute-force per-token evaluation of the NVFP4 layer (no permutation):
    each token's row is quantised with g_x, run through its selected experts
    (dequantised weights from ``experts(e)``, h quantised with g_h) and the
    shared expert, and summed with its gate weights."""
    xd = quantize_act(np.asarray(moe._f64(x_rows), dtype=np.float32), g_x)[0]
    ids = np.asarray(ids)
    w = moe._f64(w)
    out = np.zeros(xd.shape, dtype=np.float64)
    cache = {}
    for t in range(xd.shape[0]):
        for j in range(ids.shape[1]):
            e = int(ids[t, j])
            if e not in cache:
                cache[e] = experts(e)
            out[t] += w[t, j] * swiglu_ffn_nvfp4(xd[t:t + 1], *cache[e], g_h)[0]
        if shared is not None:
            out[t] += swiglu_ffn_nvfp4(xd[t:t + 1], *shared, g_h)[0]
    return out


def expert_rows_nvfp4(x_rows, w_gate, w_up, w_down, g_x, g_h) -> np.ndarray:
    """One NVFP4 expert on raw input rows: each row quantised with the static
    tensor scale g_x and dequantised, then ``swiglu_ffn_nvfp4`` (h quantised
    with g_h) on the dequantised weights.  The row function
    ``moe.moe_tokens_by_expert`` takes; with it the NVFP4 layer's per-token sum
    equals ``moe_tokens_nvfp4``."""
    xd = quantize_act(np.asarray(moe._f64(x_rows), dtype=np.float32), g_x)[0]
    return swiglu_ffn_nvfp4(xd, w_gate, w_up, w_down, g_h)
