"""fp8 e4m3 codec, block quantisation and the fp8 layer (test infrastructure only).

Codec: OCP 8-bit floating point specification (OFP8), format E4M3: 1 sign,
4 exponent bits (bias 7), 3 mantissa bits, no infinities, NaN = S.1111.111,
largest finite magnitude 1.75 * 2^8 = 448, subnormals m * 2^-9.  Encoding is
round-to-nearest-even with saturation to +-448 ("satfinite").

Block quantisation (a reading: the pages use fp8 expert GEMMs -- AFD
write-up, section 1, fp8 DeepGEMM for Qwen3-235B-A22B-FP8 -- but give no
scale convention): for each 128x128 weight block, or each 1x128 group of one
token's activations, s = amax / 448 computed in float32, q = e4m3(x / s) with
the quotient computed in float32; an all-zero block gets s = 1.  The value
represented is q * s.  Parity of this convention is unpinned by the pages.
"""
from __future__ import annotations

import numpy as np

from . import moe

E4M3_MAX = 448.0
BLOCK = 128


def _magnitudes() -> np.ndarray:
    """Value of each non-negative finite code 0x00..0x7E, from the bit fields."""
    vals = np.zeros(127, dtype=np.float64)
    for c in range(127):
        e = (c >> 3) & 0xF
        m = c & 0x7
        vals[c] = m * 2.0 ** -9 if e == 0 else (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return vals


_MAG = _magnitudes()


def decode(codes) -> np.ndarray:
    """e4m3 codes (uint8) -> float64; NaN codes (0x7F, 0xFF) -> nan."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    mag = np.where((c & 0x7F) == 0x7F, np.nan, _MAG[np.minimum(c & 0x7F, 126)])
    return np.where(c & 0x80, -mag, mag)


def encode(v) -> np.ndarray:
    """float -> e4m3 code, round to nearest (ties to the even code), saturating
    finite values beyond 448 to 448; NaN -> 0x7F.  Nearest entry of the table of
    all 127 non-negative finite magnitudes."""
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    # index of the largest magnitude <= a
    lo = np.clip(np.searchsorted(_MAG, a, side="right") - 1, 0, 126)
    hi = np.minimum(lo + 1, 126)
    dlo = a - _MAG[lo]
    dhi = _MAG[hi] - a
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (hi != lo) & ((lo & 1) == 1))
    code = np.where(pick_hi, hi, lo)
    code = np.where(a >= E4M3_MAX, 126, code)
    code = code | np.where(np.signbit(v), 0x80, 0)
    code = np.where(np.isnan(v), 0x7F, code)
    return code.astype(np.uint8)


def encode_bitfield(v) -> np.ndarray:
    """Second, independent e4m3 encoder (used to pin `encode`), from the bit
    fields: below 2^-6 the value is m * 2^-9 with m = rint(|v| * 2^9) (m = 8 is
    the smallest normal, code 0x08); otherwise |v| = f * 2^e with f in [1, 2),
    the 3-bit mantissa is rint((f - 1) * 8) (round half to even), a carry to 8
    bumps the exponent, and the code is (e + 7) << 3 | mantissa."""
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    with np.errstate(invalid="ignore", over="ignore"):
        fr, ex = np.frexp(a)                     # a = fr * 2^ex, fr in [0.5, 1)
        e = ex - 1                               # a = (2 fr) * 2^e
        mant = np.rint((2.0 * fr - 1.0) * 8.0)   # round half to even
        carry = mant >= 8.0
        e = np.where(carry, e + 1, e)
        mant = np.where(carry, 0.0, mant)
        normal = np.clip(((e + 7) << 3) + mant.astype(np.int64), 0, 126)
        sub = np.rint(a * 512.0)                 # multiples of 2^-9 (8 -> 0x08)
        code = np.where(a < 2.0 ** -6, sub, normal).astype(np.int64)
    code = np.where(a >= E4M3_MAX, 126, code)
    code = code | np.where(np.signbit(v), 0x80, 0)
    code = np.where(np.isnan(v), 0x7F, code)
    return code.astype(np.uint8)


def _scale_f32(amax_f32: np.ndarray) -> np.ndarray:
    s = (amax_f32 / np.float32(E4M3_MAX)).astype(np.float32)
    return np.where(amax_f32 == 0, np.float32(1.0), s).astype(np.float32)


def quantize_weight_blocks(w):
    """[N, K] float32 weights (N, K multiples of 128) -> (codes uint8 [N, K],
    scales float32 [N/128, K/128])."""
    w = np.asarray(moe._f64(w), dtype=np.float32)
    N, K = w.shape
    if N % BLOCK or K % BLOCK:
        raise ValueError("weight dims must be multiples of 128")
    blk = w.reshape(N // BLOCK, BLOCK, K // BLOCK, BLOCK)
    amax = np.abs(blk).max(axis=(1, 3)).astype(np.float32)
    s = _scale_f32(amax)
    q = (blk / s[:, None, :, None]).astype(np.float32)     # float32 quotient
    return encode(q).reshape(N, K), s


def quantize_act_groups(x):
    """[M, K] activations (K multiple of 128) -> (codes uint8 [M, K], scales
    float32 [M, K/128]); one scale per token per 128 consecutive features."""
    x = np.asarray(moe._f64(x), dtype=np.float32)
    M, K = x.shape
    if K % BLOCK:
        raise ValueError("feature dim must be a multiple of 128")
    g = x.reshape(M, K // BLOCK, BLOCK)
    amax = np.abs(g).max(axis=2).astype(np.float32) if M else np.zeros((0, K // BLOCK), np.float32)
    s = _scale_f32(amax)
    q = (g / s[:, :, None]).astype(np.float32)
    return encode(q).reshape(M, K), s


def dequant_weight(codes, scales) -> np.ndarray:
    N, K = codes.shape
    s = np.repeat(np.repeat(np.asarray(scales, np.float64), BLOCK, 0), BLOCK, 1)
    return decode(codes) * s[:N, :K]


def dequant_act(codes, scales) -> np.ndarray:
    M, K = codes.shape
    return decode(codes) * np.repeat(np.asarray(scales, np.float64), BLOCK, 1)[:, :K]


def swiglu_ffn_fp8(x_deq, w_gate, w_up, w_down, quantize_h=True) -> np.ndarray:
    """One fp8 expert: GEMM1 on the dequantised e4m3 input, SwiGLU in float64,
    h rounded to float32 and quantised per row in 1x128 groups (the input of
    the second GEMM is e4m3 too), then GEMM2.  Weights are already dequantised."""
    h = moe.silu(x_deq @ w_gate.T) * (x_deq @ w_up.T)
    if quantize_h:
        hq, hs = quantize_act_groups(h.astype(np.float32))
        h = dequant_act(hq, hs)
    return h @ w_down.T


def moe_layer_fp8(x, w_router, bias, experts, shared, k, score, renormalize=True,
                  route_scale=1.0, quantize_activations=True):
    """fp8 layer: routing as the bf16 layer (bf16 router), expert inputs
    quantised per token in 1x128 groups, e4m3 expert weights with 128x128
    block scales (``experts(e)`` returns the three dequantised matrices),
    intermediate h quantised the same way, all products in float64.
    ``quantize_activations=False`` keeps activations unquantised (diagnostic)."""
    x64 = moe._f64(x)
    E = moe._f64(w_router).shape[0]
    lg, ids, w = moe.route(x64, w_router, bias, k, score, renormalize, route_scale)
    counts, offsets = moe.expert_histogram(ids, E)
    perm_token, perm_slot, inv_row = moe.permutation(ids, E)
    if quantize_activations:
        xq, xs = quantize_act_groups(x64.astype(np.float32))
        x_deq = dequant_act(xq, xs)
    else:
        xq = xs = None
        x_deq = x64
    x_perm = x_deq[perm_token]
    row_weight = w[perm_token, perm_slot]
    y = np.zeros(x_perm.shape, dtype=np.float64)
    for e in range(E):
        a, b = int(offsets[e]), int(offsets[e + 1])
        if b > a:
            y[a:b] = swiglu_ffn_fp8(x_perm[a:b], *experts(e), quantize_h=quantize_activations)
    y_perm = y * row_weight[:, None]
    s = swiglu_ffn_fp8(x_deq, *shared, quantize_h=quantize_activations) if shared is not None else None
    out = moe.combine(y_perm, inv_row, s)
    return dict(logits=lg, ids=ids, weights=w, counts=counts, offsets=offsets,
                perm_token=perm_token, inv_row=inv_row, x_codes=xq, x_scales=xs,
                y_perm=y_perm, shared_out=s, out=out)


def moe_tokens_fp8(x_rows, ids, w, experts, shared):
    """Brute-force per-token evaluation of the fp8 layer (no permutation): each
    token's bf16 row is quantised in 1x128 groups, run through its selected
    experts (dequantised weights from ``experts(e)``, h quantised per row) and
    the shared expert, and summed with its gate weights."""
    x = np.asarray(moe._f64(x_rows), dtype=np.float32)
    q, s = quantize_act_groups(x)
    xd = dequant_act(q, s)
    ids = np.asarray(ids)
    w = moe._f64(w)
    out = np.zeros(xd.shape, dtype=np.float64)
    cache = {}
    for t in range(xd.shape[0]):
        for j in range(ids.shape[1]):
            e = int(ids[t, j])
            if e not in cache:
                cache[e] = experts(e)
            out[t] += w[t, j] * swiglu_ffn_fp8(xd[t:t + 1], *cache[e])[0]
        if shared is not None:
            out[t] += swiglu_ffn_fp8(xd[t:t + 1], *shared)[0]
    return out


def expert_rows_fp8(x_rows, w_gate, w_up, w_down) -> np.ndarray:
    """One fp8 expert on raw (unquantised) input rows: each row quantised in
    1x128 groups and dequantised, then ``swiglu_ffn_fp8`` on the dequantised
    weights.  The row function ``moe.moe_tokens_by_expert`` takes; with it the
    fp8 layer's per-token sum equals ``moe_tokens_fp8``."""
    q, s = quantize_act_groups(np.asarray(moe._f64(x_rows), dtype=np.float32))
    return swiglu_ffn_fp8(dequant_act(q, s), w_gate, w_up, w_down)
