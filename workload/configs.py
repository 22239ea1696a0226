"""The five MoE-layer workloads and the seeded recipe for their inputs.

Shapes follow the pages' models: a tiny layer, a Qwen3-235B-A22B-shaped
layer (E=128, top-8), a DeepSeek-V3-shaped layer (H=7168, 256 routed experts
+ 1 shared, top-8; ASAP, section 5.1 "MoE Model"), the same layer on a skewed
batch of four concatenated sequences of 0.8x8K..8K tokens (DWDP, section
4.1, table 1 workload), the DeepSeek-V3 shape at T=512 with fp8 e4m3
expert weights (AFD write-up, section 1: fp8 expert GEMMs), and the
DeepSeek-V3 layer with NVFP4 expert weights (DWDP write-up, section A4: the
DeepSeek-R1 NVFP4 checkpoint).

Input recipe (all seeded, counter-based, see workload.rng):
  x        [T,H]  ~N(0, 1)     rounded to bf16
  w_router [E,H]  ~N(0, 0.02)  bf16
  w_gate/w_up [I,H], w_down [H,I] per expert, ~N(0, 0.02) (bf16, or fp32 before
  fp8 block quantisation; bf16 before NVFP4 quantisation); shared-expert
  matrices likewise.
  NVFP4 static activation scales (what a checkpoint would carry): g_x =
  2^-8 * x_std, so a block amax up to 10.5 x_std keeps an unsaturated e4m3
  scale; g_h = 2^-4, room for |h| up to 168 (h = silu(g) u with g, u ~ N(0,
  (0.02^2) H), std 1.7 at H = 7168).
  Skewed batch: per-expert logit bias b_e = -gamma * 1.2 * ln(r_e) with r a
  seeded permutation of 1..E (Zipf, s = 1.2), and the four coldest ranks
  pushed to -30 so that they receive no tokens.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

import torch

from . import rng


@dataclass(frozen=True)
class LayerConfig:
    name: str
    T: int
    H: int
    E: int
    k: int
    I: int
    I_shared: int = 0
    score: str = "softmax"          # "softmax" | "sigmoid"
    renormalize: bool = True
    route_scale: float = 1.0
    wtype: str = "bf16"             # "bf16" | "fp8_e4m3" | "nvfp4"
    zipf_bias: bool = False
    x_std: float = 1.0
    w_std: float = 0.02
    seed: int = 0

    @property
    def R(self) -> int:
        """Routed rows, T*k."""
        return self.T * self.k

    def flops(self) -> float:
        """Algorithmic FLOP of one layer pass: routed 6RHI + shared 6TH*Is + router 2THE."""
        return (6.0 * self.T * self.k * self.H * self.I
                + 6.0 * self.T * self.H * self.I_shared
                + 2.0 * self.T * self.H * self.E)

    def with_(self, **kw) -> "LayerConfig":
        return replace(self, **kw)


# Skewed-batch sequence lengths: four sequences, each uniform in [0.8*8192, 8192].
def skewed_lengths(seed: int = 0) -> list[int]:
    u = rng.uniform01_f64(seed, rng.stream_id("seq_len"), 4)
    return [6554 + int(math.floor(v * 1639)) for v in u]


# Zipf-bias strength for E=256, H=7168, x~N(0,1), W_r~N(0,0.02): chosen so the
# hottest expert gets ~10x the mean row count (oracle/calibrate_zipf_bias.py).
ZIPF_GAMMA = 0.4514
ZIPF_S = 1.2
ZIPF_DEAD = 4          # coldest ranks forced to receive no tokens
ZIPF_DEAD_BIAS = -30.0


TINY = LayerConfig("tiny", T=256, H=512, E=8, k=2, I=1024)
QWEN3 = LayerConfig("qwen3_235b", T=8192, H=4096, E=128, k=8, I=1536)
DSV3 = LayerConfig("dsv3", T=16384, H=7168, E=256, k=8, I=2048, I_shared=2048,
                   score="sigmoid", route_scale=2.5)
DSV3_SKEW = DSV3.with_(name="dsv3_skewed", T=sum(skewed_lengths(0)), zipf_bias=True)
DSV3_FP8 = DSV3.with_(name="dsv3_fp8", T=512, wtype="fp8_e4m3")

# DeepSeek-V3 layer in bf16 at a small batch (16 rows per expert): the
# memory-bound regime of the grouped GEMMs, a parity and bench case.
DSV3_T512 = DSV3.with_(name="dsv3_bf16_t512", T=512)

# Profiling slice: DeepSeek-V3 expert shapes and rows per expert (T*k/E = 512), a
# quarter of the experts and tokens, so that one ncu capture holds a few GB.
DSV3_SLICE = DSV3.with_(name="dsv3_slice", T=4096, E=64)
# fp8 profiling slice: 16 tokens per expert as in the 512-token fp8 batch, 1/4 of the experts
DSV3_FP8_SLICE = DSV3_FP8.with_(name="dsv3_fp8_slice", T=128, E=64)

# DeepSeek-V3 layer with NVFP4 expert weights and activations, the prefill
# batch of the bf16 layer; its profiling slice like dsv3_slice.
DSV3_NVFP4 = DSV3.with_(name="dsv3_nvfp4", wtype="nvfp4")
DSV3_NVFP4_SLICE = DSV3_NVFP4.with_(name="dsv3_nvfp4_slice", T=4096, E=64)
# the NVFP4 layer at the small batch of the fp8 layer (16 rows per expert): weight streaming
DSV3_NVFP4_T512 = DSV3_NVFP4.with_(name="dsv3_nvfp4_t512", T=512)

# The DeepSeek-V3 layer at decode-sized batches (the AFD write-up, section 1,
# reads MoE utilisation at batches from 395 down to 6 tokens): T*k rows over
# 256 experts, so most experts receive no token and the layer streams the
# weights of those that do.
DECODE_T = (8, 64, 128, 395)
DSV3_DECODE = tuple(DSV3.with_(name=f"dsv3_bf16_t{t}", T=t) for t in DECODE_T)
DSV3_FP8_DECODE = tuple(DSV3_FP8.with_(name=f"dsv3_fp8_t{t}", T=t) for t in DECODE_T)

CONFIGS = {c.name: c for c in (TINY, QWEN3, DSV3, DSV3_SKEW, DSV3_FP8, DSV3_T512, DSV3_SLICE,
                                DSV3_FP8_SLICE, DSV3_NVFP4, DSV3_NVFP4_SLICE, DSV3_NVFP4_T512,
                                *DSV3_DECODE, *DSV3_FP8_DECODE)}


def nvfp4_act_scales(cfg: LayerConfig) -> tuple[float, float]:
    """Static NVFP4 tensor scales (g_x, g_h) of the synthetic checkpoint."""
    return 2.0 ** -8 * cfg.x_std, 2.0 ** -4


# ---------------------------------------------------------------- tensors
def gen_x(cfg: LayerConfig, device="cpu", row_start: int = 0, rows: int | None = None):
    rows = cfg.T - row_start if rows is None else rows
    return rng.normal_bf16(cfg.seed, rng.stream_id("x"), (rows, cfg.H), cfg.x_std,
                           device, row_start)


def gen_router(cfg: LayerConfig, device="cpu"):
    return rng.normal_bf16(cfg.seed, rng.stream_id("w_router"), (cfg.E, cfg.H), cfg.w_std, device)


def _wshape(cfg: LayerConfig, which: str, inter: int):
    return (inter, cfg.H) if which in ("gate", "up") else (cfg.H, inter)


def _rows(shape, row_start: int, rows: int | None):
    n = shape[0] - row_start if rows is None else rows
    return (n,) + tuple(shape[1:])


def gen_expert(cfg: LayerConfig, e: int, which: str, device="cpu", row_start: int = 0,
               rows: int | None = None):
    """Routed expert e's W_gate / W_up ([I,H]) or W_down ([H,I]): bf16, or float32
    (before block quantisation) for fp8 layers.  ``row_start`` / ``rows`` give a
    slice of rows, equal to the same rows of the whole matrix."""
    shape = _rows(_wshape(cfg, which, cfg.I), row_start, rows)
    f = rng.normal_f32 if cfg.wtype == "fp8_e4m3" else rng.normal_bf16
    return f(cfg.seed, rng.stream_id("w_" + which, e), shape, cfg.w_std, device, row_start)


def gen_shared(cfg: LayerConfig, which: str, device="cpu", row_start: int = 0,
               rows: int | None = None):
    shape = _rows(_wshape(cfg, which, cfg.I_shared), row_start, rows)
    f = rng.normal_f32 if cfg.wtype == "fp8_e4m3" else rng.normal_bf16
    return f(cfg.seed, rng.stream_id("ws_" + which), shape, cfg.w_std, device, row_start)


def gen_bias(cfg: LayerConfig, gamma: float | None = None):
    """float32 [E] Zipf logit bias of the skewed batch, or None."""
    if not cfg.zipf_bias:
        return None
    g = ZIPF_GAMMA if gamma is None else gamma
    perm = rng.permutation(cfg.seed, rng.stream_id("zipf_rank"), cfg.E)
    b = torch.empty(cfg.E, dtype=torch.float64)
    for rank0, e in enumerate(perm):                 # expert perm[0] is the hottest
        r = rank0 + 1
        b[e] = ZIPF_DEAD_BIAS if r > cfg.E - ZIPF_DEAD else -g * ZIPF_S * math.log(r)
    return b.to(torch.float32)
