"""Seeded synthetic inputs and layer configurations shared by the tests, the
benchmark and the oracle's harness.  Holds none of the layer's arithmetic."""
from . import rng
from .configs import (CONFIGS, DECODE_T, DSV3, DSV3_DECODE, DSV3_FP8, DSV3_FP8_DECODE, DSV3_NVFP4,
                      DSV3_SKEW, DSV3_T512, QWEN3, TINY, LayerConfig, gen_bias, gen_expert, gen_router, gen_shared, gen_x,
                      nvfp4_act_scales, skewed_lengths)

__all__ = ["rng", "CONFIGS", "TINY", "QWEN3", "DSV3", "DSV3_SKEW", "DSV3_FP8", "DSV3_T512",
           "DSV3_NVFP4", "DECODE_T", "DSV3_DECODE", "DSV3_FP8_DECODE", "LayerConfig", "nvfp4_act_scales",
           "gen_x", "gen_router", "gen_expert", "gen_shared", "gen_bias", "skewed_lengths"]
