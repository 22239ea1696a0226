"""Seeded input recipe: determinism, slice independence, distribution, shapes."""
import math

import numpy as np
import pytest
import torch

import workload as wl
from workload import rng


def test_splitmix64_reference_values():
    # SplitMix64 seeded with 0 (state advances by the golden gamma); first outputs of the
    # published generator.
    z = rng._mix(torch.tensor([rng._s64(rng.GOLDEN * i) for i in (1, 2, 3)], dtype=torch.int64))
    got = [v & rng._MASK64 for v in z.tolist()]
    assert got == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_slices_regenerate_independently():
    full = rng.normal_bf16(0, rng.stream_id("x"), (50, 64), 1.0)
    part = rng.normal_bf16(0, rng.stream_id("x"), (7, 64), 1.0, row_start=20)
    assert torch.equal(full[20:27], part)


def test_streams_and_seeds_differ():
    a = rng.normal_f32(0, rng.stream_id("w_gate", 0), (4, 32), 1.0)
    b = rng.normal_f32(0, rng.stream_id("w_gate", 1), (4, 32), 1.0)
    c = rng.normal_f32(1, rng.stream_id("w_gate", 0), (4, 32), 1.0)
    assert not torch.equal(a, b) and not torch.equal(a, c)


def test_normal_moments():
    v = rng.normal_f32(0, 99, (1 << 20,), 0.02).double()
    assert abs(v.mean().item()) < 1e-4
    assert v.std().item() == pytest.approx(0.02, rel=5e-3)
    k4 = ((v - v.mean()) ** 4).mean() / v.var() ** 2 - 3
    assert k4.item() == pytest.approx(-0.15, abs=0.02)          # Irwin-Hall(8)
    assert v.abs().max().item() < 0.02 * 4.9


def test_skewed_lengths():
    L = wl.skewed_lengths(0)
    assert len(L) == 4 and all(6554 <= l <= 8192 for l in L)
    assert wl.DSV3_SKEW.T == sum(L)


def test_zipf_bias_shape():
    b = wl.gen_bias(wl.DSV3_SKEW)
    assert b.shape == (256,) and b.dtype == torch.float32
    assert (b == -30.0).sum().item() == 4 and (b == 0).sum().item() == 1
    assert wl.gen_bias(wl.DSV3) is None


def test_config_flops():
    # 6 T k H I + 6 T H Is + 2 T H E at the DeepSeek-V3 shape: 13.05 TFLOP
    assert wl.DSV3.flops() / 1e12 == pytest.approx(13.05, abs=0.01)
    assert wl.QWEN3.flops() / 1e12 == pytest.approx(2.48, abs=0.01)
