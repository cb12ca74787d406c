"""Seeded input generator: determinism, prefix property, value distributions (CPU only)."""
import math

import numpy as np

import moe_inputs as mi


def test_same_seed_same_bytes_and_streams_differ():
    a = mi.normal_bf16(mi.SEED, 0, (1000,), 1.0)
    b = mi.normal_bf16(mi.SEED, 0, (1000,), 1.0)
    c = mi.normal_bf16(mi.SEED + 1, 0, (1000,), 1.0)
    d = mi.normal_bf16(mi.SEED, 1, (1000,), 1.0)
    assert np.array_equal(a, b) and not np.array_equal(a, c) and not np.array_equal(a, d)
    assert np.array_equal(mi.random_bytes(5, 2, (77,)), mi.random_bytes(5, 2, (77,)))


def test_counter_based_offsets():
    full = mi.normal_f64(123, 4, 100)
    part = mi.normal_f64(123, 4, 40, first=60)
    assert np.array_equal(full[60:], part)
    by = mi.random_bytes(9, 0, (64,))
    w0 = mi._get_lib().gen_draw(9, 0, 0)
    assert list(by[:8]) == [(w0 >> (8 * i)) & 0xFF for i in range(8)]


def test_x_prefix_property():
    spec = mi.WORKLOADS["qwen35_mini_moe_decode_t64"]
    x8 = mi.make_x(spec, 8)
    x64 = mi.make_x(spec, 64)
    assert np.array_equal(x8, x64[:8])


def test_distributions():
    z = mi.normal_f64(mi.SEED, 7, 200_000)
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1.0) < 0.01
    assert abs(np.mean(z ** 4) - 3.0) < 0.1          # Gaussian kurtosis
    w = mi.bf16_to_f32(mi.normal_bf16(mi.SEED, 8, (100_000,), 1.0 / math.sqrt(2048)))
    assert abs(w.std() * math.sqrt(2048) - 1.0) < 0.02
    s = mi.int_range_u8(mi.SEED, 1, (90_000,), 118, 126)
    assert s.min() == 118 and s.max() == 126
    assert np.all(np.abs(np.bincount(s)[118:] / 10_000 - 1.0) < 0.05)
    nib = mi.random_bytes(mi.SEED, 0, (64_000,))
    lo = np.bincount(nib & 0xF, minlength=16)
    hi = np.bincount(nib >> 4, minlength=16)
    assert np.all(np.abs(lo / 4000 - 1) < 0.1) and np.all(np.abs(hi / 4000 - 1) < 0.1)


def test_bf16_rounding_is_rne():
    assert mi.f64_to_bf16(1.0) == 0x3F80
    assert mi.f64_to_bf16(1.0 + 2 ** -8) == 0x3F80            # tie -> even
    assert mi.f64_to_bf16(1.0 + 3 * 2 ** -8) == 0x3F82        # tie -> even (up)
    assert mi.f64_to_bf16(-2.5) == 0xC020
    assert np.isnan(mi.bf16_to_f32(mi.f64_to_bf16(float("nan"))))


def test_zipf_bias_is_log_rank_permutation():
    spec = mi.WORKLOADS["gptoss_20b_moe_prefill_t8192"]
    b = mi.bf16_to_f32(mi.make_router_bias(spec)).astype(np.float64)
    ranks = np.rint(np.exp(-b / 1.1)).astype(int)
    assert sorted(ranks) == list(range(1, 33))


def test_layer_shapes():
    spec = mi.small_spec("gptoss", 64, 4, 2, 96, 0, 3)
    lay = mi.make_layer(spec)
    assert lay.gu_blocks.shape == (4, 192, 2, 16) and lay.gu_scales.shape == (4, 192, 2)
    assert lay.dn_blocks.shape == (4, 64, 3, 16) and lay.dn_bias.shape == (4, 64)
    spec = mi.small_spec("qwen", 64, 4, 2, 32, 48, 3)
    lay = mi.make_layer(spec)
    assert lay.gate.shape == (4, 32, 64) and lay.down.shape == (4, 64, 32)
    assert lay.sh_gate.shape == (48, 64) and lay.sh_down.shape == (64, 48)
