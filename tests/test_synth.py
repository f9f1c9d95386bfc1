"""The seeded input generator: published SplitMix64 outputs, determinism,
range splitting, bf16 rounding and the workload recipe."""
import numpy as np
import pytest

import synth
from synth import workloads as W


def test_splitmix64_published_sequence():
    # First outputs of SplitMix64 seeded with 0 (reference sequence of the
    # generator by Steele, Lea and Flood, as used to seed xoshiro generators).
    assert synth.sm64_at(0, 0) == 0xE220A8397B1DCDAF
    assert synth.sm64_at(0, 1) == 0x6E789E6AA1B965F4
    assert synth.sm64_at(0, 2) == 0x06C45D188009454F


def test_byte_stream_is_counter_based():
    seed = 0x1234
    whole = synth.random_bytes(seed, 1000)
    assert np.array_equal(whole[13:613], synth.random_bytes(seed, 600, first=13))
    v = synth.sm64_at(seed, 5)
    assert whole[40:48].tolist() == [(v >> (8 * i)) & 255 for i in range(8)]
    big = np.empty(1 << 23, np.uint8)
    synth.bytes_into(seed, big, threads=7)
    assert np.array_equal(big[:1000], whole)
    assert np.array_equal(big[-999:], synth.random_bytes(seed, 999, first=big.size - 999))


def test_normal_moments_and_determinism():
    a = synth.normal_f32(99, 200000, 0.5)
    assert abs(a.mean()) < 0.01 and abs(a.std() - 0.5) < 0.01
    assert np.array_equal(a[:11], synth.normal_f32(99, 11, 0.5))


def test_bf16_round_to_nearest_even():
    f = np.array([1.0, 1.0 + 2**-8, 1.0 + 3 * 2**-8, 1.0 + 2**-8 + 2**-20, -2.5, 0.0,
                  np.inf, 3.0e38], np.float32)
    b = synth.f32_to_bf16(f)
    assert b.tolist() == [0x3F80, 0x3F80, 0x3F82, 0x3F81, 0xC020, 0x0000, 0x7F80, 0x7F62]
    x = np.random.default_rng(1).normal(size=1000).astype(np.float32)
    back = synth.bf16_to_f32(synth.f32_to_bf16(x))
    assert (np.abs(back - x) <= np.abs(x) * 2.0**-8).all()


def test_permutation_is_a_permutation():
    p = synth.permutation(3, 256)
    assert sorted(p.tolist()) == list(range(256))
    assert not np.array_equal(p, np.arange(256))


def test_workload_recipe_shapes_and_scales():
    src = W.ExpertSource(1, 0, W.WORKLOADS[1].shape)
    cb = src.codebooks(3, W.GATE)
    assert cb.shape == (3, 256, 8) and cb.dtype == np.float32
    for s, sig in enumerate(W.STAGE_SIGMA):
        assert abs(cb[s].std() - sig) < 0.15 * sig
    c = src.codes(3, W.DOWN)
    assert c.shape == (2048, 1024 // 8, 3)
    assert abs(c.mean() - 127.5) < 1.0
    assert not np.array_equal(src.codes(3, W.GATE), src.codes(3, W.UP))
    t = src.tokens_bf16(4)
    assert t.shape == (4, 2048) and t.dtype == np.uint16
    assert np.array_equal(t[:2], src.tokens_bf16(2))
