"""Pins for the synthetic input recipe (CPU only): the distributions and structure the seeded
generators promise, checked against their closed forms."""
import numpy as np

import synth


def test_zipf_bias_is_the_log_of_a_zipf_pmf_over_a_permutation():
    E = 128
    b = synth.zipf_bias(E, seed=3, layer=5, alpha=1.1).astype(np.float64)
    rank = np.rint(np.exp(-b / 1.1)).astype(int)  # bias = -1.1 ln(rank)
    assert sorted(rank) == list(range(1, E + 1))  # every rank exactly once
    np.testing.assert_allclose(np.sort(np.exp(b))[::-1], 1.0 / np.arange(1, E + 1) ** 1.1, rtol=1e-6)
    assert not np.array_equal(b, synth.zipf_bias(E, seed=3, layer=6, alpha=1.1))  # re-drawn per layer


def test_logit_rows_have_distinct_values_and_zipf_skews_selection():
    T, E, k = 512, 128, 8
    lg = synth.gen_logits(T, E, seed=0, layer=0, zipf_alpha=1.1)
    assert all(len(np.unique(row)) == E for row in lg)
    top = np.argsort(-lg, axis=1)[:, :k]
    counts = np.bincount(top.ravel(), minlength=E)
    first = int(np.argmax(synth.zipf_bias(E, seed=0, layer=0)))  # the rank-1 expert
    assert counts[first] == counts.max() and counts[first] > 3 * T * k / E
    uni = np.bincount(np.argsort(-synth.gen_logits(T, E, seed=0, layer=0), axis=1)[:, :k].ravel(), minlength=E)
    assert uni.max() < counts.max()  # without the bias no expert is that hot


def test_x_is_bf16_standard_normal():
    x = synth.gen_x(256, 2048, seed=1)
    f = synth.bf16_bits_to_f32(x)
    assert np.array_equal(synth.f32_to_bf16_bits(f), x)  # exact bf16 values
    assert abs(f.mean()) < 0.01 and abs(f.std() - 1.0) < 0.01


def test_expert_weights_regenerate_per_expert():
    E, H, I = 6, 256, 128
    wgu, wd = synth.gen_expert_weights(E, H, I, seed=9)
    sgu, sd = synth.gen_expert_weights(E, H, I, seed=9, experts=[1, 4])
    for e in (1, 4):
        assert np.array_equal(sgu[e], wgu[e]) and np.array_equal(sd[e], wd[e])
    f = synth.bf16_bits_to_f32(wgu)
    assert abs(f.std() - 0.02) < 0.001


def test_mixed_stack_formats():
    c = synth.CONFIGS[5]
    f48 = synth.layer_formats(c, 48)
    assert f48 == ["fp8"] * 26 + ["nvfp4_w4a4"] * 22  # 48 * 17/32 = 25.5, rounded half up
    assert synth.layer_formats(c, 2) == ["fp8", "nvfp4_w4a4"]
    assert synth.layer_formats(synth.CONFIGS[4], 3) == ["nvfp4_w4a4"] * 3
