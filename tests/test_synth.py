"""The seeded input generator: compiled host version against its numpy
restatement, and the distribution it is meant to have (CPU only)."""
import numpy as np

import synth


def test_host_generator_matches_numpy_restatement():
    for seed, stream, start in ((1, 1001, 0), (4, 2003, 123456789), (2, 1, 7)):
        assert np.array_equal(synth.normal_f32(seed, stream, start, 4096),
                              synth.normal_ref(seed, stream, start, 4096))


def test_normal_moments_and_support():
    z = synth.normal_f32(9, 9, 0, 1 << 20)
    assert abs(z.mean()) < 5e-3 and abs(z.std() - 1.0) < 5e-3
    assert z.min() > -6 and z.max() < 6
    # every value is an exact multiple of 2^-20
    assert np.all(np.round(z.astype(np.float64) * 2 ** 20) == z.astype(np.float64) * 2 ** 20)


def test_bf16_weights_are_rounded_scaled_normals():
    z = synth.normal_f32(1, 1001, 0, 10000)
    b = synth.normal_bf16(1, 1001, 0, 10000, 0.02)
    assert np.array_equal(b, synth.f32_to_bf16_bits(z * np.float32(0.02)))


def test_positions_nested_and_in_range():
    w = synth.SEVEN_B
    p128 = synth.positions(w, 128)
    assert np.array_equal(synth.positions(w, 80), p128[:80])
    assert p128.min() >= w.pos_lo and p128.max() < w.pos_hi


def test_kv_slab_prefix_independent_of_batch():
    w = synth.TINY
    a = synth.kv_raw_host(w, 1, 0, 0, 4, 10)
    b = synth.kv_raw_host(w, 1, 0, 2, 1, 10)
    assert np.array_equal(a[2], b[0])
    assert np.all(a[:, :, 10:] == 0)
