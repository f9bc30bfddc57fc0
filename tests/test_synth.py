"""The seeded input generator: C build equals its numpy restatement; workload
shapes follow the stated recipes (CPU only)."""
import numpy as np

import synth


def test_c_matches_numpy_restatement():
    for seed, stream, n in ((0, 2, 1001), (123456789, 5, 64), (2**63 + 7, 3, 4097)):
        assert np.array_equal(synth.draws(seed, stream, n), synth._np_draws(seed, stream, n))
        assert np.array_equal(synth.normal_bf16_bits(seed, stream, (n,)),
                              synth._np_normal_bf16_bits(seed, stream, n))


def test_normals_look_normal():
    z = synth.normal_f64(0, 2, 200_000)
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1) < 0.01
    b = synth.bf16_bits_to_f64(synth.normal_bf16_bits(0, 2, (200_000,)))
    assert np.abs(b - z).max() <= np.abs(z).max() * 2.0 ** -8


def test_head_scale_applies_per_head():
    shape = (7, 3, 8)
    s = np.array([0.5, 1.0, 2.0])
    a = synth.bf16_bits_to_f64(synth.normal_bf16_bits(1, 2, shape))
    b = synth.bf16_bits_to_f64(synth.normal_bf16_bits(1, 2, shape, s))
    np.testing.assert_array_equal(b[:, 0], a[:, 0] * 0.5)  # power-of-two scales are exact
    np.testing.assert_array_equal(b[:, 2], a[:, 2] * 2.0)


def test_workloads():
    t = synth.tiny()
    assert t.lengths == [29, 71, 35] and t.total == 135
    assert synth.single_1024().total == 4352
    assert synth.cfg_2048().lengths == [16896, 16448]
    for seed in range(4):
        m = synth.mixed_50k(seed)
        assert 0 < m.total <= 50_000
        for (tl, H, W) in m.specs:
            assert 32 <= tl <= 512 and (H, W) in synth.MIXED_GRIDS
        e = synth.extreme_aspect(seed)
        assert [s[1:] for s in e.specs[:3]] == [(32, 128), (128, 32), (128, 128)]
        assert all(s[1:] == (64, 64) for s in e.specs[3:]) and e.total <= 50_000
        assert all(64 <= s[0] <= 512 for s in e.specs)
