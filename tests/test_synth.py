"""CPU tests of the seeded input generator (no ROCmFP4 arithmetic here)."""
import numpy as np

import synth


def test_splitmix64_reference_outputs():
    # First outputs of SplitMix64 started at state 0 (the published reference
    # sequence of the generator of Steele, Lea and Flood, as produced by
    # Vigna's splitmix64.c and Java's SplittableRandom).
    z = synth.mix64(synth.GAMMA * np.arange(1, 4, dtype=np.uint64))
    assert [int(v) for v in z] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_draws_are_counter_based_and_deterministic():
    a = synth.draws(0, 3, np.arange(100))
    b = synth.draws(0, 3, np.arange(50, 100))
    assert np.array_equal(a[50:], b)
    assert not np.array_equal(a, synth.draws(0, 4, np.arange(100)))
    assert not np.array_equal(a, synth.draws(1, 3, np.arange(100)))


def test_weight_bytes_follow_the_recipe():
    for var, bb in ((synth.DUAL, 18), (synth.FAST, 17)):
        W = synth.weights(64, 1024, var, seed=0, stream=1)
        assert W.shape == (64, 32 * bb)
        blocks = W.reshape(-1, bb)
        scales = blocks[:, 16:]
        assert set(np.unique(scales >> 3)) == set(range(4, 11))
        assert set(np.unique(scales & 7)) == set(range(8))
        nib = np.concatenate([blocks[:, :16] & 15, blocks[:, :16] >> 4]).ravel()
        counts = np.bincount(nib, minlength=16)
        assert counts.min() > 0.9 * counts.mean()
        # rows can be drawn on their own
        sub = synth.weights(64, 1024, var, seed=0, stream=1, rows=np.array([5, 63, 0]))
        assert np.array_equal(sub, W[[5, 63, 0]])


def test_series_functions_match_libm():
    u = np.linspace(1e-12, 1.0, 20001)
    assert np.max(np.abs(synth._ln(u) - np.log(u))) < 1e-14
    t = np.linspace(0.0, 1.0, 20001, endpoint=False)
    s, c = synth._sincos_turn(t)
    assert np.max(np.abs(s - np.sin(2 * np.pi * t))) < 1e-14
    assert np.max(np.abs(c - np.cos(2 * np.pi * t))) < 1e-14


def test_activations_are_standard_normal_and_rounded():
    z = synth.normal_f64(0, 7, np.arange(400000))
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1) < 0.01
    kurt = ((z - z.mean()) ** 4).mean() / z.var() ** 2
    assert abs(kurt - 3) < 0.05
    x16 = synth.activations(3, 64, synth.ACT_F16, seed=0, stream=7)
    xb = synth.activations(3, 64, synth.ACT_BF16, seed=0, stream=7)
    v = synth.normal_f64(0, 7, np.arange(192)).astype(np.float32)
    assert np.array_equal(x16.ravel(), v.astype(np.float16).view(np.uint16))
    # bf16 is within half an ulp of the fp32 value
    back = synth.bits_to_float(xb.ravel(), synth.ACT_BF16)
    assert np.all(np.abs(back - v) <= np.abs(v) * 2.0 ** -8)
    rows = synth.activations(3, 64, synth.ACT_F16, seed=0, stream=7, rows=np.array([2]))
    assert np.array_equal(rows[0], x16[2])
