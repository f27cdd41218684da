"""Host-side checks of the seeded input generator (no GPU, no method arithmetic)."""
import numpy as np

import synth


def test_deterministic_and_counter_based():
    a = synth.uniform(5, 1, 1000)
    b = synth.uniform(5, 1, 1000)
    assert np.array_equal(a, b)
    # counter mode: a window equals the same slice of a longer draw
    assert np.array_equal(synth.uniform(5, 1, 100, offset=900), a[900:])
    assert not np.array_equal(synth.uniform(6, 1, 1000), a)
    assert not np.array_equal(synth.uniform(5, 2, 1000), a)
    assert ((a > 0) & (a < 1)).all()


def test_normal_statistics_and_chunking():
    n = (1 << 22) + 7                     # crosses the internal chunk boundary
    z = synth.normal(3, 1, n)
    assert abs(z.mean()) < 3e-3 and abs(z.std() - 1) < 3e-3
    assert np.array_equal(synth.normal(3, 1, 1000), z[:1000])


def test_activation_outliers():
    x = synth.activations(2, 16, 4096, outlier_p=0.005, outlier_x=50.0)
    assert x.shape == (16, 4096) and x.dtype == np.float32
    frac = (np.abs(x) > 10).mean()        # N(0,1) beyond 10 is ~0; outliers x50 mostly are
    assert 0.003 < frac < 0.006


def test_bf16_bits_roundtrip():
    x = np.array([1.0, -2.5, 3.140625], np.float32)
    b = synth.to_bf16_bits(x)
    assert np.array_equal((b.astype(np.uint32) << 16).view(np.float32), x)
