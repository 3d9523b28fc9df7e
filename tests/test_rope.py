"""The RoPE reference pinned by closed forms and invariants, and the library's host
frequency table equal to it."""
import math

import numpy as np
import pytest

from oracle import rope


def test_base_table_closed_form():
    f = rope.yarn_freqs(128, 10000.0)
    assert f[0] == 1.0
    assert math.isclose(f[1], math.exp(-math.log(10000.0) / 64), rel_tol=1e-7)  # 0.8659643...
    assert math.isclose(f[1], 0.86596432336, rel_tol=1e-7)
    assert math.isclose(f[63], 1.1547819846894582e-4, rel_tol=1e-6)           # 10000^(-126/128)


def test_yarn_bands_and_ramp_endpoints():
    d, base, s, L, bf, bs_ = 128, 1e6, 8.0, 8192, 32.0, 1.0
    plain = rope.yarn_freqs(d, base).astype(np.float64)
    y = rope.yarn_freqs(d, base, s, L, bf, bs_).astype(np.float64)
    r = L * plain / (2 * math.pi)
    assert np.allclose(y[r > bf], plain[r > bf], rtol=0)          # fast pairs keep f
    assert np.allclose(y[r < bs_], plain[r < bs_] / s, rtol=1e-7)  # slow pairs take f / scale
    mid = (r >= bs_) & (r <= bf)
    assert mid.any()
    ratio = y[mid] / plain[mid]                                     # between 1/s and 1, falls as r falls
    assert np.all(ratio <= 1 + 1e-7) and np.all(ratio >= 1 / s - 1e-7)
    assert np.all(np.diff(ratio[np.argsort(r[mid])]) >= -1e-7)
    assert np.array_equal(rope.yarn_freqs(d, base, 1.0, L), rope.yarn_freqs(d, base))  # no scaling


def test_hand_rotation_uses_adjacent_pairs():
    x = np.array([[[1.0, 0.0, 0.0, 1.0]]])
    y = rope.apply_rope(x, [2], np.array([1.0, 0.5], dtype=np.float32), 4)
    assert np.allclose(y[0, 0], [math.cos(2), math.sin(2), -math.sin(1), math.cos(1)], atol=1e-15)
    z = np.zeros((1, 1, 8)); z[0, 0, 0] = 1.0
    w = rope.apply_rope(z, [3], rope.yarn_freqs(8, 10000.0), 8)
    assert np.count_nonzero(w[0, 0, 2:]) == 0 and w[0, 0, 4] == 0.0   # only the pair (0, 1) moves


def test_rotation_invariants():
    rng = np.random.default_rng(0)
    f = rope.yarn_freqs(64, 10000.0, 4.0, 2048)
    x = rng.standard_normal((5, 3, 64))
    pos = [0, 1, 17, 900, 70000]
    assert np.allclose(rope.apply_rope(x, [0] * 5, f, 64), x, atol=0)            # position 0
    y = rope.apply_rope(x, pos, f, 64)
    n0 = x[..., 0::2] ** 2 + x[..., 1::2] ** 2
    n1 = y[..., 0::2] ** 2 + y[..., 1::2] ** 2
    assert np.allclose(n0, n1, rtol=1e-12)                                        # pair norms
    two = rope.apply_rope(rope.apply_rope(x, [5] * 5, f, 64), [7] * 5, f, 64)
    assert np.allclose(two, rope.apply_rope(x, [12] * 5, f, 64), atol=1e-12)     # composition
    part = rope.apply_rope(x, pos, f, 32)
    assert np.array_equal(part[..., 32:], x[..., 32:])                           # rope_dim < D


def test_relative_position_property():
    """q(m) . k(n) depends on m - n only: the score RoPE is built to give."""
    rng = np.random.default_rng(1)
    f = rope.yarn_freqs(128, 1e6, 16.0, 4096)
    q, k = rng.standard_normal((1, 1, 128)), rng.standard_normal((1, 1, 128))
    for m, n in [(10, 3), (5000, 4993), (123456, 123449)]:
        a = np.dot(rope.apply_rope(q, [m], f, 128)[0, 0], rope.apply_rope(k, [n], f, 128)[0, 0])
        b = np.dot(rope.apply_rope(q, [m - n], f, 128)[0, 0], k[0, 0])
        assert math.isclose(a, b, rel_tol=1e-9, abs_tol=1e-9)


def test_query_scale_closed_form():
    s = rope.q_scale([0, 4095, 4096, 8191, 12288, 40960], 0.1, 4096)
    assert np.allclose(s, [1, 1, 1 + 0.1 * math.log(2), 1 + 0.1 * math.log(2), 1 + 0.1 * math.log(4),
                           1 + 0.1 * math.log(11)], rtol=1e-15)
    assert np.array_equal(rope.q_scale([5, 99999], 0.1, 0), [1.0, 1.0])


@pytest.mark.parametrize("args", [(128, 10000.0), (128, 1e6, 16.0, 16384, 32.0, 1.0), (64, 5e5, 4.0, 2048, 32.0, 1.0),
                                  (96, 1e4, 2.0, 1000, 16.0, 2.0)])
def test_library_table_matches_reference(pa_lib_path, args):
    import paged_kv_attention_write_gb300 as pa
    lib = pa.pa_rope_yarn_freqs(*args)
    ref = rope.yarn_freqs(*args)
    ulp = np.abs(lib.view(np.int32).astype(np.int64) - ref.view(np.int32).astype(np.int64))
    assert ulp.max() <= 1 and (ulp == 0).mean() > 0.95
