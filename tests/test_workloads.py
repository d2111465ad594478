"""The C input generator against a pure-Python restatement of its definition."""
import math

import numpy as np

import workloads as W

M64 = (1 << 64) - 1


def mix(z):
    z ^= z >> 30
    z = (z * 0xBF58476D1CE4E5B9) & M64
    z ^= z >> 27
    z = (z * 0x94D049BB133111EB) & M64
    z ^= z >> 31
    return z


def key(seed, tid):
    return mix(mix(seed) ^ ((tid * 0xD1B54A32D192ED03) & M64))


def draw(k, i):
    return mix((k + (i + 1) * 0x9E3779B97F4A7C15) & M64)


def unif(k, i):
    return ((draw(k, i) >> 11) + 0.5) * 2.0 ** -53


def normal(k, i):
    p = i // 2
    r = math.sqrt(-2.0 * math.log(unif(k, 2 * p)))
    th = 2 * math.pi * unif(k, 2 * p + 1)
    return r * (math.sin(th) if i & 1 else math.cos(th))


def test_draws_match_definition():
    k = key(7, 3)
    got = W.draws(7, 3, 100, 50)
    assert [int(x) for x in got] == [draw(k, i) for i in range(100, 150)]


def test_normal_fill_matches_definition():
    got = W.fill(5, 2, 10, (3, 5), (2, 9))
    k = key(5, 2)
    exp = np.array([[normal(k, r * 10 + c) for c in range(2, 9)] for r in range(3, 5)])
    np.testing.assert_allclose(got, exp, rtol=1e-14)


def test_sub_blocks_are_consistent():
    full = W.fill(9, 1, 64, (0, 20), (0, 64), dtype=W.DT_BF16)
    part = W.fill(9, 1, 64, (5, 9), (16, 40), dtype=W.DT_BF16)
    np.testing.assert_array_equal(full[5:9, 16:40], part)


def test_distributions():
    w = W.tiny()
    x = W.as_f64(w.x(), "f32")
    assert abs(x.mean()) < 0.02 and abs(x.std() - 1) < 0.02
    q = w.q().astype(np.float64).reshape(w.T, w.Hk, w.dk)
    np.testing.assert_allclose(np.linalg.norm(q, axis=-1), 1.0, rtol=1e-6)
    b = w.beta()
    assert b.min() > 0 and b.max() < 1
    assert (w.g() < 0).all()
    p = W.packed_varlen()
    assert sum(p.lengths) == 32768 and all(1 <= n <= 8192 for n in p.lengths)
    assert all(512 <= n for n in p.lengths[:-1])
    r = W.ragged()
    assert sum(r.lengths) == 65536 and max(r.lengths) <= 4096
    assert 200 < np.mean(r.lengths) < 400
