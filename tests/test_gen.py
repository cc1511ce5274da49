"""The seeded input generator: published SplitMix64 values, determinism, ranges."""

import numpy as np
import pytest

import gen


def test_splitmix64_published_sequence():
    # The first three outputs of SplitMix64 seeded with 0, as printed with the
    # generator's published reference implementation.
    out = gen.draws(0, 0, 3)
    assert [int(x) for x in out] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_counter_form_matches_sequential():
    # draws(state, start, n) must equal the sequential generator's outputs start..start+n-1
    M64 = (1 << 64) - 1

    def seq(state, n):
        out = []
        for _ in range(n):
            state = (state + gen.GAMMA) & M64
            z = state
            z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & M64
            z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & M64
            out.append(z ^ (z >> 31))
        return out

    st = gen.stream_state(7, gen.STREAM_B)
    full = seq(st, 40)
    assert [int(x) for x in gen.draws(st, 0, 40)] == full
    assert [int(x) for x in gen.draws(st, 17, 9)] == full[17:26]


def test_determinism_and_independence():
    a1 = gen.matrix(3, gen.STREAM_A, 33, 17)
    a2 = gen.matrix(3, gen.STREAM_A, 33, 17)
    b = gen.matrix(3, gen.STREAM_B, 33, 17)
    assert np.array_equal(a1, a2)
    assert not np.array_equal(a1, b)
    # row-major element order: a taller matrix extends the shorter one's draws
    a3 = gen.matrix(3, gen.STREAM_A, 34, 17)
    assert np.array_equal(a3[:33], a1)


def test_chunk_boundary_is_seamless():
    n = (1 << 22) + 5
    v = gen.matrix(1, gen.STREAM_A, 1, n)
    w = gen.matrix(1, gen.STREAM_A, 1, 10)
    assert np.array_equal(v[0, :10], w[0])
    tail = gen.draws(gen.stream_state(1, gen.STREAM_A), n - 3, 3)
    u = (tail >> np.uint64(11)).astype(np.float64) * 2.0 ** -53
    assert np.array_equal(v[0, -3:], (2 * u - 1).astype(np.float32))


def test_uniform_range_and_moments():
    x = gen.matrix(0, gen.STREAM_A, 512, 512, "uniform")
    assert x.dtype == np.float32
    assert x.min() >= -1.0 and x.max() <= 1.0
    assert abs(float(x.mean())) < 0.01
    assert abs(float(x.var()) - 1.0 / 3.0) < 0.01


def test_normal_moments():
    x = gen.matrix(2, gen.STREAM_A, 512, 512, "normal").astype(np.float64)
    assert np.isfinite(x).all()
    assert abs(x.mean()) < 0.01
    assert abs(x.var() - 1.0) < 0.01
    assert abs((x ** 4).mean() - 3.0) < 0.05   # Gaussian kurtosis


def test_integer_copy():
    A, B = gen.operands(6, 6, 9, seed=0, integer_copy=True)
    assert A.shape == (6, 9) and B.shape == (9, 6)
    for x in (A, B):
        assert np.array_equal(x, np.round(x))
        assert x.min() >= -4 and x.max() <= 4
    big = gen.matrix(0, gen.STREAM_A_INT, 100, 100, "int")
    assert set(np.unique(big).tolist()) == set(range(-4, 5))
    Au, _ = gen.operands(6, 6, 9, seed=0)
    assert not np.array_equal(A, np.round(Au))


def test_strided_buffer():
    m = gen.matrix(0, 0, 3, 5)
    s = gen.strided(m, 8)
    assert s.shape == (3, 8)
    assert np.array_equal(s[:, :5], m)
    assert np.isnan(s[:, 5:]).all()
    with pytest.raises(ValueError):
        gen.strided(m, 4)


def test_workloads_table():
    assert gen.WORKLOADS["square_8192"] == (8192, 8192, 8192, "normal", 2)
    assert gen.WORKLOADS["ragged_3001x4999x2047"][:3] == (3001, 4999, 2047)
