"""The seeded input generator: determinism, ranges and distribution moments."""
import numpy as np

from dense_fp32_matrix_strict_gb300 import inputs


def test_splitmix64_reference_values():
    # splitmix64 seeded with 0: the first outputs published with the algorithm
    # (Steele, Lea, Flood 2014; also java.util.SplittableRandom's mixer).
    key = np.uint64(0)
    e = np.arange(1, 4, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = inputs._mix(key + e * inputs.GAMMA)
    assert [int(v) for v in z] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_deterministic_and_offset_consistent():
    a = inputs.raw(7, 1, 1000)
    b = inputs.raw(7, 1, 600, offset=400)
    assert np.array_equal(a[400:], b[:600])
    assert not np.array_equal(inputs.raw(7, 2, 10), inputs.raw(7, 1, 10))
    assert not np.array_equal(inputs.raw(8, 1, 10), inputs.raw(7, 1, 10))


def test_chunking_does_not_change_values():
    x = inputs.fill("normal", 3, 0, 37, 51)
    y = inputs.fill("normal", 3, 0, 37, 51, chunk=100)
    assert np.array_equal(x, y)
    u = inputs.fill("uniform", 3, 0, 37, 51)
    v = inputs.fill("uniform", 3, 0, 37, 51, chunk=64)
    assert np.array_equal(u, v)


def test_uniform_range_and_moments():
    x = inputs.fill("uniform", 0, 0, 512, 512).astype(np.float64)
    assert x.min() >= -1.0 and x.max() <= 1.0 - 2.0 ** -23
    assert np.all(x * 2 ** 23 == np.round(x * 2 ** 23))
    assert abs(x.mean()) < 0.01 and abs(x.var() - 1 / 3) < 0.01


def test_int_values():
    x = inputs.fill("int", 1, 0, 256, 256)
    vals, counts = np.unique(x, return_counts=True)
    assert list(vals) == list(range(-4, 5))
    assert counts.min() > 0.9 * x.size / 9


def test_normal_moments():
    x = inputs.fill("normal", 2, 1, 512, 512, sigma=0.02).astype(np.float64)
    assert abs(x.mean()) < 1e-3 and abs(x.std() - 0.02) < 5e-4
    assert np.all(np.isfinite(x))


def test_sample_entries_cover_edges():
    r, c = inputs.sample_entries(4093, 5120, n=1000)
    assert r.min() >= 0 and r.max() == 4092 and c.min() >= 0 and c.max() == 5119
    lin = r * 5120 + c
    assert np.all(np.diff(lin) > 0)
    assert np.count_nonzero(r == 4092) == 5120 and np.count_nonzero(c == 5119) >= 4093
    for (i, j) in [(0, 0), (0, 5119), (4092, 0), (4092, 5119)]:
        assert np.any((r == i) & (c == j))


def test_workloads_match_named_shapes():
    w = inputs.WORKLOADS
    assert (w["sq4096_uniform"].M, w["sq4096_uniform"].K) == (4096, 4096)
    rg = w["ragged_4093x5120x1531_normal"]
    assert (rg.M, rg.N, rg.K, rg.alpha, rg.beta) == (4093, 5120, 1531, 0.7, -1.3)
    llm = w["llm_8192x14336x4096"]
    assert (llm.M, llm.N, llm.K, llm.sigma_b, llm.dist_c) == (8192, 14336, 4096, 0.02, "zeros")
    assert w["sq1024_int"].exact and (w["sq1024_int"].alpha, w["sq1024_int"].beta) == (2.0, -1.0)
