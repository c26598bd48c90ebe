"""The library's host checksum of a result tile, against numpy (no GPU).

bits_sum is the sum of the float32 bit patterns read as unsigned 32-bit
integers, modulo 2**64 (numpy's uint64 sum wraps the same way); value_sum is
the double sum of the values.
"""
import numpy as np
import pytest


@pytest.fixture(scope="module")
def sec():
    import sparse_embedding_exact_gb300 as sec
    from sparse_embedding_exact_gb300 import build

    build.build()
    return sec


def _numpy_sums(t):
    bits = int(np.ascontiguousarray(t).view(np.uint32).astype(np.uint64).sum(dtype=np.uint64))
    return bits, float(t.astype(np.float64).sum())


@pytest.mark.parametrize("shape,window", [((7, 33), None), ((300, 5000), (17, 4001)), ((1, 1), None),
                                          ((2049, 513), (0, 512))])
def test_host_checksum_matches_numpy(sec, shape, window):
    rng = np.random.default_rng(5)
    big = rng.standard_normal(shape).astype(np.float32)
    big[0, 0] = -0.0  # sign bit set: the unsigned reading matters
    t = big if window is None else big[:, window[0]:window[1]]  # rows stay contiguous, ld > cols
    bits, value = sec.tile_checksum_host(t)
    nb, nv = _numpy_sums(t)
    assert bits == nb
    assert abs(value - nv) <= 1e-9 * max(1.0, abs(nv)) + 1e-6


def test_host_checksum_sees_one_flipped_bit(sec):
    rng = np.random.default_rng(6)
    t = rng.standard_normal((64, 256)).astype(np.float32)
    a, _ = sec.tile_checksum_host(t)
    u = t.view(np.uint32)
    u[40, 200] ^= 1 << 7
    b, _ = sec.tile_checksum_host(t)
    assert a != b


def test_host_checksum_empty_and_bad_arguments(sec):
    assert sec.tile_checksum_host(np.zeros((0, 8), np.float32)) == (0, 0.0)
    with pytest.raises(AssertionError):
        sec.tile_checksum_host(np.zeros((4, 4), np.float64))
