"""Full-size invariants of the oracle's tile encoder (L=16, T=256; not gpu).

Page "EXL3 Intel Arc Quantizer", Core Implemented Architecture items 1, 4, 5;
the test list on that page names the checks mirrored here: shift-register
identity, circular ring topology, container round trips, path-cost tracking and
bounded distortion.  The distortion floor is the Gaussian distortion-rate bound
D(R) = sigma^2 2^(-2R) at R = K bits per sample.
"""
import numpy as np
import pytest

import oracle


@pytest.fixture(scope="module")
def gaussian_tiles():
    rng = np.random.default_rng(2024)
    return rng.standard_normal((64, 16, 16)).astype(np.float32).reshape(64 * 16, 16)


@pytest.fixture(scope="module")
def encoded(gaussian_tiles):
    Y = gaussian_tiles.reshape(64, 256)
    # lay the 64 tiles side by side as a 16 x 1024 matrix (tile t at column 16t)
    M = np.concatenate([Y[t].reshape(16, 16) for t in range(64)], axis=1)
    out = {}
    for K in (1, 2, 3, 4):
        out[K] = oracle.encode_matrix(M, K, 1.0)
    return Y, out


@pytest.mark.parametrize("K", [1, 2, 3, 4])
def test_ring_shift_and_cost_invariants(encoded, K):
    Y, res = encoded
    states, costs = res[K]
    cb = oracle.mul1_table()
    low = (1 << (16 - K)) - 1
    for t in range(Y.shape[0]):
        st = states[t].astype(np.int64)
        # consecutive states share 16-K bits (shift register)
        assert np.all((st[1:] >> K) == (st[:-1] & low))
        # ring: first state's predecessor is the last state
        assert (st[0] >> K) == (st[-1] & low)
        # decode of the packed container reproduces every state
        words = oracle.pack(states[t], K)
        assert words.size == 16 * K
        assert np.array_equal(oracle.unpack_states(words, K), states[t])
        # reported cost = left-to-right fp32 sum of the branch metrics
        c = np.float32(0.0)
        for i in range(256):
            d = np.float32(Y[t, i] - cb[st[i]])
            c = np.float32(c + np.float32(d * d))
        assert c == np.float32(costs[t])


def test_distortion_nonincreasing_in_K_and_above_shannon(encoded):
    Y, res = encoded
    mses = {K: float(res[K][1].astype(np.float64).sum() / Y.size) for K in res}
    for K in (1, 2, 3):
        assert mses[K + 1] <= mses[K]
    var = float(Y.astype(np.float64).var())
    for K, m in mses.items():
        assert m >= var * 2.0 ** (-2 * K) * 0.95   # sample variance slack
        assert m <= var * 2.0 ** (-2 * K) * 2.0    # within 3 dB of the bound


def test_encode_tile_is_deterministic(gaussian_tiles):
    y = gaussian_tiles.reshape(64, 256)[0]
    a = oracle.encode_tile(y, 2)
    b = oracle.encode_tile(y, 2)
    assert np.array_equal(a[0], b[0]) and a[1] == b[1] and a[2] == b[2]
