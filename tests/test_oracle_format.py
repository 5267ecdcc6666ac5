"""Pins for the oracle's packing and state decode (not gpu).

Page "EXL3 Intel Arc Quantizer", Core Implemented Architecture item 5:
MSB-first packing of the low K bits of each state, with the SWAP16 half-word
swap; item 11: the per-tile container is 16*K int16 words.  The expected words
below are worked out by hand from that description (tests/golden/pack_k2.txt
and pack_k3.txt hold them with their derivation).
"""
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line)
    return rows


def _codes_to_states(codes, K, L=16):
    """Build the circular-window states for a given code sequence."""
    T = len(codes)
    n = int(np.ceil(L / K))
    st = []
    for i in range(T):
        s = 0
        for j in range(i - n + 1, i + 1):
            s = (s << K) | int(codes[j % T])
        st.append(s & ((1 << L) - 1))
    return np.array(st, dtype=np.uint32)


@pytest.mark.parametrize("name,K", [("pack_k2.txt", 2), ("pack_k3.txt", 3)])
def test_pack_golden_words(name, K):
    rows = _read_golden(name)
    for r in rows:
        codes_s, words_s = r.split("->")
        codes = np.zeros(256, dtype=np.uint32)
        for item in codes_s.split():
            pos, val = item.split("=")
            codes[int(pos)] = int(val)
        want = np.zeros(16 * K, dtype=np.uint16)
        for item in words_s.split():
            idx, val = item.split("=")
            want[int(idx)] = int(val, 16)
        assert np.array_equal(oracle.pack(codes, K), want), r


@pytest.mark.parametrize("K", [1, 2, 3, 4])
def test_pack_unpack_roundtrip_all_states(K):
    rng = np.random.default_rng(K)
    for _ in range(20):
        codes = rng.integers(0, 1 << K, 256).astype(np.uint32)
        st = _codes_to_states(codes, K)
        words = oracle.pack(st, K)
        assert words.size == 16 * K
        assert np.array_equal(oracle.unpack_states(words, K), st)


@pytest.mark.parametrize("K", [1, 2, 3, 4])
def test_known_states_decode(K):
    """A stream whose first n = ceil(16/K) codes spell s decodes to state s at
    position n-1 (all 65536 states for K=2, a random sample otherwise)."""
    n = int(np.ceil(16 / K))
    rng = np.random.default_rng(K)
    base = rng.integers(0, 1 << K, 256).astype(np.uint32)
    states = np.arange(65536) if K == 2 else np.concatenate(
        [[0, 1, 65535, 32768], rng.integers(0, 65536, 3000)])
    for s in states:
        codes = base.copy()
        v = int(s)
        for j in range(n - 1, -1, -1):
            codes[j] = v & ((1 << K) - 1)
            v >>= K
        # pack reads only the low K bits of each entry, so codes can be passed directly
        assert oracle.unpack_states(oracle.pack(codes, K), K)[n - 1] == s


def test_all_zero_and_single_code_windows():
    for K in (1, 2, 3, 4):
        z = oracle.pack(np.zeros(256, np.uint32), K)
        assert not z.any()
        assert not oracle.unpack_states(z, K).any()
        n = int(np.ceil(16 / K))
        for i in (0, 5, 100, 255):
            codes = np.zeros(256, np.uint32)
            codes[i] = (1 << K) - 1
            st = oracle.unpack_states(oracle.pack(_codes_to_states(codes, K), K), K)
            nz = set(np.nonzero(st)[0].tolist())
            assert nz == {(i + j) % 256 for j in range(n)}


@pytest.mark.parametrize("K", [2, 3, 4])
def test_one_bit_flip_changes_exactly_the_covering_windows(K):
    rng = np.random.default_rng(7)
    codes = rng.integers(0, 1 << K, 256).astype(np.uint32)
    st = _codes_to_states(codes, K)
    words = oracle.pack(st, K)
    # undo SWAP16 to find the stream position of each word bit
    for trial in range(40):
        w = int(rng.integers(0, words.size))
        b = int(rng.integers(0, 16))
        flipped = words.copy()
        flipped[w] ^= np.uint16(1 << b)
        stream_word = w ^ 1            # SWAP16 pairs words (2m, 2m+1)
        pos = stream_word * 16 + (15 - b)
        got = oracle.unpack_states(flipped, K)
        changed = set(np.nonzero(got != st)[0].tolist())
        n_bits = 256 * K
        want = {i for i in range(256)
                if ((pos - ((i + 1) * K - 16)) % n_bits) < 16}
        assert changed == want
