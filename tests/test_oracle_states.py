"""Pins for trellis state extraction and tile layout (TensorFold #837, "What
this changes": the trellis decode of 16x16 K-bit tiles).  The window reading is
checked against the shift-register recurrence that defines a bitshift trellis,
against hand-built single-bit tiles and against plain string slicing."""

import numpy as np
import pytest

from oracle import exl3_oracle as O

KS = list(range(1, 9))


def _random_tile(K, seed):
    return np.random.default_rng([seed, K]).integers(0, 1 << 32, size=8 * K, dtype=np.uint64).astype(np.uint32)


@pytest.mark.parametrize("K", KS)
def test_zero_and_one_tiles(K):
    assert np.all(O.tile_states(np.zeros(8 * K, np.uint32), K) == 0)
    assert np.all(O.tile_states(np.full(8 * K, 0xFFFFFFFF, np.uint32), K) == 0xFFFF)


@pytest.mark.parametrize("K", KS)
def test_single_bit_reaches_exactly_the_covering_states(K):
    nbits = 256 * K
    rng = np.random.default_rng(K)
    for b in list(rng.integers(0, nbits, size=12)) + [0, nbits - 1]:
        w = np.zeros(8 * K, np.uint32)
        w[b // 32] = np.uint32(1 << (31 - b % 32))
        s = O.tile_states(w, K)
        for p in range(256):
            start = (p + 1) * K - 16
            i = (b - start) % nbits            # offset of bit b inside the window
            expect = (1 << (15 - i)) if i < 16 else 0
            assert s[p] == expect, (K, b, p)
        # the bit is seen by ceil or floor of 16/K states
        assert np.count_nonzero(s) in (16 // K, -(-16 // K))


@pytest.mark.parametrize("K", KS)
def test_window_equals_shift_register(K):
    """s_p = ((s_{p-1} << K) | c_p) mod 2^16 with c_p the K bits [pK, pK+K)."""
    w = _random_tile(K, 1)
    bits = O.tile_bits(w, K).astype(np.int64)
    chunk = [int("".join(str(x) for x in bits[p * K:(p + 1) * K]), 2) for p in range(256)]
    s = O.tile_states(w, K)
    for p in range(256):
        assert s[p] == (((int(s[p - 1]) << K) | chunk[p]) & 0xFFFF)


@pytest.mark.parametrize("K", KS)
def test_string_slicing_brute_force(K):
    w = _random_tile(K, 2)
    bitstr = "".join(format(int(x), "032b") for x in w)
    n = len(bitstr)
    s = O.tile_states(w, K)
    lib = O.c_oracle()
    cs = np.zeros(256, np.uint32)
    lib.oracle_tile_states(np.ascontiguousarray(w).ctypes.data, K, cs.ctypes.data)
    for p in range(256):
        start = (p + 1) * K - 16
        window = "".join(bitstr[(start + i) % n] for i in range(16))
        assert s[p] == int(window, 2) == cs[p]


@pytest.mark.parametrize("K", [1, 3, 4, 8])
def test_tile_layout_and_tile_order(K):
    """A bit set in tile (tk, tn) changes exactly W[16tk + p%16, 16tn + p//16] for
    the positions p whose state covers it."""
    in_f, out_f = 48, 64
    T = np.zeros((in_f // 16, out_f // 16, 8 * K), np.uint32)
    tk, tn, b = 2, 1, 37 * K + 3
    T[tk, tn, b // 32] = np.uint32(1 << (31 - b % 32))
    base = O.codebook_values(np.array([0]), O.MCG)[0]
    for impl in ("numpy", "c"):
        W = O.decode_projection(T, K, O.MCG, impl)
        changed = set(zip(*np.nonzero(W != base)))
        expect = set()
        for p in range(256):
            i = (b - ((p + 1) * K - 16)) % (256 * K)
            if i < 16:
                expect.add((16 * tk + p % 16, 16 * tn + p // 16))
        assert changed == expect


@pytest.mark.parametrize("K", KS)
@pytest.mark.parametrize("cb", [O.MUL1, O.MCG, O.INST3])
def test_numpy_and_c_decoders_agree(K, cb):
    T = np.random.default_rng([7, K, cb]).integers(0, 1 << 32, size=(3, 2, 8 * K),
                                                   dtype=np.uint64).astype(np.uint32)
    a = O.decode_projection(T, K, cb, "numpy")
    c = O.decode_projection(T, K, cb, "c")
    assert a.shape == (48, 32)
    assert np.array_equal(a, c)
