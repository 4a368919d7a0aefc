"""Pins for the oracle's codebooks (TensorFold #837, "What this changes":
mul1 / mcg / 3inst).  Closed forms worked by hand, IEEE-field arithmetic that
does not go through numpy's float16, and whole-state-space invariants."""

import math

import numpy as np
import pytest

from oracle import exl3_oracle as O

ALL = np.arange(65536, dtype=np.int64)


def test_closed_forms_by_hand():
    # mcg, s = 0: x = 0 -> x' = 0x3B603B60; 0x3B60 = +2^(14-15) * (1 + 864/1024)
    assert O.codebook_values(np.array([0]), O.MCG)[0] == 2 * 0.921875
    # mcg, s = 1: x = 0xCBAC1FED -> x' = 0xB0CC348D
    #   0x348D = +2^-2 * (1 + 141/1024) = 1165/4096;  0xB0CC = -2^-3 * (1 + 204/1024) = -614/4096
    assert O.codebook_values(np.array([1]), O.MCG)[0] == 551 / 4096
    # mcg, s = 0xFFFF: x = 0x5440E013 -> x' = 0x3F20BB73 ; sum = 1741/2048
    assert O.codebook_values(np.array([0xFFFF]), O.MCG)[0] == 1741 / 2048
    # 3inst, s = 0: x = b = 0x03D45AA4 -> x' = 0x38B431C4
    #   0x31C4 = 2^-3 * (1 + 452/1024);  0x38B4 = 2^-1 * (1 + 180/1024)
    assert O.codebook_values(np.array([0]), O.INST3)[0] == 0.18017578125 + 0.587890625
    # 3inst, s = 1: x = a + b = 0x0925D716 -> x' = 0x3245BC76 ; sum = -7531/8192
    assert O.codebook_values(np.array([1]), O.INST3)[0] == -7531 / 8192
    # mul1, s = 0: bytes sum 0 ; s = 1: x = 0x83DCD12D, bytes 45+209+220+131 = 605
    assert O.codebook_values(np.array([0]), O.MUL1)[0] == -510 / math.sqrt(21845)
    assert O.codebook_values(np.array([1]), O.MUL1)[0] == 95 / math.sqrt(21845)


def _half_fields_times_2_13(h):
    """A normal binary16 with exponent field 12..15, times 2^13, as an exact integer."""
    sign = (h >> 15) & 1
    expo = (h >> 10) & 0x1F
    frac = h & 0x3FF
    assert np.all((expo >= 12) & (expo <= 15))
    mag = (1024 + frac) << (expo - 12)          # (1 + f/1024) 2^(e-15) * 2^13
    return np.where(sign == 1, -mag, mag)


@pytest.mark.parametrize("cb,a,b", [(O.MCG, 0xCBAC1FED, 0), (O.INST3, 89226354, 64248484)])
def test_half_sum_codebooks_from_ieee_fields(cb, a, b):
    x = (a * ALL + b) & 0xFFFFFFFF
    x = (x & 0x8FFF8FFF) ^ 0x3B603B60
    ref = _half_fields_times_2_13(x & 0xFFFF) + _half_fields_times_2_13(x >> 16)
    got = O.codebook_values(ALL, cb) * 8192.0
    assert np.array_equal(got, ref.astype(np.float64))
    # the mask keeps every half a normal number of magnitude in [1/8, 2)
    lo, hi = O.codebook_halves(ALL, cb)
    for v in (lo, hi):
        assert np.all((np.abs(v) >= 0.125) & (np.abs(v) < 2.0))


def test_mul1_is_centred_byte_sum():
    v = O.codebook_values(ALL, O.MUL1)
    k = v * math.sqrt(21845) + 510
    assert np.allclose(k, np.round(k), atol=1e-9)
    assert k.min() >= 0 and k.max() <= 1020
    rng = np.random.default_rng(5)
    for s in rng.integers(0, 65536, size=64):
        x = (0x83DCD12D * int(s)) % (1 << 32)
        assert round(k[s]) == sum(x.to_bytes(4, "little"))


@pytest.mark.parametrize("cb", [O.MUL1, O.MCG, O.INST3])
def test_c_and_numpy_codebooks_agree_on_every_state(cb):
    lib = O.c_oracle()
    c = np.array([lib.oracle_codebook(int(s), cb) for s in range(0, 65536, 7)])
    assert np.array_equal(c, O.codebook_values(np.arange(0, 65536, 7), cb))
