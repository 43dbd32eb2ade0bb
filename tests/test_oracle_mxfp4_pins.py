"""Pins of the oracle's MXFP4 quantiser (OCP Microscaling block format), on CPU: the E2M1
magnitudes against their bit-level definition, the block scale 2^(floor(log2 max) - 2), exact
round trips of values on the grid, ties to the even mantissa at every midpoint, saturation,
the error bound of one half grid step, zero blocks, the nibble order of the packing, and the
nearest-value rule against brute force over all 16 codes."""
import numpy as np
import pytest

import oracle


def e2m1_value(code):
    """Value of a 4-bit E2M1 code from its bits: sign, exponent (bias 1), mantissa."""
    s = -1.0 if code & 8 else 1.0
    e = (code >> 1) & 3
    m = code & 1
    return s * (m * 0.5 if e == 0 else (1 + m / 2) * 2.0 ** (e - 1))


def test_magnitudes_match_the_bit_level_definition():
    for code in range(16):
        assert oracle.E2M1_MAGNITUDES[code & 7] * (-1 if code & 8 else 1) == e2m1_value(code)


def test_block_scale_is_floor_log2_of_the_maximum_minus_two():
    for amax, e in [(1.0, -2), (0.999, -3), (6.0, 0), (7.99, 0), (8.0, 1), (0.0123, -9), (2.0 ** -100, -102)]:
        w = np.zeros(32)
        w[5] = amax
        _, sc = oracle.mxfp4_quantize(w)
        assert int(sc[0]) - 127 == e


def test_values_on_the_grid_round_trip_exactly():
    rng = np.random.default_rng(0)
    for e in (-10, -3, 0, 4):
        mags = oracle.E2M1_MAGNITUDES[rng.integers(0, 8, size=(50, 32))]
        sign = np.where(rng.random((50, 32)) < 0.5, -1.0, 1.0)
        w = sign * mags * 2.0 ** e
        w[:, 0] = 6.0 * 2.0 ** e                        # block maximum 6 * 2^e: scale 2^e
        p, s = oracle.mxfp4_quantize(w)
        assert np.all(s.astype(int) - 127 == e)
        assert np.array_equal(oracle.mxfp4_dequantize(p, s), w)


@pytest.mark.parametrize("m,expect", [(0.25, 0.0), (0.75, 1.0), (1.25, 1.0), (1.75, 2.0), (2.5, 2.0),
                                      (3.5, 4.0), (5.0, 4.0), (6.5, 6.0), (7.9, 6.0), (0.26, 0.5), (4.99, 4.0)])
def test_ties_to_even_and_saturation(m, expect):
    w = np.zeros(32)
    w[0] = 4.0                                          # scale 1
    w[1], w[2] = m, -m
    p, s = oracle.mxfp4_quantize(w)
    d = oracle.mxfp4_dequantize(p, s)
    assert s[0] == 127 and d[1] == expect and d[2] == -expect


def test_error_within_half_a_grid_step():
    rng = np.random.default_rng(1)
    w = rng.normal(size=(200, 64)) * np.exp(rng.normal(size=(200, 1)))
    p, s = oracle.mxfp4_quantize(w)
    d = oracle.mxfp4_dequantize(p, s)
    X = np.repeat(np.ldexp(1.0, s.astype(int) - 127), 32, axis=-1)
    m = np.abs(w) / X
    half_step = np.where(m < 2, 0.25, np.where(m < 4, 0.5, 1.0))
    bound = np.where(m <= 6, half_step, m - 6) * X
    assert np.all(np.abs(d - w) <= bound * (1 + 1e-12))


def test_zero_block_and_nibble_order():
    p, s = oracle.mxfp4_quantize(np.zeros(32))
    assert s[0] == 0 and not p.any()
    w = np.zeros(32)
    w[0], w[1], w[2] = 4.0, 1.0, -0.5                   # codes 6, 2, 9 at scale 1
    p, s = oracle.mxfp4_quantize(w)
    assert p[0] == (6 | (2 << 4)) and p[1] == 9


def test_nearest_code_against_brute_force():
    rng = np.random.default_rng(2)
    w = rng.normal(size=(100, 32))
    p, s = oracle.mxfp4_quantize(w)
    codes = np.empty(w.shape, dtype=np.int64)
    codes[:, 0::2], codes[:, 1::2] = p & 15, p >> 4
    X = np.ldexp(1.0, s.astype(int)[:, 0] - 127)
    vals = np.array([e2m1_value(c) for c in range(16)])
    for r in range(w.shape[0]):
        for i in range(32):
            v = w[r, i] / X[r]
            err = np.abs(vals - v)
            best = err.min()
            ok = [c for c in range(16) if err[c] == best and (c & 8) == (8 if v < 0 else 0)]
            # the chosen code is a nearest one of the right sign, even mantissa on a tie
            assert codes[r, i] in ok, (r, i, v)
            if len(ok) > 1:
                assert codes[r, i] % 2 == 0
