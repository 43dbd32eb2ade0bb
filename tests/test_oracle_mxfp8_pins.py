"""Pins of the oracle's MXFP8 activation quantiser (OCP Microscaling block format with FP8
E4M3 elements) and of where the MXFP4 layer applies it, on CPU: every E4M3 code against its
bit-level definition, the block scale 2^(floor(log2 max) - 8), exact round trips of every
finite value, ties to the even mantissa at every midpoint of a binade, saturation at 448, the
subnormal grid, -0 for negative values that round to zero, the nearest-value rule against
brute force over all 254 finite codes, the half-step error bound, and a scalar-loop statement
of a tiny MXFP4 layer."""
import math

import numpy as np
import pytest

import oracle


def e4m3_by_bits(code):
    """Value of an 8-bit E4M3 code from its bits: sign, 4 exponent bits (bias 7), 3 mantissa bits."""
    s = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 15
    m = code & 7
    if e == 15 and m == 7:
        return math.nan
    if e == 0:
        return s * m * 2.0 ** -9
    return s * (8 + m) * 2.0 ** (e - 10)


FINITE = [c for c in range(256) if not math.isnan(e4m3_by_bits(c))]
VALUES = np.array([e4m3_by_bits(c) for c in FINITE])


def test_every_code_decodes_to_its_bit_level_value():
    assert len(FINITE) == 254
    dec = oracle.e4m3_decode(np.arange(256))
    for c in range(256):
        ref = e4m3_by_bits(c)
        assert (math.isnan(ref) and math.isnan(dec[c])) or dec[c] == ref
    assert VALUES.max() == 448.0 and np.min(np.abs(VALUES[VALUES != 0])) == 2.0 ** -9


@pytest.mark.parametrize("amax,e", [(1.0, -8), (0.999, -9), (448.0, 0), (511.9, 0), (512.0, 1),
                                    (3.0e-3, -17), (2.0 ** -100, -108), (2.0 ** -200, -127), (1.0e30, 91)])
def test_block_scale_is_floor_log2_of_the_maximum_minus_eight(amax, e):
    v = np.zeros(32)
    v[7] = -amax
    _, sc = oracle.mxfp8_quantize(v)
    assert int(sc[0]) - 127 == e


def test_every_finite_value_round_trips_exactly():
    for e in (-20, -5, 0, 3, 60):
        v = np.resize(VALUES, (8, 32)) * 2.0 ** e
        v[:, 0] = 448.0 * 2.0 ** e                     # block maximum 448 * 2^e: scale 2^e
        codes, sc = oracle.mxfp8_quantize(v)
        assert np.all(sc.astype(int) - 127 == e)
        assert np.array_equal(oracle.mxfp8_dequantize(codes, sc), v)


def test_midpoints_go_to_the_even_mantissa():
    pos = np.unique(VALUES[VALUES > 0])
    for lo, hi in zip(pos[:-1], pos[1:]):
        mid = (lo + hi) / 2
        v = np.zeros(32)
        v[0] = 448.0                                   # scale 1
        v[1], v[2], v[3], v[4] = mid, -mid, np.nextafter(mid, 0), np.nextafter(mid, 1e9)
        codes, sc = oracle.mxfp8_quantize(v)
        d = oracle.mxfp8_dequantize(codes, sc)
        even = lo if int(oracle.e4m3_encode(np.array([lo]), np.array([False]))[0]) % 2 == 0 else hi
        assert d[1] == even and d[2] == -even, (lo, hi)
        assert d[3] == lo and d[4] == hi


@pytest.mark.parametrize("x,expect", [(448.0, 448.0), (460.0, 448.0), (464.0, 448.0), (500.0, 448.0),
                                      (511.99, 448.0), (416.0, 416.0), (431.9, 416.0), (432.0, 448.0), (440.0, 448.0)])
def test_saturation_at_448(x, expect):
    """The top binade [256, 512) has step 32: 416 and 448 are its last values (432 ties to 448,
    the even mantissa); everything past 448 saturates."""
    v = np.zeros(32)
    v[0] = 300.0                                       # floor(log2 300) = 8: scale 1
    v[1] = x
    codes, sc = oracle.mxfp8_quantize(v)
    assert sc[0] == 127 and oracle.mxfp8_dequantize(codes, sc)[1] == expect


def test_subnormal_grid_and_negative_zero():
    v = np.zeros(32)
    v[0] = 256.0                                       # scale 1: values below 2^-6 are subnormal
    v[1:6] = [2.0 ** -9, 1.5 * 2.0 ** -9, 2.5 * 2.0 ** -9, 0.5 * 2.0 ** -9, 7.5 * 2.0 ** -9]
    v[6], v[7] = -0.4 * 2.0 ** -9, -0.0
    codes, sc = oracle.mxfp8_quantize(v)
    d = oracle.mxfp8_dequantize(codes, sc)
    assert list(d[1:6] / 2.0 ** -9) == [1.0, 2.0, 2.0, 0.0, 8.0]   # ties to even; 8 * 2^-9 = 2^-6
    assert codes[5] == 0x08                            # 2^-6 is the first normal: E = 1, m = 0
    assert codes[6] == 0x80 and codes[7] == 0x00 and d[6] == 0.0


def test_zero_block():
    codes, sc = oracle.mxfp8_quantize(np.zeros((2, 64)))
    assert np.all(codes == 0) and np.all(sc == 0)


def test_nearest_value_against_brute_force():
    rng = np.random.default_rng(4)
    v = rng.normal(size=(64, 32)) * np.exp(3 * rng.normal(size=(64, 1)))
    codes, sc = oracle.mxfp8_quantize(v)
    d = oracle.mxfp8_dequantize(codes, sc)
    X = np.ldexp(1.0, sc.astype(np.int64) - 127)[:, :, None].repeat(32, -1).reshape(64, 32)
    for i in range(64):
        for j in range(32):
            cand = VALUES * X[i, j]
            dist = np.abs(cand - v[i, j])
            best = cand[dist == dist.min()]
            assert d[i, j] in best
            assert (codes[i, j] >= 0x80) == (v[i, j] < 0)


def test_error_within_half_a_grid_step():
    rng = np.random.default_rng(5)
    v = rng.normal(size=(300, 64)) * np.exp(rng.normal(size=(300, 1)))
    codes, sc = oracle.mxfp8_quantize(v)
    d = oracle.mxfp8_dequantize(codes, sc)
    X = np.repeat(np.ldexp(1.0, sc.astype(np.int64) - 127), 32, axis=-1)
    a = np.abs(v) / X
    step = np.ldexp(1.0, (np.maximum(np.floor(np.log2(np.maximum(a, 2.0 ** -30))), -6) - 3).astype(np.int64))
    sat = a > 448.0                                    # past the largest value: saturation
    assert sat.any() and np.all(np.abs(d[sat]) == 448.0 * X[sat])
    assert np.all(np.abs(d - v)[~sat] <= 0.5 * step[~sat] * X[~sat])
    assert np.all(a < 512.0)


def test_scalar_loop_layer_matches_the_oracle():
    """A tiny MXFP4 layer written as scalar loops (tokens, features, contraction): x_lat and h
    are the MXFP8 round trips of their rows in blocks of 32; the weights are dequantised MXFP4."""
    rng = np.random.default_rng(6)
    T, d, dl, E, k, I, Is = 3, 64, 64, 3, 2, 64, 32
    inp = dict(x=rng.normal(size=(T, d)), W_r=rng.normal(size=(E, d)) / 8, bias=np.zeros(E),
               W_in=rng.normal(size=(dl, d)) / 8, gamma=1 + 0.1 * rng.normal(size=dl),
               W_out=rng.normal(size=(d, dl)) / 8, W13_s=rng.normal(size=(1, 2 * Is, d)) / 8,
               W2_s=rng.normal(size=(1, d, Is)) / 6)
    inp["W13"] = oracle.mxfp4_dequantize(*oracle.mxfp4_quantize(rng.normal(size=(E, 2 * I, dl)) / 8))
    inp["W2"] = oracle.mxfp4_dequantize(*oracle.mxfp4_quantize(rng.normal(size=(E, dl, I)) / 8))
    ref = oracle.forward(inp, k, mx_activations=True)
    sel, gates = ref["topk_idx"], ref["gates"]
    slot_pos = oracle.permutation(sel, E)[3]
    forced = dict(x_lat=np.zeros((T, dl)), h=np.zeros((T * k, I)), slot_pos=slot_pos)
    for t in range(T):
        x_lat = [sum(inp["x"][t, i] * inp["W_in"][o, i] for i in range(d)) for o in range(dl)]
        x_q = oracle.mxfp8_round_trip(np.array(x_lat))
        forced["x_lat"][t] = x_q
        c = [0.0] * dl
        for j in range(k):
            e = int(sel[t, j])
            h = []
            for f in range(I):
                g = sum(x_q[i] * inp["W13"][e][f, i] for i in range(dl))
                u = sum(x_q[i] * inp["W13"][e][I + f, i] for i in range(dl))
                h.append(4 * math.tanh(g / 4) / (1 + math.exp(-g)) * 25 * math.tanh(u / 25))
            h_q = oracle.mxfp8_round_trip(np.array(h))
            forced["h"][slot_pos[t, j]] = h_q
            for o in range(dl):
                c[o] += gates[t, j] * sum(h_q[f] * inp["W2"][e][o, f] for f in range(I))
        assert np.allclose(c, ref["c"][t], rtol=1e-12, atol=1e-12)
    # the same decisions handed in as forced ones (rows of h in permutation order) give the same layer
    again = oracle.forward(inp, k, forced_topk_idx=sel, forced_mx=forced)
    assert np.allclose(again["y"], ref["y"], rtol=1e-12, atol=1e-12)
    sub = oracle.forward(inp, k, forced_topk_idx=sel, forced_mx=forced, tokens=[2, 0])
    assert np.allclose(sub["y"], ref["y"][[2, 0]], rtol=1e-12, atol=1e-12)
