"""Pins for the oracle's e4m3 quantiser (CPU).

The e4m3 format is fixed by its published definition (OCP 8-bit floating
point, E4M3): 1 sign, 4 exponent bits (bias 7), 3 mantissa bits, subnormals
m * 2^-9, no infinities, largest finite 448.  The values below follow from
that definition by hand; a slip in the oracle's decode (bias, subnormal
scale, NaN placement) or encode (tie rule, saturation, sign) fails one."""
import numpy as np

from oracle import quant as oq


def test_decode_known_codes():
    t = oq.decode_table()
    want = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x38: 1.0, 0x39: 1.125,
            0x3C: 1.5, 0x40: 2.0, 0x30: 0.5, 0x77: 240.0, 0x78: 256.0, 0x7E: 448.0,
            0xB8: -1.0, 0xFE: -448.0, 0x80: 0.0}
    for code, v in want.items():
        assert t[code] == v, hex(code)
    assert np.signbit(t[0x80])
    assert np.isnan(t[0x7F]) and np.isnan(t[0xFF])
    assert np.isnan(t).sum() == 2


def test_every_finite_code_round_trips():
    t = oq.decode_table()
    codes = np.array([c for c in range(256) if not np.isnan(t[c])], dtype=np.uint8)
    assert np.array_equal(oq.encode(t[codes]), codes)


def test_ties_go_to_the_even_code_and_halfway_rounds_up_or_down():
    # between 1.0 (0x38) and 1.125 (0x39): the midpoint goes to 0x38, just above to 0x39
    assert oq.encode([1.0625])[0] == 0x38
    assert oq.encode([1.0625 + 1e-9])[0] == 0x39
    # between 1.125 (0x39) and 1.25 (0x3A): the midpoint goes to 0x3A
    assert oq.encode([1.1875])[0] == 0x3A
    assert oq.encode([1.1875 - 1e-9])[0] == 0x39
    # subnormal midpoint between 2^-9 (0x01) and 2 * 2^-9 (0x02) -> 0x02; below 2^-10 -> 0
    assert oq.encode([1.5 * 2.0 ** -9])[0] == 0x02
    assert oq.encode([0.5 * 2.0 ** -9])[0] == 0x00
    assert oq.encode([0.5 * 2.0 ** -9 + 1e-12])[0] == 0x01


def test_saturation_and_sign():
    assert list(oq.encode([448.0, 460.0, 1e6, -1e6, -0.0, -1.0])) == [0x7E, 0x7E, 0x7E, 0xFE, 0x80, 0xB8]


def test_nearest_value_on_random_inputs():
    rng = np.random.default_rng(0)
    x = rng.standard_normal(100000) * 64.0
    y = oq.decode(oq.encode(x))
    t = oq.decode_table()
    finite = np.sort(np.unique(np.abs(t[~np.isnan(t)])))
    # brute force: no representable value is strictly closer
    a = np.abs(x)
    best = np.min(np.abs(finite[None, :] - np.minimum(a, 448.0)[:, None]), axis=1)
    assert np.all(np.abs(np.abs(y) - np.minimum(a, 448.0)) <= best + 0.0)
    assert np.all(np.sign(y) == np.sign(x))


def test_quantize_multiplies_in_float32():
    # 1 + 2^-23 is a float32 value; times 1.0 it stays above the tie point of
    # nothing, but (1.0625 + 2^-20) * 1 in float32 keeps the bit that moves
    # the tie: the product is taken in float32 before the e4m3 rounding.
    x = np.float32(1.0625) + np.float32(2.0 ** -20)
    assert oq.quantize([x], 1.0)[0] == 0x39
    assert oq.quantize([np.float32(1.0625)], 1.0)[0] == 0x38
