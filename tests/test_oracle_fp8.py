"""Pins for the oracle's FP8 block quantization (no GPU).

* the E4M3 format's closed forms: the encodings of chosen values (largest
  finite 448, one, the smallest normal 2^-6 and subnormal 2^-9, ties to even,
  saturation, the sign of zero) and the values of chosen codes;
* brute force: every rounding equals the nearest of the 254 finite code
  values (ties to the even code), found by search over the whole table;
* the code table round-trips;
* the block scale: the smallest power of two with amax <= 448 * 2^k, checked
  against its definition; blocks are independent;
* the dequantized weight is within half a code spacing (times the scale) of
  the original and is what the decode functions compute with.
"""
import numpy as np
import pytest

from oracle import mla_oracle as om

FINITE = np.array([c for c in range(256) if c not in (0x7F, 0xFF)])


def test_encodings_of_chosen_values():
    cases = {448.0: 0x7E, 1.0: 0x38, -2.0: 0xC0, 2.0 ** -6: 0x08, 2.0 ** -9: 0x01, 7 * 2.0 ** -9: 0x07,
             2.0 ** -10: 0x00,           # half the smallest subnormal: tie to the even code 0
             3 * 2.0 ** -11: 0x01,       # above the tie: up
             1.0625: 0x38,               # 1 + 1/16: tie between 1.0 (even) and 1.125
             1.1875: 0x3A,               # tie between 1.125 and 1.25 (even)
             500.0: 0x7E, -1e9: 0xFE,    # saturation
             -1e-5: 0x80, 0.0: 0x00}     # rounds to zero, sign kept
    for x, code in cases.items():
        got = int(om.e4m3_bits(om.e4m3_round(np.array([x])))[0])
        assert got == code, f"{x}: {got:#x} != {code:#x}"


def test_values_of_chosen_codes():
    cases = {0x7E: 448.0, 0x01: 2.0 ** -9, 0x08: 2.0 ** -6, 0x3F: 1.875, 0xFE: -448.0, 0x38: 1.0, 0x40: 2.0,
             0x77: 240.0, 0x00: 0.0}
    for code, v in cases.items():
        assert om.e4m3_value(np.array([code]))[0] == v


def test_code_table_round_trips():
    vals = om.e4m3_value(FINITE)
    assert np.array_equal(om.e4m3_bits(om.e4m3_round(vals)), FINITE.astype(np.uint8))
    # 127 distinct non-negative values (with +0 and -0 equal)
    assert len(np.unique(np.abs(vals))) == 127


def test_rounding_is_nearest_code_by_brute_force():
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.standard_normal(4000) * 10.0 ** rng.uniform(-4, 2.7, 4000),
                        om.e4m3_value(FINITE[:126]) * 1.0,                   # exact codes
                        (om.e4m3_value(FINITE[1:126]) + om.e4m3_value(FINITE[:125])) / 2])  # ties
    x = x[np.abs(x) <= 448]
    table = om.e4m3_value(FINITE)
    got = om.e4m3_round(x)
    for xi, gi in zip(x, got):
        d = np.abs(table - xi)
        best = np.flatnonzero(d == d.min())
        cand = table[best]
        if len(set(np.abs(cand))) > 1:           # a tie: the code with an even mantissa
            even = [c for c, v in zip(FINITE[best], cand) if (c & 1) == 0]
            assert abs(gi) == abs(om.e4m3_value(np.array([even[0]]))[0]), (xi, gi, cand)
        else:
            assert abs(gi) == abs(cand[0]), (xi, gi, cand)


def test_block_scale_exponent_definition():
    for amax, k in [(448.0, 0), (449.0, 1), (224.0, -1), (224.5, 0), (0.0, 0), (1.0, -8), (0.05, -13)]:
        assert om.block_scale_exponent(amax) == k, amax
    rng = np.random.default_rng(5)
    for amax in 10.0 ** rng.uniform(-6, 4, 500):
        k = om.block_scale_exponent(amax)
        assert amax <= 448.0 * 2.0 ** k and amax > 448.0 * 2.0 ** (k - 1)


def test_block_quantization_blocks_are_independent_and_close():
    rng = np.random.default_rng(9)
    w = 0.02 * rng.standard_normal((300, 260))
    w[128:256, 0:128] *= 1000.0                       # one loud block
    r = om.quantize_fp8_blocks(w)
    assert r["exp"].shape == (3, 3)
    k_quiet = om.block_scale_exponent(float(np.max(np.abs(w[0:128, 0:128]))))
    assert r["exp"][0, 0] == k_quiet and r["exp"][1, 0] > k_quiet + 5
    # |w - q s| <= half the code spacing at |w| (2^(e-4) s), spacing 2^-9 s below 2^-6 s
    for i in range(3):
        for j in range(3):
            sl = (slice(i * 128, (i + 1) * 128), slice(j * 128, (j + 1) * 128))
            s = 2.0 ** r["exp"][i, j]
            a = np.abs(w[sl]) / s
            half = np.where(a >= 2.0 ** -6, 2.0 ** (np.floor(np.log2(np.maximum(a, 1e-300))) - 4), 2.0 ** -10) * s
            assert np.all(np.abs(w[sl] - r["w"][sl]) <= half * (1 + 1e-12))
    # the codes decode to the stored weights
    exp_full = np.repeat(np.repeat(r["exp"], 128, 0), 128, 1)[:300, :260]
    np.testing.assert_array_equal(om.e4m3_value(r["codes"]) * 2.0 ** exp_full, r["w"])


def test_quantized_weights_change_only_the_five_matrices():
    dims = om.Dims(d=16, H=2, q_lora=8, kv_lora=8, nope=4, rope=4, v=4)
    rng = np.random.default_rng(1)
    w = {n: (1 + 0.1 * rng.standard_normal(s)) if n.startswith("g_") else 0.3 * rng.standard_normal(s)
         for n, s in om.weight_shapes(dims).items()}
    q = om.quantize_weights_fp8(w)
    for n in w:
        if n in om.FP8_MATRICES:
            assert not np.array_equal(q[n], w[n]) and np.max(np.abs(q[n] - w[n])) <= np.max(np.abs(w[n])) / 16
        else:
            assert q[n] is w[n]
