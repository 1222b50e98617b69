"""Pins of the oracle's Q4_0 dequantisation and binary16 encoder.

Format ("02 . 8m/8m(2) -- Tiled wmma f16 prefill GEMM (LANDED)", section 3.2): 32 weights per
18-byte block, an f16 scale d then 16 bytes; weight i is the low nibble of byte i, weight 16+i
its high nibble; value d * (nibble - 8) rounded to binary16.  The expected values below are
worked by hand from that definition and from the binary16 format, or come from numpy's own
float16 conversion (an independent implementation).
"""
import numpy as np
import pytest

import oracle


def block(d_bits: int, q: list[int]) -> bytes:
    assert len(q) == 16
    return bytes([d_bits & 0xff, d_bits >> 8] + q)


def decode_values(blocks: bytes, N: int, K: int) -> np.ndarray:
    raw = np.frombuffer(blocks, dtype=np.uint8).reshape(N, -1)
    return oracle.q4_0_to_f16(raw, N, K).view(np.float16).astype(np.float64)


# ------------------------------------------------------------------ binary16 encoder
ENCODER_CASES = [
    (1.0, 0x3C00), (-2.0, 0xC000), (65504.0, 0x7BFF), (65519.99, 0x7BFF),
    (65520.0, 0x7C00),                      # halfway between 65504 and 65536: ties to even = overflow
    (2.0 ** -24, 0x0001), (2.0 ** -25, 0x0000), (1.5 * 2.0 ** -25, 0x0001), (2.0 ** -14, 0x0400),
    (1023 * 2.0 ** -24, 0x03FF), (1023.5 * 2.0 ** -24, 0x0400),   # subnormal tie rounds up to the even normal
    (1 + 2.0 ** -11, 0x3C00), (1 + 3 * 2.0 ** -11, 0x3C02),        # ties go to the even fraction
    (-0.0, 0x8000), (float("inf"), 0x7C00), (float("-inf"), 0xFC00), (1e9, 0x7C00),
]


@pytest.mark.parametrize("x,bits", ENCODER_CASES)
def test_f16_encoder_worked_values(x, bits):
    assert oracle.f64_to_f16_bits(x) == bits


def all_encoder_cases():
    for x, bits in ENCODER_CASES:
        test_f16_encoder_worked_values(x, bits)


def test_f16_encoder_nan():
    b = oracle.f64_to_f16_bits(float("nan"))
    assert (b & 0x7C00) == 0x7C00 and (b & 0x03FF) != 0


def test_f16_encoder_matches_numpy_on_random_values():
    g = np.random.default_rng(7)
    xs = np.concatenate([g.normal(0, 1, 4000), g.normal(0, 1e-5, 4000), g.normal(0, 3e4, 2000),
                         g.uniform(-7e4, 7e4, 2000)])
    got = np.array([oracle.f64_to_f16_bits(x) for x in xs], dtype=np.uint16)
    with np.errstate(over="ignore"):
        ref = xs.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, ref)


def test_f16_encoder_round_trips_every_finite_half():
    bits = np.arange(0, 0x10000, dtype=np.uint32)
    finite = bits[(bits & 0x7C00) != 0x7C00].astype(np.uint16)
    vals = oracle.decode_f16(finite)
    back = np.array([oracle.f64_to_f16_bits(v) for v in vals[::7]], dtype=np.uint16)
    assert np.array_equal(back, finite[::7])


# ------------------------------------------------------------------ Q4_0 decode
def test_q4_0_nibble_order_and_offset():
    # d = 1: byte i holds low nibble i and high nibble 15 - i.
    q = [i | ((15 - i) << 4) for i in range(16)]
    v = decode_values(block(0x3C00, q), 1, 32)[0]
    assert list(v[:16]) == [i - 8 for i in range(16)]
    assert list(v[16:]) == [7 - i for i in range(16)]


def test_q4_0_scale_and_sign():
    q = [0x8F] * 16                          # low nibble 15 -> +7, high nibble 8 -> 0
    v = decode_values(block(0xB800, q), 1, 32)[0]   # d = -0.5
    assert np.all(v[:16] == -3.5) and np.all(v[16:] == 0.0)


def test_q4_0_product_rounds_to_nearest_even():
    # d = 1 + 2^-10; 7 * d = 7.0068359375 lies between the binary16 neighbours 7.00390625 and
    # 7.0078125 (spacing 2^-8) at 1.75 spacings above 7: it rounds up to 7.0078125.
    v = decode_values(block(0x3C01, [0x0F] * 16), 1, 32)[0]
    assert np.all(v[:16] == 7.0078125) and np.all(v[16:] == -8 * (1 + 2.0 ** -10))


def test_q4_0_subnormal_products():
    # d = 3 * 2^-24 (subnormal): -7 d and 7 d are subnormals, exact.
    v = decode_values(block(0x0003, [0x1F] * 16), 1, 32)[0]
    assert np.all(v[:16] == 21 * 2.0 ** -24) and np.all(v[16:] == -21 * 2.0 ** -24)
    # d = 1023 * 2^-24: 7 d = 7161 * 2^-24 needs 13 bits; at exponent -12 the spacing is 4 * 2^-24,
    # 7161 / 4 = 1790.25 -> 1790 -> 7160 * 2^-24.
    v = decode_values(block(0x03FF, [0x0F] * 16), 1, 32)[0]
    assert np.all(v[:16] == 7160 * 2.0 ** -24)


def test_q4_0_overflow_is_infinite():
    v = decode_values(block(0x7BFF, [0x0F] * 16), 1, 32)[0]     # 7 * 65504 > 65520
    assert np.all(np.isinf(v[:16])) and np.all(v[16:] < 0) and np.all(np.isinf(v[16:]))


def test_q4_0_rows_pitch_and_block_order():
    # Two rows of two blocks at a 40-byte pitch (4 padding bytes that must be ignored).
    rows = []
    for n in range(2):
        r = b""
        for b in range(2):
            d = [0x3C00, 0x4000][b]                       # 1.0, 2.0
            r += block(d, [((n + b + i) % 16) for i in range(16)])
        rows.append(r + bytes([0xAA] * 4))
    v = decode_values(b"".join(rows), 2, 64)
    for n in range(2):
        for b, d in enumerate((1.0, 2.0)):
            exp = [d * (((n + b + i) % 16) - 8) for i in range(16)] + [-8 * d] * 16
            assert list(v[n, 32 * b:32 * b + 32]) == exp


def test_q4_0_rejects_bad_shapes():
    with pytest.raises(ValueError):
        oracle.q4_0_to_f16(np.zeros((1, 18), np.uint8), 1, 40)        # K not a multiple of 32
    with pytest.raises(ValueError):
        oracle.q4_0_to_f16(np.zeros((1, 30), np.uint8), 1, 64)        # pitch shorter than 2 blocks


def test_q4_0_gemm_identity_selects_dequantised_weights():
    # A = I (M = K): C[m, n] = W[n, m], the dequantised weight itself (exact).
    N, K = 5, 32
    g = np.random.default_rng(3)
    raw = np.zeros((N, 18), np.uint8)
    for n in range(N):
        raw[n] = np.frombuffer(block(int(np.float16(0.25 * (n + 1)).view(np.uint16)),
                                     list(g.integers(0, 256, 16))), np.uint8)
    W = oracle.q4_0_to_f16(raw, N, K).view(np.float16).astype(np.float64)
    A = np.eye(K, dtype=np.float16).view(np.uint16)
    C = oracle.gemm_ref_q4_0(K, N, K, A, oracle.OR_ROW, raw)
    assert np.array_equal(C, W.T)


# Zero-argument pins, also run against planted mistakes by test_oracle_mutations.
PINS = [all_encoder_cases, test_f16_encoder_nan, test_f16_encoder_matches_numpy_on_random_values,
        test_q4_0_nibble_order_and_offset, test_q4_0_scale_and_sign, test_q4_0_product_rounds_to_nearest_even,
        test_q4_0_subnormal_products, test_q4_0_overflow_is_infinite, test_q4_0_rows_pitch_and_block_order,
        test_q4_0_gemm_identity_selects_dequantised_weights]
