"""Pins of the oracle's 8-bit float decoding and of FP8-input products.

The formats are the OCP 8-bit floating point ones (E4M3: bias 7, no infinities, S.1111.111 NaN,
largest 448; E5M2: bias 15, IEEE-style).  Expected values are worked by hand from those
definitions, or come from torch's own float8 conversions (an independent implementation)."""
import math

import numpy as np
import pytest
import torch

import oracle

E4M3_CASES = [(0x00, 0.0), (0x80, -0.0), (0x01, 2.0 ** -9), (0x07, 7 * 2.0 ** -9), (0x08, 2.0 ** -6),
              (0x38, 1.0), (0x39, 1.125), (0x40, 2.0), (0xC0, -2.0), (0x7E, 448.0), (0xFE, -448.0),
              (0x77, 240.0), (0x3F, 1.875)]
E5M2_CASES = [(0x00, 0.0), (0x01, 2.0 ** -16), (0x03, 3 * 2.0 ** -16), (0x04, 2.0 ** -14), (0x3C, 1.0),
              (0x3D, 1.25), (0xBC, -1.0), (0x7B, 57344.0), (0x7C, math.inf), (0xFC, -math.inf)]


def _dec(code, b):
    return float(oracle.decode(np.array([b], dtype=np.uint8), code)[0])


def test_e4m3_worked_values():
    for b, v in E4M3_CASES:
        got = _dec(oracle.OR_E4M3, b)
        assert got == v and math.copysign(1, got) == math.copysign(1, v), hex(b)
    assert math.isnan(_dec(oracle.OR_E4M3, 0x7F)) and math.isnan(_dec(oracle.OR_E4M3, 0xFF))


def test_e5m2_worked_values():
    for b, v in E5M2_CASES:
        assert _dec(oracle.OR_E5M2, b) == v, hex(b)
    for b in (0x7D, 0x7E, 0x7F, 0xFD):
        assert math.isnan(_dec(oracle.OR_E5M2, b))


@pytest.mark.parametrize("code,tdt", [(oracle.OR_E4M3, torch.float8_e4m3fn), (oracle.OR_E5M2, torch.float8_e5m2)])
def test_fp8_decode_matches_torch_on_every_byte(code, tdt):
    bits = torch.arange(256, dtype=torch.int64).to(torch.uint8)
    ref = bits.view(tdt).to(torch.float64).numpy()
    got = oracle.decode(bits.numpy(), code)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_fp8_product_small_integers_exact():
    """Integers in [-3, 3] are exact in E4M3; the oracle's product equals an int64 product."""
    g = torch.Generator().manual_seed(5)
    A = torch.randint(-3, 4, (9, 40), generator=g)
    B = torch.randint(-3, 4, (40, 7), generator=g)
    ref = (A @ B).double().numpy()
    Af = A.to(torch.float8_e4m3fn)
    Bf = B.t().contiguous().to(torch.float8_e4m3fn)                     # stored N x K
    got = oracle.gemm_ref(9, 7, 40, Af, oracle.OR_ROW, Bf, oracle.OR_COL, oracle.OR_E4M3)
    assert np.array_equal(got, ref)


def test_fp8_mixed_sign_subnormal_product():
    # a = 2^-9 (E4M3 smallest subnormal), b = -448: the single product is -448 * 2^-9 = -0.875.
    A = np.array([[0x01]], dtype=np.uint8)
    B = np.array([[0xFE]], dtype=np.uint8)
    got = oracle.gemm_ref(1, 1, 1, A, oracle.OR_ROW, B, oracle.OR_COL, oracle.OR_E4M3)
    assert got[0, 0] == -0.875


PINS = [test_e4m3_worked_values, test_e5m2_worked_values, test_fp8_product_small_integers_exact,
        test_fp8_mixed_sign_subnormal_product,
        lambda: test_fp8_decode_matches_torch_on_every_byte(oracle.OR_E4M3, torch.float8_e4m3fn),
        lambda: test_fp8_decode_matches_torch_on_every_byte(oracle.OR_E5M2, torch.float8_e5m2)]
