"""Pins for the oracle's stage functions: MX GEMVs, RMSNorm, KV quantisation, SwiGLU FFN.

Expected values come from independent routes: numpy matrix products over matrices that
the test decodes with torch's float8 conversion and the MX specification's e2m1 table,
closed forms for special inputs, and exactness properties.
"""
import numpy as np
import pytest
import torch

from tests.helpers import bf16_f64

E2M1 = np.array([0, .5, 1, 1.5, 2, 3, 4, 6, -0., -.5, -1, -1.5, -2, -3, -4, -6])


def _bf16(a: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _dq8(codes, scales):
    v = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    s = np.exp2(scales.astype(np.float64) - 127)
    return v * np.repeat(np.repeat(s, 32, 0), 32, 1)


def _dq4(packed, scales):
    lo, hi = packed & 0xF, packed >> 4
    nib = np.stack([lo, hi], -1).reshape(packed.shape[0], -1)
    return E2M1[nib] * np.repeat(np.exp2(scales.astype(np.float64) - 127), 32, 1)


@pytest.mark.parametrize("rows,n,k", [(1, 64, 96), (5, 96, 160), (11, 32, 32)])
def test_gemv_mxfp8_matches_numpy(orc, rows, n, k):
    rng = np.random.default_rng(rows * 7 + n)
    codes = rng.integers(0, 256, (n, k), dtype=np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x3C                       # no NaN codes
    scales = rng.integers(110, 135, (n // 32, k // 32), dtype=np.uint8)
    x = _bf16(rng.standard_normal((rows, k)))
    got = orc.gemv_mxfp8(x, codes, scales)
    want = bf16_f64(x) @ _dq8(codes, scales).T
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12 * np.abs(want).max())


@pytest.mark.parametrize("rows,n,k", [(1, 16, 64), (4, 48, 128), (9, 8, 32)])
def test_gemv_mxfp4_matches_numpy(orc, rows, n, k):
    rng = np.random.default_rng(rows * 13 + n)
    packed = rng.integers(0, 256, (n, k // 2), dtype=np.uint8)
    scales = rng.integers(115, 135, (n, k // 32), dtype=np.uint8)
    x = _bf16(rng.standard_normal((rows, k)))
    got = orc.gemv_mxfp4(x, packed, scales)
    want = bf16_f64(x) @ _dq4(packed, scales).T
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12 * np.abs(want).max())


def test_gemv_mxfp4_nibble_order_and_scale_index(orc):
    # element 0 of row 0 is in the LOW nibble; element 33 of row 1 uses scale[1][1]
    n, k = 2, 64
    packed = np.zeros((n, k // 2), np.uint8)
    scales = np.full((n, k // 32), 127, np.uint8)
    packed[0, 0] = 0x02            # element 0 = 1.0, element 1 = 0
    packed[1, 16] = 0x60           # element 32 = 0, element 33 = 4.0
    scales[1, 1] = 129             # x4
    x = np.zeros((1, k), np.float32)
    x[0, 0], x[0, 1], x[0, 33] = 3.0, 5.0, 0.5
    y = orc.gemv_mxfp4(_bf16(x), packed, scales)
    assert y[0, 0] == 3.0 and y[0, 1] == 0.5 * 4.0 * 4.0


def test_gemv_mxfp8_block_scale_index(orc):
    # a 64x64 matrix of ones (code 0x38) with one block scaled: W[j,k] uses scale[j/32][k/32]
    codes = np.full((64, 64), 0x38, np.uint8)
    scales = np.full((2, 2), 127, np.uint8)
    scales[1, 0] = 130                                  # rows 32..63, cols 0..31 -> x8
    x = np.zeros((1, 64), np.float32)
    x[0, 5] = 1.0
    y = orc.gemv_mxfp8(_bf16(x), codes, scales)
    assert np.all(y[0, :32] == 1.0) and np.all(y[0, 32:] == 8.0)


def test_gemv_power_of_two_exact(orc):
    rng = np.random.default_rng(3)
    k, n = 256, 32
    codes = rng.choice(np.array([0x38, 0x40, 0x30, 0xB8, 0x00], np.uint8), (n, k))
    scales = rng.integers(120, 130, (1, k // 32), dtype=np.uint8)
    x = np.exp2(rng.integers(-4, 4, (3, k))).astype(np.float32) * rng.choice([-1, 1], (3, k))
    y = orc.gemv_mxfp8(_bf16(x), codes, scales)
    want = x.astype(np.float64) @ _dq8(codes, scales).T
    assert np.array_equal(y, want)                      # every term exact, every sum exact


def test_rmsnorm_constant_row_and_scale_invariance(orc):
    dim = 512
    g = _bf16(1 + 0.1 * np.random.default_rng(4).standard_normal(dim))
    for c in [0.75, -3.0, 1e-2]:
        x = _bf16(np.full((1, dim), c))
        y = bf16_f64(orc.rmsnorm(x, g, 0.0))
        want = np.sign(c) * bf16_f64(g)                 # |c| / sqrt(c^2) = 1
        assert np.array_equal(y[0], bf16_f64(_bf16(want)))
    x = _bf16(np.random.default_rng(5).standard_normal((3, dim)))
    x2 = _bf16(bf16_f64(x) * 2.0)                       # exact doubling
    assert np.array_equal(orc.rmsnorm(x, g, 0.0), orc.rmsnorm(x2, g, 0.0))


def test_rmsnorm_unit_rms(orc):
    dim = 1024
    ones = _bf16(np.ones(dim))
    x = _bf16(np.random.default_rng(6).standard_normal((4, dim)) * 5)
    y = bf16_f64(orc.rmsnorm(x, ones, 0.0))
    assert np.allclose(np.sqrt((y ** 2).mean(1)), 1.0, atol=2e-3)
    # eps enters as mean(x^2) + eps: a row of zeros stays zero
    z = orc.rmsnorm(np.zeros((1, dim), np.uint16), ones, 1e-6)
    assert not z.any()


def test_kv_quant_ties_saturation_and_zero(orc):
    kv = np.zeros(16, np.float32)
    kv[0] = 448.0                                       # amax 448 -> scale exactly 1
    kv[1], kv[2], kv[3] = 1.0625, 1.1875, -1.0625       # midpoints -> even codes
    kv[4] = 2.0 ** -10                                  # midpoint of 0 and 2^-9 -> even (0)
    codes, s = orc.kv_quant(_bf16(kv))
    assert s == np.float32(1.0)
    assert codes[0] == 0x7E and codes[1] == 0x38 and codes[2] == 0x3A and codes[3] == 0xB8
    assert codes[4] == 0x00
    codes, s = orc.kv_quant(np.zeros(16, np.uint16))
    assert s == np.float32(1.0) and not codes.any()


def test_kv_quant_roundtrip_error(orc):
    rng = np.random.default_rng(7)
    for _ in range(20):
        kv = _bf16(rng.standard_normal(512) * rng.uniform(0.01, 10))
        codes, s = orc.kv_quant(kv)
        v = bf16_f64(kv)
        amax = np.abs(v).max()
        assert np.float32(s) == np.float32(np.float32(amax) / np.float32(448.0))
        deq = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy() * float(s)
        # e4m3 keeps 3 mantissa bits: relative error <= 2^-4 for normals, plus subnormal floor
        assert np.all(np.abs(deq - v) <= np.abs(v) * 2.0 ** -4 + float(s) * 2.0 ** -10 + 1e-12)
        assert np.abs(codes & 0x7F).max() == 0x7E       # the largest element maps to 448


def test_ffn_matches_numpy_composition(orc):
    rng = np.random.default_rng(8)
    H, I, rows = 128, 64, 3
    x = _bf16(rng.standard_normal((rows, H)))
    gu = rng.integers(0, 256, (2 * I, H // 2), dtype=np.uint8)
    gu_s = rng.integers(124, 129, (2 * I, H // 32), dtype=np.uint8)
    d = rng.integers(0, 256, (H, I // 2), dtype=np.uint8)
    d_s = rng.integers(118, 124, (H, I // 32), dtype=np.uint8)
    t, y = orc.ffn(x, gu, gu_s, d, d_s, I, 7.0, fmt4=True)
    a = bf16_f64(x) @ _dq4(gu, gu_s).T
    g, u = np.clip(a[:, :I], -7, 7), np.clip(a[:, I:], -7, 7)
    t_want = _bf16(g / (1 + np.exp(-g)) * u)
    assert np.mean(t == t_want) > 0.995                 # bf16 rounding of near-ties may differ
    y_want = bf16_f64(t) @ _dq4(d, d_s).T
    np.testing.assert_allclose(y, y_want, rtol=1e-10, atol=1e-10 * np.abs(y_want).max())
    assert np.abs(a).max() > 7.0                        # the clamp is exercised
