"""Pins for the oracle's number formats: MX element/scale decode, e4m3 encode, bf16 rounding.

Each check is against something other than the oracle itself: the worked values of the
OCP MX specification (tests/golden/mx_formats.txt), brute force over the whole code
space, or torch's own float8 / bfloat16 conversions.
"""
import math
import os

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "mx_formats.txt")


def _golden():
    rows = []
    for line in open(GOLDEN):
        line = line.split("#")[0].strip()
        if line:
            fmt, code, val = line.split()
            rows.append((fmt, int(code, 0), float(val)))
    return rows


def test_golden_worked_values(orc):
    dec = {"e4m3": orc.e4m3, "e2m1": orc.e2m1, "e8m0": orc.e8m0}
    rows = _golden()
    assert len(rows) >= 30
    for fmt, code, val in rows:
        got = dec[fmt](code)
        if math.isnan(val):
            assert math.isnan(got), (fmt, hex(code))
        else:
            assert got == val and math.copysign(1, got) == math.copysign(1, val), (fmt, hex(code), got, val)


def test_e4m3_matches_torch_float8_for_every_code(orc):
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in range(256):
        got = orc.e4m3(c)
        if math.isnan(ref[c]):
            assert math.isnan(got), hex(c)
        else:
            assert got == ref[c], (hex(c), got, ref[c])


def test_e4m3_code_space_structure(orc):
    pos = [orc.e4m3(c) for c in range(0x7F)]            # 0x00 .. 0x7E
    assert all(b > a for a, b in zip(pos, pos[1:]))      # strictly increasing
    assert pos[-1] == 448.0
    assert [orc.e4m3(c | 0x80) for c in range(0x7F)] == [-v for v in pos]
    sub = pos[:8]                                        # subnormals: uniform spacing 2^-9
    assert np.allclose(np.diff(sub), 2.0 ** -9, rtol=0, atol=0)
    for e in range(1, 16):                               # each binade: 8 equal steps
        vals = [orc.e4m3((e << 3) | m) for m in range(8 if e < 15 else 7)]
        steps = np.diff(vals)
        assert np.all(steps == steps[0])


def test_e2m1_table_and_sign(orc):
    mags = [orc.e2m1(n) for n in range(8)]
    assert mags == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    assert [orc.e2m1(n | 8) for n in range(8)] == [-m for m in mags]


def test_e8m0_is_power_of_two(orc):
    for e in range(255):
        assert orc.e8m0(e) == 2.0 ** (e - 127)
    assert math.isnan(orc.e8m0(255))


def _brute_e4m3(v: float) -> int:
    """Nearest finite e4m3 code by exhaustive search; ties go to the even code."""
    if math.isnan(v):
        return 0x7F
    sign = 0x80 if math.copysign(1, v) < 0 else 0
    a = min(abs(v), 448.0)
    best, bd = None, None
    for c in range(0x7F):
        d = abs(torch.tensor([c], dtype=torch.uint8).view(torch.float8_e4m3fn).item() - a)
        if bd is None or d < bd or (d == bd and c % 2 == 0 and best % 2 == 1):
            best, bd = c, d
    return sign | best


def test_encode_e4m3_is_nearest_even_and_saturates(orc):
    rng = np.random.default_rng(0)
    vals = list(rng.standard_normal(400) * np.exp2(rng.uniform(-12, 10, 400)))
    # exact midpoints between neighbouring codes, both sides of the subnormal boundary
    for c in [0x00, 0x01, 0x06, 0x07, 0x08, 0x38, 0x39, 0x3A, 0x6F, 0x7D]:
        lo = torch.tensor([c], dtype=torch.uint8).view(torch.float8_e4m3fn).item()
        hi = torch.tensor([c + 1], dtype=torch.uint8).view(torch.float8_e4m3fn).item()
        vals += [(lo + hi) / 2, -(lo + hi) / 2]
    vals += [448.0, 449.0, 464.0, 500.0, 1e9, -1e9, 0.0, -0.0, 1e-30, -1e-30]
    for v in vals:
        v32 = float(np.float32(v))
        assert orc.encode_e4m3(v32) == _brute_e4m3(v32), v32


def test_encode_e4m3_agrees_with_torch_in_range(orc):
    rng = np.random.default_rng(1)
    v = (rng.standard_normal(5000) * 100).astype(np.float32)
    v = np.clip(v, -448, 448)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([orc.encode_e4m3(float(x)) for x in v], dtype=np.uint8)
    assert np.array_equal(got, ref)


def test_round_bf16_matches_torch(orc):
    rng = np.random.default_rng(2)
    v = (rng.standard_normal(20000) * np.exp2(rng.uniform(-140, 120, 20000))).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([orc.round_bf16(float(x)) for x in v])
    assert np.array_equal(got, ref)


def test_round_bf16_ties_to_even(orc):
    assert orc.round_bf16(1 + 2.0 ** -8) == 1.0                    # midpoint -> even (1.0)
    assert orc.round_bf16(1 + 3 * 2.0 ** -8) == 1 + 2.0 ** -6      # midpoint -> even
    assert orc.round_bf16(1 + 2.0 ** -8 + 2.0 ** -30) == 1 + 2.0 ** -7
    assert orc.bf16_bits(1.0) == 0x3F80 and orc.bf16_bits(-2.0) == 0xC000


@pytest.mark.parametrize("g,u", [(-10, 1), (-7, 1), (0, 3), (7, 1), (10, 1), (2, 10), (2, -10), (10, -10)])
def test_swiglu_clamp_closed_form(orc, g, u):
    gc, uc = max(-7, min(7, g)), max(-7, min(7, u))
    want = gc / (1 + math.exp(-gc)) * uc
    assert orc.swiglu(g, u, 7.0) == pytest.approx(want, rel=1e-15, abs=0)
