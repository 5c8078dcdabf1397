"""Pins of the oracle's LM-head logits (the producer fused in front of chain verification),
each independent of the code it checks:

- bf16 rounding: values that IEEE 754 round-to-nearest-even fixes by hand (ties to the even
  significand, a value just above a tie that a float intermediate would round twice, the
  subnormal spacing 2^-133, overflow to infinity at the first tie above the largest finite
  bf16, NaN, signed zero);
- on every fp32 value the rounding agrees with the bit-level fp32 -> bf16 rounding of the
  input generators (a separate implementation: integer arithmetic on the bit pattern);
- the product: exact rational arithmetic (Python fractions) on tiny non-square shapes, rounded
  to bf16 by exact integer rounding, must give the oracle's bit patterns (a transposed operand,
  a dropped term or a wrong index changes them);
- the integer-grid workload keeps every logit an exact multiple of 2^-9, so the oracle's
  float64 values are exact there.
"""

from fractions import Fraction

import numpy as np
import pytest

from workloads import bf16_to_f32, f32_to_bf16, lmhead_grid

INF = 0x7F80


@pytest.mark.parametrize("x,bits", [
    (1.0, 0x3F80),
    (1 + 2.0 ** -8, 0x3F80),                 # tie: to the even significand (down)
    (1 + 3 * 2.0 ** -8, 0x3F82),             # tie: to the even significand (up)
    (1 + 2.0 ** -8 + 2.0 ** -40, 0x3F81),    # just above a tie: up (via float it would tie)
    (1 + 2.0 ** -8 - 2.0 ** -40, 0x3F80),
    (-2.5, 0xC020),
    (3.140625, 0x4049),
    (2.0 ** -133, 0x0001),                   # the smallest bf16 subnormal
    (2.0 ** -134, 0x0000),                   # tie between 0 and it: to even (zero)
    (3 * 2.0 ** -134, 0x0002),               # tie between 1 and 2 units: to even
    (2.0 ** -126, 0x0080),                   # the smallest normal
    ((2 - 2.0 ** -7) * 2.0 ** 127, 0x7F7F),  # the largest finite bf16
    ((2 - 2.0 ** -8) * 2.0 ** 127, INF),     # tie above it: to infinity
    (-1e300, 0x8000 | INF),
    (0.0, 0x0000),
    (-0.0, 0x8000),
    (float("inf"), INF),
    (float("nan"), 0x7FC0),
])
def test_round_bf16_by_hand(orc, x, bits):
    assert int(orc.round_bf16(np.array([x]))[0]) == bits


def test_round_bf16_matches_bit_level_rounding_on_floats(orc):
    """For values a float holds exactly, rounding from double equals rounding the float's bit
    pattern with integer arithmetic (the input generators' conversion)."""
    rng = np.random.default_rng(11)
    x = (rng.standard_normal(200000) * np.exp2(rng.integers(-60, 60, 200000))).astype(np.float32)
    # ties: floats whose low 16 bits are exactly 0x8000, with odd and even kept parts
    tie = (rng.integers(0x3F000000 >> 16, 0x47000000 >> 16, 2000).astype(np.uint32) << 16) | 0x8000
    x = np.concatenate([x, tie.view(np.float32), -tie.view(np.float32)])
    np.testing.assert_array_equal(orc.round_bf16(x.astype(np.float64)), f32_to_bf16(x))


def _exact_bf16_bits(q: Fraction) -> int:
    """bf16 bit pattern of the exact rational q (normal range), round to nearest even, by
    integer arithmetic: q = n * 2^e with 2^7 <= n < 2^8 after rounding."""
    if q == 0:
        return 0
    sign = 0x8000 if q < 0 else 0
    a = abs(q)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    n = round(a / Fraction(2) ** (e - 7))     # Python rounds ties to even
    if n == 256:
        n, e = 128, e + 1
    assert -126 <= e <= 127
    return sign | ((e + 127) << 7) | (n - 128)


@pytest.mark.parametrize("M,V,H,seed", [(3, 5, 4, 0), (2, 7, 9, 1), (5, 3, 16, 2), (1, 1, 1, 3)])
def test_lm_head_logits_brute_force(orc, M, V, H, seed):
    rng = np.random.default_rng(seed)
    h = f32_to_bf16((rng.standard_normal((M, H)) * 1.7).astype(np.float32))
    w = f32_to_bf16((rng.standard_normal((V, H)) * 0.6).astype(np.float32))
    hf, wf = bf16_to_f32(h), bf16_to_f32(w)
    want = np.empty((M, V), np.uint16)
    for m in range(M):
        for v in range(V):
            s = sum(Fraction(float(hf[m, k])) * Fraction(float(wf[v, k])) for k in range(H))
            want[m, v] = _exact_bf16_bits(s)
    got, exact = orc.lm_head_logits(h, w)
    assert got.shape == (M, V) and exact.shape == (M, V)
    np.testing.assert_array_equal(got, want)


def test_lm_head_logits_grid_is_exact(orc):
    li = lmhead_grid(B=3, gamma=2, V=512, Ht=192, Hd=128)
    bits, exact = orc.lm_head_logits(li.hidden_t, li.head_t)
    assert bits.shape == (3 * 3, 512)
    scaled = exact * 512
    np.testing.assert_array_equal(scaled, np.round(scaled))   # multiples of 2^-9
    assert np.abs(exact).max() < 2.0 ** 15
    # the grid's two models: draft logits stay close to the target's at the same position
    dbits, dexact = orc.lm_head_logits(li.hidden_d, li.head_d)
    tgt_rows = exact.reshape(3, 3, 512)[:, :2].reshape(6, 512)
    assert 0.5 < np.std(dexact - tgt_rows) < 2.0
    assert 2.0 < np.std(exact) < 4.5
