"""Pins of the oracle's LM head (CPU only).

bf16_round_f64 (one rounding of a double to bf16, ties to even): against torch's fp32 -> bf16
conversion on values fp32 holds exactly (a library routine), against an exact-rational
rounding (fractions.Fraction) on doubles that fp32 cannot hold, and on hand-worked cases:
values where rounding through fp32 first gives another answer, ties, subnormals, overflow,
signed zero and NaN.  lm_head_logits: one-hot hidden rows give the (scaled) W column bit for
bit (W is [V][d] with V != d, so a transposed operand fails), small-integer operands agree
with numpy's exact int64 matmul, and ld padding leaves the columns past V at zero."""
import math
from fractions import Fraction

import numpy as np
import torch

import oracle

BF16_MAX = Fraction(2) ** 127 * (2 - Fraction(1, 128))


def _bits_of(x32) -> np.ndarray:
    """bf16 bit patterns of fp32 values via torch (round to nearest, ties to even)."""
    t = torch.from_numpy(np.ascontiguousarray(x32, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _rne_exact(x: float) -> int:
    """Nearest bf16 to the double x, ties to even, by exact rational arithmetic: the
    quantum at x's binade is 2^(e - 8) for 2^(e-1) <= |x| < 2^e, never below 2^-133."""
    sign = 0x8000 if math.copysign(1.0, x) < 0 else 0
    a = abs(Fraction(x))
    if a == 0:
        return sign
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e <= a:          # make 2^(e-1) <= a < 2^e
        e += 1
    while Fraction(2) ** (e - 1) > a:
        e -= 1
    qe = max(e - 8, -133)
    k = a / Fraction(2) ** qe
    n = k.numerator // k.denominator
    rem = k - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    val = n * Fraction(2) ** qe
    if val > BF16_MAX:
        return sign | 0x7F80
    f = np.array([float(val)], np.float32)   # exact: at most 8 significant bits
    assert Fraction(float(f[0])) == val
    return sign | int(f.view(np.uint32)[0] >> 16)


def test_round_agrees_with_torch_on_fp32_values():
    rng = np.random.default_rng(7)
    mant = rng.uniform(1.0, 2.0, 6000)
    expo = rng.integers(-140, 128, 6000)
    x = (mant * np.exp2(expo.astype(np.float64))).astype(np.float32)
    x = np.concatenate([x, -x[:2000], np.float32([1.0, 3.0, 65504.0, 1e-40, -1e-42])])
    x = x[np.isfinite(x)]
    want = _bits_of(x)
    got = np.array([oracle.bf16_round_f64(float(v)) for v in x], np.uint16)
    assert np.array_equal(got, want)


def test_round_agrees_with_exact_rational_rounding():
    rng = np.random.default_rng(11)
    vals = []
    for _ in range(1500):
        e = int(rng.integers(-140, 127))
        m = 1.0 + float(rng.integers(0, 1 << 52)) * 2.0 ** -52
        vals.append(math.copysign(math.ldexp(m, e), rng.choice([-1.0, 1.0])))
    # midpoints and their neighbours one double ulp away
    for b in rng.integers(0x0001, 0x7F7F, 300):
        lo = Fraction(float(np.array([int(b) << 16], np.uint32).view(np.float32)[0]))
        hi = Fraction(float(np.array([(int(b) + 1) << 16], np.uint32).view(np.float32)[0]))
        mid = float((lo + hi) / 2)
        vals += [mid, math.nextafter(mid, 0.0), math.nextafter(mid, math.inf)]
    for v in vals:
        assert oracle.bf16_round_f64(v) == _rne_exact(v), v


def test_round_hand_worked_cases():
    cases = [
        # 1 + 2^-8 is halfway between 1 (0x3F80) and 1 + 2^-7 (0x3F81): a tiny excess rounds
        # up, although rounding to fp32 first would drop it and round the tie to even
        (1 + 2.0 ** -8 + 2.0 ** -30, 0x3F81),
        (-(1 + 2.0 ** -8 + 2.0 ** -30), 0xBF81),
        (1 + 2.0 ** -8, 0x3F80),                 # tie: even mantissa (0x00)
        (1 + 3 * 2.0 ** -8, 0x3F82),             # tie: even mantissa (0x02)
        (2.0 ** -133, 0x0001),                   # smallest subnormal
        (2.0 ** -134, 0x0000),                   # tie between 0 and 2^-133: to 0
        (3 * 2.0 ** -134, 0x0002),               # tie between 1 and 2 quanta: to 2
        (2.0 ** -134 + 2.0 ** -160, 0x0001),
        (127 * 2.0 ** -133 + 2.0 ** -134, 0x0080),  # largest subnormal + half: to 2^-126
        (float(BF16_MAX), 0x7F7F),
        (float(BF16_MAX) + 2.0 ** 119, 0x7F80),  # halfway to 2^128: ties to even overflow
        (float(BF16_MAX) + 2.0 ** 118, 0x7F7F),
        (1e300, 0x7F80),
        (-1e300, 0xFF80),
        (0.0, 0x0000),
        (-0.0, 0x8000),
        (math.inf, 0x7F80),
    ]
    for x, want in cases:
        assert oracle.bf16_round_f64(x) == want, (x, hex(oracle.bf16_round_f64(x)), hex(want))
    nan = oracle.bf16_round_f64(math.nan)
    assert (nan & 0x7F80) == 0x7F80 and (nan & 0x007F) != 0


def test_lm_head_one_hot_rows_pick_a_column_of_w():
    rng = np.random.default_rng(3)
    V, d = 37, 11
    Wf = rng.normal(0.0, 1.0, (V, d)).astype(np.float32)
    W = _bits_of(Wf)
    Wv = (W.astype(np.uint32) << 16).view(np.float32)
    rows = []
    picks = []
    for r in range(9):
        j, k = int(rng.integers(0, d)), int(rng.integers(-3, 4))
        h = np.zeros(d, np.float32)
        h[j] = 2.0 ** k
        rows.append(h)
        picks.append((j, k))
    H = _bits_of(np.stack(rows))
    got, exact, abssum = oracle.lm_head_logits(H, W, exact=True)
    for r, (j, k) in enumerate(picks):
        col = Wv[:, j].astype(np.float64) * 2.0 ** k
        assert np.array_equal(exact[r], col)
        assert np.array_equal(abssum[r], np.abs(col))
        assert np.array_equal(got[r], _bits_of(col.astype(np.float32)))


def test_lm_head_small_integers_match_exact_matmul():
    rng = np.random.default_rng(5)
    rows, d, V = 5, 300, 257
    Hi = rng.integers(-8, 9, (rows, d))
    Wi = rng.integers(-8, 9, (V, d))
    H = _bits_of(Hi.astype(np.float32))
    W = _bits_of(Wi.astype(np.float32))
    got, exact, abssum = oracle.lm_head_logits(H, W, exact=True)
    ref = Hi @ Wi.T                                   # exact int64
    assert np.array_equal(exact, ref.astype(np.float64))
    assert np.array_equal(abssum, (np.abs(Hi) @ np.abs(Wi).T).astype(np.float64))
    assert np.abs(ref).max() < 2 ** 24                # exact in fp32, so torch rounds the same value
    assert np.array_equal(got, _bits_of(ref.astype(np.float32)))
    assert (ref != (got.astype(np.uint32) << 16).view(np.float32)).any()  # some sums did round


def test_lm_head_ld_padding():
    rng = np.random.default_rng(9)
    H = _bits_of(rng.normal(0, 1, (3, 16)).astype(np.float32))
    W = _bits_of(rng.normal(0, 1, (21, 16)).astype(np.float32))
    a = oracle.lm_head_logits(H, W)
    b = oracle.lm_head_logits(H, W, ld=24)
    assert b.shape == (3, 24)
    assert np.array_equal(b[:, :21], a)
    assert (b[:, 21:] == 0).all()
