"""Pins of the oracle's single-pass-read, embedding and commit functions (CPU only).

choice_probs: closed forms (two tokens, uniform row), the full distribution summing to one,
probability ratios exp((x_i - x_j) / T), unused slots.  embed_canvas: a plain lookup returns
E's bit patterns, every rounding checked against an independent exact-rational rounding
(fractions.Fraction, both neighbours compared, ties to even), invalid tokens.  commit: a
hand-worked fixture."""
import math
from fractions import Fraction

import numpy as np
import pytest

import oracle
from entropy_bounded_denoising_gb300 import synth


def _bf16_bits(x):
    return (np.asarray(x, np.float32).view(np.uint32) >> 16).astype(np.uint16)


def _bf16_value(bits: int) -> Fraction:
    f = np.array([int(bits) << 16], np.uint32).view(np.float32)[0]
    return Fraction(float(f))


def _rne_bf16_exact(q: Fraction) -> int:
    """Nearest bf16 (ties to even) of an exact rational, by comparing both neighbours."""
    f = np.float32(float(q))               # within one fp32 ulp of q
    b = int(np.array([f], np.float32).view(np.uint32)[0]) >> 16
    cands = {(b + k) & 0xFFFF for k in (-2, -1, 0, 1, 2)}
    best = None
    for c in cands:
        if (c & 0x7F80) == 0x7F80:         # skip inf / NaN patterns
            continue
        err = abs(_bf16_value(c) - q)
        key = (err, c & 1)                 # smaller error, then even mantissa
        if best is None or key < best[0]:
            best = (key, c)
    return best[1]


def _rne_fp32_exact(q: Fraction) -> Fraction:
    f = np.float32(float(q))
    u = int(np.array([f], np.float32).view(np.uint32)[0])
    cands = []
    for k in (-1, 0, 1):
        g = np.array([u + k], np.uint32).view(np.float32)[0]
        cands.append((abs(Fraction(float(g)) - q), (u + k) & 1, Fraction(float(g))))
    cands.sort()
    return cands[0][2]


# ------------------------------------------------------------------ choice_probs
def test_choice_two_tokens_closed_form():
    for a, b, T in [(0.0, 1.0, 1.0), (2.5, -1.25, 0.5), (10.0, 9.0, 2.0), (-3.0, -3.0, 1.0)]:
        row = np.array([[a, b]], np.float32)
        p = oracle.choice_probs(row, [T], np.array([[0, 1]], np.int32))[0]
        pa = 1.0 / (1.0 + math.exp((b - a) / T))
        assert abs(p[0] - pa) <= 1e-15 and abs(p[1] - (1.0 - pa)) <= 1e-15


def test_choice_uniform_row():
    V = 1000
    row = np.full((1, V), 3.0, np.float32)
    p = oracle.choice_probs(row, [0.7], np.array([[0, 17, 999]], np.int32))[0]
    assert np.allclose(p, 1.0 / V, rtol=1e-13)


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_choice_full_distribution_sums_to_one(dtype):
    V = 3000
    x = synth.host_logits(synth.logits(1, 4, V, seed=3, step=1, scale=(0.5, 12.0), dtype=dtype))[0]
    ch = np.tile(np.arange(V, dtype=np.int32), (4, 1))
    T = np.array([1.0, 0.5, 1.3, 2.0])
    p = oracle.choice_probs(x, T, ch)
    assert np.allclose(p.sum(axis=1), 1.0, rtol=0, atol=1e-12)
    # ratios: p_i / p_j = exp((x_i - x_j) / T)
    if dtype == "bf16":
        xv = (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    else:
        xv = x.astype(np.float64)
    for r in range(4):
        i, j = 5, 2000
        assert abs(math.log(p[r, i] / p[r, j]) - (xv[r, i] - xv[r, j]) / T[r]) <= 1e-9


def test_choice_unused_slots_are_zero():
    row = np.array([[1.0, 2.0, 3.0]], np.float32)
    p = oracle.choice_probs(row, [1.0], np.array([[-1, 3, 1000, 2]], np.int32))[0]
    assert p[0] == 0.0 and p[1] == 0.0 and p[2] == 0.0 and p[3] > 0.6


# ------------------------------------------------------------------ embed_canvas
def test_bf16_round_against_exact_rounding():
    rng = np.random.default_rng(1)
    vals = np.concatenate([rng.standard_normal(4000) * 10.0 ** rng.integers(-6, 6, 4000),
                           [1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -(1.0 + 2 ** -8), 1.0 + 2 ** -8 + 2 ** -20,
                            0.0, -0.0, 65504.0, 1e-30]]).astype(np.float32)
    for v in vals:
        got = oracle.bf16_round(float(v))
        if v == 0.0:
            assert got in (0x0000, 0x8000)
            continue
        assert got == _rne_bf16_exact(Fraction(float(v))), (float(v), hex(got))


def test_embed_plain_lookup_is_exact():
    V, d = 50, 24
    E = _bf16_bits(np.random.default_rng(2).standard_normal((V, d)) * 0.02)
    cv = np.array([[0, 49, 7, 7], [3, 1, 2, 48]], np.int32)
    out = oracle.embed_canvas(cv, E)
    assert np.array_equal(out, E[cv.reshape(-1)])


def test_embed_fma_against_exact_arithmetic():
    rng = np.random.default_rng(3)
    V, d = 20, 16
    E = _bf16_bits(rng.standard_normal((V, d)))
    cv = rng.integers(0, V, 6).astype(np.int32)
    delta = _bf16_bits(rng.standard_normal((6, d)) * 0.3)
    for scale in (1.0, 64.0, 0.70710677):
        out = oracle.embed_canvas(cv, E, delta, scale)
        s = Fraction(float(np.float32(scale)))
        for r in range(6):
            for j in range(d):
                q = s * _bf16_value(E[cv[r], j]) + _bf16_value(delta[r, j])
                want = _rne_bf16_exact(_rne_fp32_exact(q))
                assert out[r, j] == want, (scale, r, j)


def test_embed_invalid_tokens_give_zero_rows():
    E = _bf16_bits(np.ones((4, 8)))
    out = oracle.embed_canvas(np.array([-1, 4, 2], np.int32), E, _bf16_bits(np.ones((3, 8))))
    assert (out[0] == 0).all() and (out[1] == 0).all() and (out[2] == _bf16_bits(2.0)).all()


# ------------------------------------------------------------------ commit
def test_commit_fixture():
    conv = np.array([1, 0, 1, 1], np.uint8)
    active = np.array([1, 1, 0, 1], np.uint8)       # canvas 2 committed in an earlier step
    argmax = np.arange(12, dtype=np.int32).reshape(4, 3)
    tokens = np.full((4, 3), -9, np.int32)
    prev = np.full((4, 3), 5, np.int32)
    stable = np.array([3, 2, 4, 1], np.int32)
    r = oracle.commit(conv, active, argmax, tokens, prev, stable)
    assert list(r["committed"]) == [1, 0, 0, 1]
    assert (r["tokens"][0] == [0, 1, 2]).all() and (r["tokens"][3] == [9, 10, 11]).all()
    assert (r["tokens"][1] == -9).all() and (r["tokens"][2] == -9).all()
    assert (r["prev_argmax"][[0, 3]] == -1).all() and (r["prev_argmax"][[1, 2]] == 5).all()
    assert list(r["stable_count"]) == [0, 2, 4, 0]
