"""Pins for the fp64 oracle: each check ties it to something other than itself -- a closed
form, a hand-worked example, brute force, a library routine or an invariant -- so that a
dropped term, a wrong sign or index, or a transposed operand fails one of them.

Sources: the DiffusionGemma vLLM page ("DiffusionGemma: vLLM이 네이티브로 지원하는 최초의
디퓨전 언어 모델(dLLM)"), sections "엔트로피 기반 디노이징" (entropy equation H(p), the
entropy-bound rule, the convergence rule), "자기 조건화" (self-conditioning) and
"DiffusionGemmaModelState와 DiffusionSampler" (Gumbel-max candidate, renoise, argmax canvas);
Salmon et al., SC'11, for Philox-4x32.
"""
import ctypes
import itertools
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import scipy.stats

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
NEG_INF = np.float32(-np.inf)


# ----------------------------------------------------------------------------- Philox
M0, M1 = 0xD2511F53, 0xCD9E8D57
W0, W1 = 0x9E3779B9, 0xBB67AE85
MASK = 0xFFFFFFFF


def _philox_inverse(out, key, rounds):
    """Undo Philox-4x32 round by round.  Each round is a bijection: the low halves of the
    two products give back X0 and X2 through the multipliers' inverses mod 2^32, and the
    high halves then unmask X1 and X3.  Round keys are replayed in reverse order."""
    inv0, inv1 = pow(M0, -1, 1 << 32), pow(M1, -1, 1 << 32)
    keys = []
    k0, k1 = key
    for r in range(rounds):
        if r:
            k0, k1 = (k0 + W0) & MASK, (k1 + W1) & MASK
        keys.append((k0, k1))
    y0, y1, y2, y3 = (int(v) for v in out)
    for k0, k1 in reversed(keys):
        x2 = (y1 * inv1) & MASK
        x0 = (y3 * inv0) & MASK
        hi1 = (M1 * x2) >> 32
        hi0 = (M0 * x0) >> 32
        x1 = y0 ^ hi1 ^ k0
        x3 = y2 ^ hi0 ^ k1
        y0, y1, y2, y3 = x0, x1, x2, x3
    return [y0, y1, y2, y3]


@pytest.mark.parametrize("rounds", [1, 2, 10])
def test_philox_is_the_published_bijection(rounds):
    rng = np.random.default_rng(1)
    for _ in range(200):
        ctr = rng.integers(0, 1 << 32, 4, dtype=np.uint64).astype(np.uint32)
        key = rng.integers(0, 1 << 32, 2, dtype=np.uint64).astype(np.uint32)
        out = oracle.philox4x32(ctr, key, rounds)
        assert _philox_inverse(out, [int(k) for k in key], rounds) == [int(c) for c in ctr]


def test_philox_statistics():
    # byte histogram of 40000 outputs (160000 words) and single-bit avalanche
    rng = np.random.default_rng(2)
    words = []
    for i in range(40000):
        words.extend(oracle.philox4x32([i, 7, 3, 0], [0x1234, 0x5678]))
    b = np.array(words, np.uint32).view(np.uint8)
    chi2, p = scipy.stats.chisquare(np.bincount(b, minlength=256))
    assert p > 1e-4, (chi2, p)
    flips = []
    for _ in range(300):
        ctr = rng.integers(0, 1 << 32, 4, dtype=np.uint64).astype(np.uint32)
        key = rng.integers(0, 1 << 32, 2, dtype=np.uint64).astype(np.uint32)
        bit = int(rng.integers(0, 128))
        c2 = ctr.copy()
        c2[bit // 32] ^= np.uint32(1 << (bit % 32))
        a = oracle.philox4x32(ctr, key)
        z = oracle.philox4x32(c2, key)
        flips.append(sum(bin(int(x) ^ int(y)).count("1") for x, y in zip(a, z)))
    assert abs(np.mean(flips) - 64.0) < 2.0


def test_uniform_mapping():
    assert oracle.uniform(0) == 2.0 ** -24
    assert oracle.uniform(0xFFFFFFFF) == 1.0 - 2.0 ** -24
    rng = np.random.default_rng(3)
    ws = np.sort(rng.integers(0, 1 << 32, 2000, dtype=np.uint64))
    us = [oracle.uniform(int(w)) for w in ws]
    assert all(a <= b for a, b in zip(us, us[1:]))
    for u in us[:200]:
        assert float(np.float32(u)) == u          # exact in fp32
        assert 0.0 < u < 1.0


def test_token_mapping():
    for V in (2, 7, 1024, 262144, 152064):
        assert oracle.token(0, 0, V) == 0
        assert oracle.token(0xFFFFFFFF, 0xFFFFFFFF, V) == V - 1
    # uniform over V = 7 on random words
    rng = np.random.default_rng(4)
    counts = np.zeros(7)
    for _ in range(14000):
        w0, w1 = (int(x) for x in rng.integers(0, 1 << 32, 2, dtype=np.uint64))
        t = oracle.token(w0, w1, 7)
        assert 0 <= t < 7
        counts[t] += 1
    assert scipy.stats.chisquare(counts).pvalue > 1e-4
    # the token is the integer part of x * V / 2^64: monotone in x and splits [0, 2^64) evenly
    assert oracle.token(0x80000000, 0, 2) == 1 and oracle.token(0x7FFFFFFF, 0xFFFFFFFF, 2) == 0
    assert oracle.token(0x40000000, 0, 4) == 1 and oracle.token(0xC0000000, 0, 4) == 3


def test_random_tokens_cover_vocab():
    V = 5
    seen = [oracle.random_token(9, 1, 0, i, oracle.STREAM_RENOISE, V) for i in range(5000)]
    counts = np.bincount(seen, minlength=V)
    assert scipy.stats.chisquare(counts).pvalue > 1e-4
    # streams and steps give different draws
    a = [oracle.random_token(9, 1, 0, i, oracle.STREAM_RENOISE, 1 << 30) for i in range(64)]
    b = [oracle.random_token(9, 1, 0, i, oracle.STREAM_INIT, 1 << 30) for i in range(64)]
    c = [oracle.random_token(9, 1, 1, i, oracle.STREAM_RENOISE, 1 << 30) for i in range(64)]
    assert a != b and a != c


# ----------------------------------------------------------------------------- entropy
@pytest.mark.parametrize("V", [1024, 32768, 152064, 262144])
def test_entropy_uniform_is_log_V(V):
    row = np.full(V, 1.25, np.float32)
    for T in (1.0, 0.3):
        r = oracle.row_stats(row, T=T, sample=False)
        # a sequential fp64 sum of V terms is exact to within V * 2^-53 relative
        bound = V * 2.0 ** -53
        assert r["entropy"] == pytest.approx(math.log(V), rel=bound)
        assert r["entropy_alt"] == pytest.approx(math.log(V), rel=bound)
        assert r["lse"] == pytest.approx(1.25 / T + math.log(V), rel=1e-12)
        assert r["argmax"] == 0


def test_entropy_one_hot_and_supports():
    row = np.full(8, NEG_INF, np.float32)
    row[5] = 3.0
    r = oracle.row_stats(row, sample=True)
    assert r["entropy"] == 0.0 and r["entropy_alt"] == 0.0
    assert r["argmax"] == 5 and r["sample"] == 5
    for j in range(4):   # uniform over 2^j of 8 entries -> j ln 2
        row = np.full(8, NEG_INF, np.float32)
        row[: 1 << j] = -2.0
        assert oracle.row_stats(row, sample=False)["entropy"] == pytest.approx(j * math.log(2), abs=1e-15)


def test_entropy_two_point_is_binary_entropy():
    for a, b, T in [(0.0, 1.0, 1.0), (2.0, -3.0, 0.7), (5.0, 5.0, 2.0)]:
        row = np.full(16, NEG_INF, np.float32)
        row[3], row[11] = a, b
        p = scipy.special.expit((a - b) / T)
        ref = scipy.stats.entropy([p, 1 - p])
        r = oracle.row_stats(row, T=T, sample=False)
        assert r["entropy"] == pytest.approx(ref, rel=1e-12)


def test_entropy_matches_library_and_alt_form():
    rng = np.random.default_rng(5)
    for s in (0.5, 2.0, 8.0, 40.0):
        for T in (1.0, 0.5, 1.5):
            row = (rng.standard_normal(4096) * s).astype(np.float32)
            r = oracle.row_stats(row, T=T, sample=False)
            p = scipy.special.softmax(row.astype(np.float64) / T)
            # -p log p of a probability next to 1 carries an absolute rounding error of a
            # few ulp(1) in either evaluation, hence the absolute floor
            assert r["entropy"] == pytest.approx(scipy.stats.entropy(p), rel=1e-10, abs=1e-15)
            assert r["lse"] == pytest.approx(scipy.special.logsumexp(row.astype(np.float64) / T), rel=1e-13)
            if r["entropy"] > 1e-6:
                assert r["entropy_alt"] == pytest.approx(r["entropy"], rel=1e-9)
            assert 0.0 <= r["entropy"] <= math.log(4096) + 1e-12


def test_entropy_near_one_hot_alt_form_is_accurate():
    # one entry 30 above the rest: H = r (1 + 30) - ... with r = (V-1) e^-30; the split
    # form keeps full relative accuracy where log(1 + r) in one sum would lose it
    V = 1024
    row = np.zeros(V, np.float32)
    row[17] = 30.0
    r = oracle.row_stats(row, sample=False)
    rr = (V - 1) * math.exp(-30.0)
    ref = math.log1p(rr) + 30.0 * rr / (1.0 + rr)
    assert r["entropy_alt"] == pytest.approx(ref, rel=1e-12)
    assert r["entropy"] == pytest.approx(ref, rel=1e-6)


def test_entropy_increases_with_temperature():
    rng = np.random.default_rng(6)
    row = (rng.standard_normal(512) * 3).astype(np.float32)
    Hs = [oracle.row_stats(row, T=T, sample=False)["entropy"] for T in (0.2, 0.5, 1.0, 2.0, 5.0)]
    assert all(a < b for a, b in zip(Hs, Hs[1:]))


def test_bf16_input_path():
    rng = np.random.default_rng(7)
    f = (rng.standard_normal(300) * 4).astype(np.float32)
    bits = (f.view(np.uint32) >> 16).astype(np.uint16)          # truncation to bf16
    widened = (bits.astype(np.uint32) << 16).view(np.float32)
    a = oracle.row_stats(bits, T=0.8, seed=3, position=2)
    b = oracle.row_stats(widened, T=0.8, seed=3, position=2)
    assert a == b


def test_argmax_ties_lowest_index():
    row = np.zeros(10, np.float32)
    row[[4, 7]] = 2.0
    assert oracle.row_stats(row, sample=False)["argmax"] == 4
    assert oracle.row_stats(np.zeros(10, np.float32), sample=False)["argmax"] == 0


# ----------------------------------------------------------------------------- sampling
def test_sample_one_hot_finite_margin():
    row = np.zeros(64, np.float32)
    row[40] = 1000.0
    for pos in range(50):
        r = oracle.row_stats(row, seed=11, position=pos)
        assert r["sample"] == 40
        assert r["score1"] - r["score2"] > 1000.0 - 16.7 - 2.9


@pytest.mark.parametrize("T", [1.0, 0.5])
def test_gumbel_max_samples_softmax(T):
    x = np.array([0.0, 1.0, -1.0, 2.0, 0.5, -2.0, 1.5, 0.25], np.float32)
    p = scipy.special.softmax(x.astype(np.float64) / T)
    counts = np.zeros(8)
    for pos in range(100):
        for step in range(200):
            counts[oracle.row_stats(x, T=T, seed=5, request_id=3, step=step, position=pos)["sample"]] += 1
    res = scipy.stats.chisquare(counts, p * counts.sum())
    assert res.pvalue > 1e-4, (counts, p)


def test_gumbel_noise_range_and_distribution():
    g = np.array([oracle.gumbel(1, 2, 3, 4, v) for v in range(20000)])
    gmax = -math.log(-math.log(1 - 2.0 ** -24))
    gmin = -math.log(-math.log(2.0 ** -24))
    assert g.max() <= gmax and g.min() >= gmin
    assert abs(g.mean() - np.euler_gamma) < 0.03              # Gumbel(0,1) mean
    assert abs(g.var() - math.pi ** 2 / 6) < 0.08


# ----------------------------------------------------------------------------- acceptance
def _golden():
    with open(os.path.join(GOLDEN, "acceptance_4x8.json")) as f:
        return json.load(f)


def _support_logits(g):
    V = g["V"]
    x = np.full((1, len(g["supports"]), V), NEG_INF, np.float32)
    for i, sup in enumerate(g["supports"]):
        x[0, i, sup] = 0.5
    return x


def _params(n, **kw):
    p = {"temperature": np.ones(n, np.float32), "beta": np.ones(n, np.float32),
         "tau": np.full(n, 0.5, np.float32), "k": np.full(n, 2, np.int32),
         "max_steps": np.full(n, 64, np.int32), "min_accept": np.ones(n, np.int32),
         "step": np.zeros(n, np.int32), "request_id": np.arange(n, dtype=np.uint32),
         "flags": np.full(n, oracle.ACTIVE, np.uint32)}
    for k, v in kw.items():
        p[k] = np.broadcast_to(np.asarray(v, p[k].dtype), (n,)).copy()
    return p


def test_acceptance_hand_worked_4x8():
    g = _golden()
    x = _support_logits(g)
    L = x.shape[1]
    for case in g["cases"]:
        p = _params(1, beta=case["beta"], min_accept=case["min_accept"])
        out = oracle.denoise_step(x, p, seed=1, canvas=np.zeros((1, L)),
                                  prev_argmax=np.full((1, L), -1), stable_count=np.zeros(1))
        ln2 = math.log(2)
        assert out["entropy"][0] == pytest.approx([e * ln2 for e in g["entropy_in_ln2"]], abs=1e-15)
        assert list(out["argmax"][0]) == g["argmax"]
        assert out["mean_entropy"][0] == pytest.approx(g["mean_entropy_in_ln2"] * ln2, rel=1e-14)
        assert sorted(np.nonzero(out["accept_mask"][0])[0].tolist()) == case["accepted"], case
        assert out["n_accept"][0] == len(case["accepted"])
        # accepted positions keep their sample; samples lie in the support
        for i in range(L):
            assert out["sample"][0, i] in g["supports"][i]
            if out["accept_mask"][0, i]:
                assert out["canvas"][0, i] == out["sample"][0, i]


def _worked_step():
    with open(os.path.join(GOLDEN, "step_worked_5x4x8.json")) as f:
        return json.load(f)


def _contract_token(seed, request_id, step, position, V):
    """A renoise token by the random-number contract, restated here from its definition: the
    Philox-4x32-10 block (pinned above as the published bijection) at counter (0, position,
    step, 1 | seed bits 32..55 << 8) and key (low word of seed, request_id); the token is the
    integer part of (w0:w1) * V / 2^64 in exact integer arithmetic."""
    w = oracle.philox4x32([0, position, step, 1 | (((seed >> 32) & 0xFFFFFF) << 8)],
                          [seed & 0xFFFFFFFF, request_id])
    return ((int(w[0]) << 32) | int(w[1])) * V >> 64


def worked_step_inputs(g):
    """Logits [n, L, V] (fp32), parameters and initial state of the hand-worked whole step."""
    n, L, V = len(g["canvases"]), g["L"], g["V"]
    x = np.full((n, L, V), NEG_INF, np.float32)
    for c, cv in enumerate(g["canvases"]):
        for i, sup in enumerate(cv["supports"]):
            x[c, i, sup] = 0.5
    flag = {"active": oracle.ACTIVE, "read_only": oracle.READ_ONLY}
    p = {"temperature": np.array([cv["temperature"] for cv in g["canvases"]], np.float32),
         "beta": np.array([cv["beta"] for cv in g["canvases"]], np.float32),
         "tau": np.array([cv["tau"] for cv in g["canvases"]], np.float32),
         "k": np.array([cv["k"] for cv in g["canvases"]], np.int32),
         "max_steps": np.array([cv["max_steps"] for cv in g["canvases"]], np.int32),
         "min_accept": np.array([cv["min_accept"] for cv in g["canvases"]], np.int32),
         "step": np.zeros(n, np.int32),
         "request_id": np.array([cv["request_id"] for cv in g["canvases"]], np.uint32),
         "flags": np.array([sum(flag[f] for f in cv["flags"]) for cv in g["canvases"]], np.uint32)}
    return x, p, np.array(g["initial_canvas"], np.int32)


def check_worked_step(g, t, out, canvas_before, ent_tol, lse_rel):
    """The outputs of step t against the hand-worked values (out: canvas, prev_argmax,
    stable_count, accept_mask, argmax, entropy, lse, converged, mean_entropy, n_accept)."""
    ln2 = math.log(2)
    for c, cv in enumerate(g["canvases"]):
        if cv.get("inactive"):
            assert np.array_equal(out["canvas"][c], canvas_before[c]), (t, c)
            assert (out["prev_argmax"][c] == -1).all() and out["stable_count"][c] == 0, (t, c)
            continue
        ctx = (t, c, cv["what"][:40])
        H = np.array(cv["entropy_in_ln2"], np.float64) * ln2
        assert np.all(np.abs(out["entropy"][c] - H) <= ent_tol), (ctx, out["entropy"][c])
        lse = 0.5 / cv["temperature"] + np.log([len(s) for s in cv["supports"]])
        assert np.all(np.abs(out["lse"][c] - lse) <= lse_rel * np.maximum(np.abs(lse), 1.0)), (ctx, out["lse"][c])
        assert out["argmax"][c].tolist() == cv["argmax"], ctx
        assert out["prev_argmax"][c].tolist() == cv["argmax"], ctx
        assert abs(out["mean_entropy"][c] - cv["mean_entropy_in_ln2"] * ln2) <= ent_tol, ctx
        assert sorted(np.nonzero(out["accept_mask"][c])[0].tolist()) == cv["accepted"], ctx
        assert int(out["n_accept"][c]) == len(cv["accepted"]), ctx
        read_only = "read_only" in cv["flags"]
        for i in range(g["L"]):
            if read_only:
                want = canvas_before[c, i]
            elif i in cv["accepted"]:
                want = cv["supports"][i][0]          # a one-token support: its sample
            else:
                want = _contract_token(g["seed"], cv["request_id"], t, i, g["V"])
            assert out["canvas"][c, i] == want, (ctx, i)
        assert int(out["stable_count"][c]) == cv["stable_count"][t], ctx
        assert int(out["converged"][c]) == cv["converged"][t], ctx


def test_whole_step_hand_worked_5x4x8():
    """The composed step (statistics, acceptance, canvas update, convergence) over three
    steps against values worked out by hand from the method's rules (the fixture's source
    says which): five canvases covering acceptance by the budget, the step cap, read-only,
    inactive and nothing-accepted canvases."""
    g = _worked_step()
    x, p, canvas = worked_step_inputs(g)
    n, L = canvas.shape
    prev, stable = np.full((n, L), -1, np.int32), np.zeros(n, np.int32)
    for t in range(g["steps"]):
        p["step"][:] = t
        out = oracle.denoise_step(x, p, g["seed"], canvas, prev, stable)
        check_worked_step(g, t, out, canvas, ent_tol=1e-15, lse_rel=1e-15)
        canvas, prev, stable = out["canvas"], out["prev_argmax"], out["stable_count"]


def test_acceptance_entropy_only_cases():
    for case in _golden()["entropy_only_cases"]:
        r = oracle.accept(case["H"], case["beta"], case["min_accept"])
        assert r["order"][: r["n_accept"]].tolist() == case["accepted_in_order"], case
        assert r["mask"].sum() == len(case["accepted_in_order"])


def test_acceptance_brute_force():
    """For L <= 12: the accepted count is the largest size of any subset whose entropies
    sum to <= beta, and the accepted set is the (H, index)-smallest subset of that size.
    Entropies are multiples of 1/16 so every sum is exact."""
    rng = np.random.default_rng(8)
    for trial in range(300):
        L = int(rng.integers(1, 13))
        H = rng.integers(0, 48, L) / 16.0
        if trial % 3 == 0:
            H[rng.integers(0, L, L // 2)] = H[0]            # ties
        beta = float(rng.integers(-2, 80)) / 16.0 + (0.0 if trial % 2 else 1.0 / 32)
        best = 0
        for m in range(L, 0, -1):
            if any(sum(H[list(S)]) <= beta for S in itertools.combinations(range(L), m)):
                best = m
                break
        r = oracle.accept(H, beta, min_accept=0)
        assert r["n_accept"] == best, (H, beta)
        keys = sorted((H[i], i) for i in range(L))
        assert sorted(np.nonzero(r["mask"])[0].tolist()) == sorted(i for _, i in keys[:best])
        r1 = oracle.accept(H, beta, min_accept=1)
        assert r1["n_accept"] == max(best, 1)


def test_acceptance_invariants():
    rng = np.random.default_rng(9)
    for _ in range(50):
        H = rng.exponential(1.0, 64)
        prev = -1
        for beta in np.linspace(0, 80, 41):
            r = oracle.accept(H, beta, 1)
            assert r["n_accept"] >= prev
            prev = r["n_accept"]
            acc, rej = H[r["mask"] == 1], H[r["mask"] == 0]
            if acc.size and rej.size:
                assert acc.max() <= rej.min()


# ----------------------------------------------------------------------------- full step
def _random_logits(rng, n, L, V, s=3.0):
    return (rng.standard_normal((n, L, V)) * rng.uniform(0.5, s, (n, L, 1))).astype(np.float32)


def test_step_invariants_and_renoise():
    rng = np.random.default_rng(10)
    n, L, V = 3, 20, 50
    x = _random_logits(rng, n, L, V)
    p = _params(n, beta=[1.0, 5.0, 30.0], step=[0, 3, 7], request_id=[5, 6, 7])
    out = oracle.denoise_step(x, p, seed=0xABCDEF0123, canvas=np.zeros((n, L)),
                              prev_argmax=np.full((n, L), -1), stable_count=np.zeros(n))
    for c in range(n):
        for i in range(L):
            if out["accept_mask"][c, i]:
                assert out["canvas"][c, i] == out["sample"][c, i]
            else:
                assert out["canvas"][c, i] == oracle.random_token(
                    0xABCDEF0123, p["request_id"][c], p["step"][c], i, oracle.STREAM_RENOISE, V)
            r = oracle.row_stats(x[c, i], seed=0xABCDEF0123, request_id=int(p["request_id"][c]),
                                 step=int(p["step"][c]), position=i)
            assert r["sample"] == out["sample"][c, i] and r["argmax"] == out["argmax"][c, i]
        acc = out["entropy"][c][out["accept_mask"][c] == 1]
        rej = out["entropy"][c][out["accept_mask"][c] == 0]
        if acc.size and rej.size:
            assert acc.max() <= rej.min()
    assert out["n_accept"][0] <= out["n_accept"][1] <= out["n_accept"][2]
    assert (out["prev_argmax"] == out["argmax"]).all()


def test_convergence_hand_sequences():
    rng = np.random.default_rng(11)
    L, V = 8, 16
    sharp = np.zeros((1, L, V), np.float32)
    sharp[0, np.arange(L), rng.integers(0, V, L)] = 40.0     # mean entropy ~ 0
    flat = _random_logits(rng, 1, L, V, s=0.6)               # mean entropy ~ log V
    for logits, tau, expect in [(sharp, 0.5, [0, 0, 1]), (flat, 0.5, [0, 0, 0])]:
        p = _params(1, k=2, tau=tau, max_steps=64)
        canvas, prev, stable = np.zeros((1, L)), np.full((1, L), -1), np.zeros(1)
        stables, convs = [], []
        for step in range(3):
            p["step"][:] = step
            out = oracle.denoise_step(logits, p, 1, canvas, prev, stable)
            canvas, prev, stable = out["canvas"], out["prev_argmax"], out["stable_count"]
            stables.append(int(stable[0]))
            convs.append(int(out["converged"][0]))
        assert stables == [0, 1, 2]
        assert convs == expect
    # a change of argmax resets the count
    p = _params(1, k=2, tau=100.0)
    out = oracle.denoise_step(sharp, p, 1, np.zeros((1, L)), np.full((1, L), -1), np.zeros(1))
    prev = out["prev_argmax"].copy()
    prev[0, 3] = (prev[0, 3] + 1) % V
    out2 = oracle.denoise_step(sharp, p, 1, out["canvas"], prev, np.array([5]))
    assert out2["stable_count"][0] == 0 and out2["converged"][0] == 0
    # the step cap converges regardless: S = 1 at step 0, S = 4 at step 3
    for S, step in [(1, 0), (4, 3)]:
        q = _params(1, max_steps=S, step=step, tau=0.0)
        o = oracle.denoise_step(flat, q, 1, np.zeros((1, L)), np.full((1, L), -1), np.zeros(1))
        assert o["converged"][0] == 1
    q = _params(1, max_steps=5, step=3, tau=0.0)
    o = oracle.denoise_step(flat, q, 1, np.zeros((1, L)), np.full((1, L), -1), np.zeros(1))
    assert o["converged"][0] == 0


def test_read_only_and_inactive():
    rng = np.random.default_rng(12)
    n, L, V = 3, 6, 32
    x = _random_logits(rng, n, L, V)
    flags = [oracle.ACTIVE | oracle.READ_ONLY, 0, oracle.ACTIVE]
    p = _params(n, max_steps=[1, 8, 8])
    p["flags"] = np.array(flags, np.uint32)
    canvas0 = rng.integers(0, V, (n, L)).astype(np.int32)
    out = oracle.denoise_step(x, p, 2, canvas0, np.full((n, L), -1), np.zeros(n))
    assert (out["canvas"][0] == canvas0[0]).all() and out["accept_mask"][0].sum() == 0
    assert out["converged"][0] == 1 and (out["sample"][0] == -1).all()
    assert (out["canvas"][1] == canvas0[1]).all() and (out["prev_argmax"][1] == -1).all()
    assert out["entropy"][1].sum() == 0 and out["converged"][1] == 0


def _check_canvas_init(canvas_init, random_token):
    """The Prefill case's canvas: uniform tokens of the init stream (2), position by position,
    for active canvases only -- not the renoise stream's tokens."""
    n, L, V = 2, 300, 7
    p = _params(n, step=[0, 3])
    p["flags"] = np.array([oracle.ACTIVE, 0], np.uint32)
    c = canvas_init(n, L, V, p, 77)
    assert c[0].min() >= 0 and c[0].max() < V and (c[1] == 0).all()
    assert scipy.stats.chisquare(np.bincount(c[0], minlength=V)).pvalue > 1e-4
    req, step = int(p["request_id"][0]), int(p["step"][0])
    init = [random_token(77, req, step, i, oracle.STREAM_INIT, V) for i in range(L)]
    renoise = [random_token(77, req, step, i, oracle.STREAM_RENOISE, V) for i in range(L)]
    assert np.sum(np.array(init) != np.array(renoise)) > L // 2   # the streams differ
    assert list(c[0]) == init


def test_canvas_init_tokens():
    _check_canvas_init(lambda n, L, V, p, seed: oracle.canvas_init(n, L, V, p, seed), oracle.random_token)


# ----------------------------------------------------------------------------- self-conditioning
def _bf16(a):
    a = np.asarray(a, np.float32)
    return ((a.view(np.uint32) + 0x8000) >> 16).astype(np.uint16)   # round-half-up is fine here


def _widen(b):
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def test_pe_one_hot_uniform_linear():
    rng = np.random.default_rng(13)
    V, d = 40, 12
    E = _bf16(rng.standard_normal((V, d)) * 0.02)
    Ef = _widen(E)
    P = np.zeros((3, V))
    P[0, 17] = 1.0
    P[1, :] = 1.0 / V
    P[2] = rng.dirichlet(np.ones(V))
    pe = oracle.pe_from_probs(P, E)
    assert (pe[0] == Ef[17]).all()
    np.testing.assert_allclose(pe[1], Ef.mean(axis=0), rtol=1e-12, atol=1e-18)
    Q = rng.dirichlet(np.ones(V), 2)
    a, b = 0.3, 0.7
    lhs = oracle.pe_from_probs(a * Q[:1] + b * Q[1:], E)
    rhs = a * oracle.pe_from_probs(Q[:1], E) + b * oracle.pe_from_probs(Q[1:], E)
    np.testing.assert_allclose(lhs, rhs, rtol=1e-12, atol=1e-18)
    np.testing.assert_allclose(pe[2], P[2] @ Ef, rtol=1e-12, atol=1e-18)   # library matmul


def _check_gelu(gelu):
    """GELU in its tanh form (Hendrycks & Gimpel) against the exact GELU x * Phi(x):
    * the tanh form is built to agree with x Phi(x) to second order at 0, so
      (gelu(x) - x / 2) / x^2 -> 1 / sqrt(2 pi) (this fixes the tanh argument's scale);
    * with the published cubic coefficient its largest distance from x Phi(x) is 4.73e-4
      (over all x); the pin allows 4.8e-4 (a cubic coefficient of 0.04 or 0.05 gives
      2.9e-3 / 3.0e-3, a scale of 0.8 gives 6.4e-4);
    * gelu(x) - gelu(-x) = x, gelu(0) = 0, and the tails tend to x and 0."""
    assert gelu(0.0) == 0.0
    xs = np.linspace(-8.0, 8.0, 16001)
    exact = 0.5 * xs * (1.0 + scipy.special.erf(xs / math.sqrt(2.0)))   # x * Phi(x)
    got = np.array([gelu(float(x)) for x in xs])
    assert np.abs(got - exact).max() < 4.8e-4
    for x in (1e-4, -1e-4, 3e-5):
        assert abs((gelu(x) - 0.5 * x) / (x * x) - 1.0 / math.sqrt(2.0 * math.pi)) < 1e-6
    for x in (0.3, 1.7, 4.0):
        assert abs(gelu(x) - gelu(-x) - x) < 1e-15 * max(1.0, x)
    assert gelu(30.0) == pytest.approx(30.0)
    assert abs(gelu(-30.0)) < 1e-12


def test_gelu_tanh_properties():
    _check_gelu(oracle.gelu_tanh)


def _mutant_oracle(tmp_path, old, new):
    """A copy of the oracle compiled with one planted mistake (the text `old` of its C
    source replaced by `new`), loaded on its own: the product oracle is never touched."""
    import ctypes
    import subprocess
    src = open(os.path.join(os.path.dirname(oracle.__file__), "dg_oracle.c")).read()
    assert src.count(old) == 1, old
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(old, new))
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O2", "-fPIC", "-shared", "-std=gnu11", "-o", str(so), str(path), "-lm"], check=True)
    lib = ctypes.CDLL(str(so))
    lib.orc_gelu_tanh.argtypes = [ctypes.c_double]
    lib.orc_gelu_tanh.restype = ctypes.c_double
    lib.orc_random_token.argtypes = [ctypes.c_uint64] + [ctypes.c_uint32] * 5
    lib.orc_random_token.restype = ctypes.c_uint32
    P = ctypes.c_void_p
    lib.orc_canvas_init.argtypes = [P, ctypes.c_int64, ctypes.c_int32, ctypes.c_int64, P, P, P, ctypes.c_uint64]

    def canvas_init(n, L, V, p, seed):
        out = np.zeros((n, L), np.int32)
        st = np.ascontiguousarray(p["step"], np.int32)
        rq = np.ascontiguousarray(p["request_id"], np.uint32)
        fl = np.ascontiguousarray(p["flags"], np.uint32)
        lib.orc_canvas_init(out.ctypes.data, n, L, V, st.ctypes.data, rq.ctypes.data, fl.ctypes.data, seed)
        return out
    return lib, canvas_init


@pytest.mark.parametrize("old,new", [("const double k = sqrt(2.0 / M_PI);", "const double k = 0.8;"),
                                     ("0.044715 * z * z * z", "0.04 * z * z * z")])
def test_planted_gelu_mistakes_fail_the_pin(tmp_path, old, new):
    lib, _ = _mutant_oracle(tmp_path, old, new)
    with pytest.raises(AssertionError):
        _check_gelu(lib.orc_gelu_tanh)


def test_planted_canvas_init_stream_fails_the_pin(tmp_path):
    lib, canvas_init = _mutant_oracle(tmp_path, "(uint32_t)i, ORC_STREAM_INIT, (uint32_t)V);",
                                      "(uint32_t)i, ORC_STREAM_RENOISE, (uint32_t)V);")
    with pytest.raises(AssertionError):
        _check_canvas_init(canvas_init, oracle.random_token)


@pytest.mark.parametrize("old,new", [
    # a rejected position renoised with the next position's draw
    ("(uint32_t)step[c], (uint32_t)i, ORC_STREAM_RENOISE, (uint32_t)V);",
     "(uint32_t)step[c], (uint32_t)i + 1u, ORC_STREAM_RENOISE, (uint32_t)V);"),
    # either convergence condition instead of both
    ("(st >= k[c] && Hbar < (double)tau[c])", "(st >= k[c] || Hbar < (double)tau[c])"),
    # the stable count not reset when the argmax canvas changes
    ("int32_t st = same ? stable_count[c] + 1 : 0;", "int32_t st = stable_count[c] + 1;"),
    # the step cap one step late
    ("(step[c] + 1 >= max_steps[c])", "(step[c] >= max_steps[c])"),
])
def test_planted_step_mistakes_fail_the_worked_step(tmp_path, monkeypatch, old, new):
    lib, _ = _mutant_oracle(tmp_path, old, new)
    P, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    lib.orc_denoise_step.argtypes = [P, ctypes.c_int, i64, i64, i32, i64] + [P] * 9 + [ctypes.c_uint64] + [P] * 15 + [ctypes.c_int]
    lib.orc_philox4x32.argtypes = [P, P, ctypes.c_int, P]
    monkeypatch.setattr(oracle, "_lib", lib)   # the wrapper calls the mutant; restored after the test
    g = _worked_step()
    x, p, canvas = worked_step_inputs(g)
    n, L = canvas.shape
    prev, stable = np.full((n, L), -1, np.int32), np.zeros(n, np.int32)
    with pytest.raises(AssertionError):
        for t in range(g["steps"]):
            p["step"][:] = t
            out = oracle.denoise_step(x, p, g["seed"], canvas, prev, stable)
            check_worked_step(g, t, out, canvas, ent_tol=1e-15, lse_rel=1e-15)
            canvas, prev, stable = out["canvas"], out["prev_argmax"], out["stable_count"]


def test_gated_mlp_closed_forms():
    rng = np.random.default_rng(14)
    d, h = 6, 10
    pe = rng.standard_normal((4, d))
    Z = np.zeros((h, d), np.uint16)
    Wd = _bf16(rng.standard_normal((d, h)))
    assert (oracle.gated_mlp(pe, Z, _bf16(rng.standard_normal((h, d))), Wd) == 0).all()
    # d = h = 1: delta = wd * gelu(wg z) * (wu z)
    wg, wu, wd = _bf16([[0.75]]), _bf16([[-1.5]]), _bf16([[2.0]])
    for z in (-2.0, 0.5, 3.0):
        got = oracle.gated_mlp(np.array([[z]]), wg, wu, wd)[0, 0]
        ref = 2.0 * oracle.gelu_tanh(0.75 * z) * (-1.5 * z)
        assert got == pytest.approx(ref, rel=1e-14)
    # the general case against library matmuls in fp64
    Wg, Wu = _bf16(rng.standard_normal((h, d)) * 0.3), _bf16(rng.standard_normal((h, d)) * 0.3)
    g = pe @ _widen(Wg).T
    u = pe @ _widen(Wu).T
    gelu = 0.5 * g * (1.0 + scipy.special.erf(g / math.sqrt(2.0)))
    ref = (gelu * u) @ _widen(Wd).T
    got = oracle.gated_mlp(pe, Wg, Wu, Wd)
    np.testing.assert_allclose(got, ref, rtol=5e-3, atol=1e-3 * np.abs(ref).max())


def test_probs_from_logits_is_softmax():
    rng = np.random.default_rng(15)
    x = (rng.standard_normal((3, 200)) * 5).astype(np.float32)
    T = np.array([1.0, 0.4, 1.3])
    P = oracle.probs_from_logits(x, T)
    np.testing.assert_allclose(P, scipy.special.softmax(x.astype(np.float64) / T[:, None], axis=1),
                               rtol=1e-12, atol=1e-300)
