"""GPU parity of the LM head fused with the step's statistics (dg_lm_head_logits,
dg_lm_head_denoise_step) against the oracle: logits = bf16(hidden . W^T), rounded once,
then the oracle's denoising step on exactly those logits.

With small-integer operands every dot product is exact in fp32, so the stored logits must
equal the oracle's bit for bit, and the step's outputs follow dg_denoise_step's comparison
rules (decisions exact except counted boundary positions, entropy 1e-5 relative, lse 1e-6).
With normal operands the fp32 accumulation can fall on the other side of a bf16 rounding
midpoint: a stored logit may then differ, but only to the rounding of a sum within the
accumulation's error bound of the exact one, and the statistics agree within the
first-order effect of those differences.  At the benchmark's full size (8 x 256, V = 262144,
d = 4096) sampled rows are checked against the oracle and every canvas's decisions against
dg_denoise_step run on the stored logits."""
import numpy as np
import pytest
import torch

import entropy_bounded_denoising_gb300 as dg
from entropy_bounded_denoising_gb300 import synth
import oracle

from helpers import BOUNDARY, H_ATOL, H_RTOL, LSE_ATOL, LSE_RTOL, StepBuffers, compare_step, run_step

pytestmark = pytest.mark.gpu
DEV = "cuda"
SEED = 0x1EAD5EED
SENTINEL = 0x7FC1  # a NaN pattern the library never writes


def _params(n, rng, roles):
    """roles: one of "normal", "read_only", "inactive", "sample_all" per canvas."""
    p = {"temperature": rng.uniform(0.5, 1.5, n).astype(np.float32),
         "beta": rng.uniform(2.0, 16.0, n).astype(np.float32), "tau": np.full(n, 0.3, np.float32),
         "k": np.full(n, 2, np.int32), "max_steps": np.full(n, 64, np.int32),
         "min_accept": np.ones(n, np.int32), "step": np.ones(n, np.int32),
         "request_id": np.arange(n, dtype=np.uint32) + 77, "flags": np.full(n, dg.DG_ACTIVE, np.uint32)}
    for c, r in enumerate(roles):
        if r == "read_only":
            p["flags"][c] = dg.DG_ACTIVE | dg.DG_READ_ONLY
            p["max_steps"][c] = 1
        elif r == "inactive":
            p["flags"][c] = 0
        elif r == "sample_all":
            p["flags"][c] = dg.DG_ACTIVE | dg.DG_SAMPLE_ALL
    return p


def _run(hidden, W, p, V, ld, canvas0, prev0, stable0):
    n, L, _ = hidden.shape
    b = StepBuffers.make(n, L, DEV, canvas0, prev0, stable0)
    logits = torch.full((n, L, ld), SENTINEL, dtype=torch.int16, device=DEV).view(torch.bfloat16)
    pt = dg.params_tensor(p, DEV)
    dg.dg_clear_device_status()
    dg.dg_lm_head_denoise_step(hidden, W, pt, SEED, logits, b.canvas, b.prev, b.stable, b.accept,
                               b.argmax, b.sample, b.entropy, b.lse, b.converged, b.mean_entropy,
                               b.n_accept, V=V)
    torch.cuda.synchronize()
    return b, logits, pt


def _no_sample_all(p):
    q = {k: np.asarray(v).copy() for k, v in p.items()}
    q["flags"] = q["flags"] & ~np.uint32(dg.DG_SAMPLE_ALL)
    return q


@pytest.mark.parametrize("n,L,V,ld,d,roles", [
    (4, 200, 5003, 5008, 192, ("normal", "read_only", "inactive", "sample_all")),
    (2, 256, 32768, 32768, 512, ("normal", "normal")),
    (3, 37, 300, 304, 64, ("normal", "inactive", "normal")),
    (1, 1, 2, 8, 8, ("normal",)),
])
def test_lm_head_step_exact_operands(n, L, V, ld, d, roles):
    rng = np.random.default_rng(V + d)
    hidden = synth.hidden_states(n, L, d, seed=d, kind="int", device=DEV)
    W = synth.lm_head_weights_int(V, d, seed=V, device=DEV)
    p = _params(n, rng, roles)
    canvas0 = rng.integers(0, V, (n, L)).astype(np.int32)
    prev0 = np.where(rng.random((n, 1)) < 0.5, -1, rng.integers(0, V, (n, L))).astype(np.int32)
    stable0 = rng.integers(0, 2, n).astype(np.int32)
    b, logits, _ = _run(hidden, W, p, V, ld, canvas0, prev0, stable0)
    assert dg.dg_get_device_status() == 0
    got = synth.bf16_bits(logits)
    hb, Wb = synth.bf16_bits(hidden), synth.bf16_bits(W)
    ref = np.zeros((n, L, ld), np.uint16)
    for c in range(n):
        if roles[c] == "inactive":
            assert (got[c] == SENTINEL).all(), c            # rows of inactive canvases untouched
            continue
        ref[c] = oracle.lm_head_logits(hb[c], Wb, ld=ld)
        assert np.array_equal(got[c, :, :V], ref[c, :, :V]), c
        assert (got[c, :, V:] == SENTINEL).all()            # padding columns untouched
    o = oracle.denoise_step(ref, p, SEED, canvas0, prev0, stable0, ld=ld, V=V)
    g = b.host()
    rep = compare_step(g, o, _no_sample_all(p), V, SEED, canvas0, prev0, stable0)
    print(rep)
    # DG_SAMPLE_ALL has no effect on the fused step: samples only where accepted
    drawn = g["sample"] >= 0
    for c in range(n):
        if roles[c] in ("normal", "sample_all"):
            assert np.array_equal(drawn[c], g["accept"][c] == 1), c


def test_lm_head_logits_only():
    n, L, V, d = 2, 130, 1000, 136
    hidden = synth.hidden_states(n, L, d, seed=5, kind="int", device=DEV)
    W = synth.lm_head_weights_int(V, d, seed=6, device=DEV)
    p = _params(n, np.random.default_rng(1), ("normal", "inactive"))
    logits = torch.full((n, L, V), float("nan"), dtype=torch.bfloat16, device=DEV)
    dg.dg_clear_device_status()
    dg.dg_lm_head_logits(hidden, W, dg.params_tensor(p, DEV), logits)
    torch.cuda.synchronize()
    assert dg.dg_get_device_status() == 0
    got = synth.bf16_bits(logits)
    assert np.array_equal(got[0], oracle.lm_head_logits(synth.bf16_bits(hidden)[0], synth.bf16_bits(W)))
    assert torch.isnan(logits[1].float()).all()


def test_lm_head_step_normal_operands():
    """bf16 operands with normal entries (the LM head tied to the embedding table): a stored
    logit may differ from the oracle's only where some sum within the fp32 accumulation's
    error bound of the exact one rounds to it (one bf16 step near a rounding midpoint; more
    where the sum nearly cancels)."""
    n, L, V, d = 2, 256, 32768, 1024
    rng = np.random.default_rng(17)
    hidden = synth.hidden_states(n, L, d, seed=21, kind="normal", device=DEV)
    E = synth.weights(V, d, 8, seed=22, device=DEV)[0]
    p = _params(n, rng, ("normal", "normal"))
    canvas0 = rng.integers(0, V, (n, L)).astype(np.int32)
    b, logits, _ = _run(hidden, E, p, V, V, canvas0, np.full((n, L), -1, np.int32), np.zeros(n, np.int32))
    assert dg.dg_get_device_status() == 0
    got = synth.bf16_bits(logits)
    g = b.host()
    hb, Eb = synth.bf16_bits(hidden), synth.bf16_bits(E)
    flips_total = 0
    for c in range(n):
        ref, exact, abssum = oracle.lm_head_logits(hb[c], Eb, exact=True)
        diff = got[c] != ref
        flips_total += int(diff.sum())
        if diff.any():
            # the stored value must be the rounding of some sum within the fp32 accumulation's
            # error bound of the exact one (rounding is monotone: bracket by the bound's ends)
            gv = (got[c][diff].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
            bound = d * 2.0 ** -23 * abssum[diff]          # fp32 accumulation, any order (x2)
            for e, bd, v in zip(exact[diff], bound, gv):
                lo = np.array([oracle.bf16_round_f64(e - bd) << 16], np.uint32).view(np.float32)[0]
                hi = np.array([oracle.bf16_round_f64(e + bd) << 16], np.uint32).view(np.float32)[0]
                assert lo <= v <= hi, (e, bd, v)
        T = float(p["temperature"][c])
        x = (ref.astype(np.uint32) << 16).view(np.float32).astype(np.float64) / T
        xg = (got[c].astype(np.uint32) << 16).view(np.float32).astype(np.float64) / T
        for i in range(L):
            st = oracle.row_stats(ref[i], T, sample=False)
            m = x[i].max()
            pr = np.exp(x[i] - st["lse"])
            dl = np.abs(xg[i] - x[i])
            # first-order effect of the flipped logits (x2 margin)
            h_slack = 2 * float((pr * dl * (np.abs(np.log(np.maximum(pr, 1e-300)) + st["entropy"]) + dl)).sum())
            l_slack = 2 * float((pr * dl).sum())
            assert abs(g["entropy"][c, i] - st["entropy"]) <= H_RTOL * st["entropy"] + H_ATOL + h_slack, (c, i)
            assert abs(g["lse"][c, i] - st["lse"]) <= (LSE_RTOL * abs(st["lse"]) + LSE_ATOL) + l_slack, (c, i)
            if g["argmax"][c, i] != st["argmax"]:
                # only where a flipped logit reaches the maximum
                assert dl[g["argmax"][c, i]] > 0 or dl[st["argmax"]] > 0, (c, i)
                assert xg[i][g["argmax"][c, i]] == xg[i].max() and x[i][st["argmax"]] == m
    print(f"logits one bf16 step off (near-midpoint sums): {flips_total} of {n * L * V}")


def _near_cut(H, beta, min_accept, rel=1e-5):
    """Whether a canvas's acceptance cut is within `rel` of a decision boundary (the sort
    or the budget), judged on fp64 entropies."""
    Hs = np.sort(H.astype(np.float64))
    cs = np.cumsum(Hs)
    n_acc = min(max(int(min_accept), int((cs <= beta).sum())), len(Hs))
    near = False
    if 0 < n_acc < len(Hs):
        near |= abs(Hs[n_acc] - Hs[n_acc - 1]) <= rel * max(Hs[n_acc], 1e-30)
    for j in (n_acc - 1, n_acc):
        if 0 <= j < len(Hs):
            near |= abs(cs[j] - beta) <= rel * max(abs(beta), 1e-30)
    return near


def test_lm_head_batched_full_size():
    """The benchmark's LM-head workload, 8 x 256 positions, V = 262144, d = 4096, with
    small-integer operands (exact logits): sampled rows against the oracle, and every
    canvas's outputs against dg_denoise_step run on the stored logits (same samples and
    tokens wherever the acceptance is not within 1e-5 of a boundary)."""
    wl = synth.WORKLOADS["batched"]
    n, L, V, d = wl.n, wl.L, wl.V, wl.d
    hidden = synth.hidden_states(n, L, d, seed=wl.seed, kind="int", device=DEV)
    W = synth.lm_head_weights_int(V, d, seed=wl.seed, device=DEV)
    p = synth.canvas_params(wl, step=1)
    rng = np.random.default_rng(wl.seed)
    canvas0 = rng.integers(0, V, (n, L)).astype(np.int32)
    prev0, stable0 = np.full((n, L), -1, np.int32), np.zeros(n, np.int32)
    b, logits, pt = _run(hidden, W, p, V, V, canvas0, prev0, stable0)
    assert dg.dg_get_device_status() == 0
    g = b.host()
    b2 = StepBuffers.make(n, L, DEV, canvas0, prev0, stable0)
    run_step(logits, pt, SEED, b2)
    torch.cuda.synchronize()
    assert dg.dg_get_device_status() == 0
    g2 = b2.host()
    assert np.array_equal(g["argmax"], g2["argmax"])
    assert np.allclose(g["entropy"], g2["entropy"], rtol=2 * H_RTOL, atol=2 * H_ATOL)
    assert np.allclose(g["lse"], g2["lse"], rtol=2 * LSE_RTOL, atol=0)
    compared = 0
    for c in range(n):
        if _near_cut(g2["entropy"][c], float(p["beta"][c]), int(p["min_accept"][c])):
            continue
        compared += 1
        for k in ("accept", "canvas", "sample", "prev", "stable", "n_accept"):
            assert np.array_equal(g[k][c], g2[k][c]), (c, k)
    assert compared >= n - 1
    hb, Wb = synth.bf16_bits(hidden), synth.bf16_bits(W)
    got = synth.bf16_bits(logits)
    for (c, i) in [(0, 0), (1, 77), (3, 128), (5, 255), (7, 3), (7, 200)]:
        ref = oracle.lm_head_logits(hb[c, i:i + 1], Wb)[0]
        assert np.array_equal(got[c, i], ref), (c, i)
        st = oracle.row_stats(ref, float(p["temperature"][c]), SEED, int(p["request_id"][c]),
                              int(p["step"][c]), i, sample=True)
        assert g["argmax"][c, i] == st["argmax"]
        assert abs(g["entropy"][c, i] - st["entropy"]) <= H_RTOL * st["entropy"] + H_ATOL
        assert abs(g["lse"][c, i] - st["lse"]) <= (LSE_RTOL * abs(st["lse"]) + LSE_ATOL)
        if g["accept"][c, i] and g["sample"][c, i] != st["sample"]:
            gap = (st["score1"] - st["score2"]) / max(abs(st["score1"]), 1.0)
            assert gap < BOUNDARY, (c, i)


def test_lm_head_strided_operands_and_bad_rows():
    """Row strides past d (hidden [.., d + 8], W [.., d + 16]); a canvas with T = 0 (status
    DG_DEV_BAD_PARAM, its statistics and decisions left untouched, its logits still written);
    a NaN in one hidden row (status DG_DEV_NAN_INF_ROW).  The other canvas matches the oracle."""
    n, L, V, d = 3, 64, 777, 96
    hb_full = synth.hidden_states(n, L, d + 8, seed=31, kind="int", device=DEV)
    hidden = hb_full[:, :, :d]
    Wf = synth.lm_head_weights_int(V, d + 16, seed=32, device=DEV)
    W = Wf[:, :d]
    rng = np.random.default_rng(33)
    p = _params(n, rng, ("normal", "normal", "normal"))
    p["temperature"][1] = 0.0
    hidden[2, 5, 3] = float("nan")
    canvas0 = rng.integers(0, V, (n, L)).astype(np.int32)
    prev0, stable0 = np.full((n, L), -1, np.int32), np.zeros(n, np.int32)
    b, logits, _ = _run(hidden, W, p, V, 784, canvas0, prev0, stable0)
    st = dg.dg_get_device_status()
    assert st & dg.DG_DEV_BAD_PARAM and st & dg.DG_DEV_NAN_INF_ROW
    g = b.host()
    got = synth.bf16_bits(logits)
    hbits, wbits = synth.bf16_bits(hidden.contiguous()), synth.bf16_bits(W.contiguous())
    for c in (0, 1):
        assert np.array_equal(got[c, :, :V], oracle.lm_head_logits(hbits[c], wbits)), c
    assert np.isnan((got[2, 5, :V].astype(np.uint32) << 16).view(np.float32)).all()
    # the canvas with T = 0: nothing but its logits written
    assert (g["entropy"][1] == -1.0).all() and (g["argmax"][1] == -7).all()
    assert (g["canvas"][1] == canvas0[1]).all() and g["converged"][1] == 7
    ref = np.zeros((1, L, 784), np.uint16)
    ref[0] = oracle.lm_head_logits(hbits[0], wbits, ld=784)
    pc = {k: np.asarray(v)[:1].copy() for k, v in p.items()}
    o = oracle.denoise_step(ref, pc, SEED, canvas0[:1], prev0[:1], stable0[:1], ld=784, V=V)
    rep = compare_step({k: v[:1] for k, v in g.items()}, o, pc, V, SEED, canvas0[:1], prev0[:1], stable0[:1])
    print(rep)
    # the NaN row is flagged; the rest of its canvas keeps finite statistics
    rows = np.arange(L) != 5
    assert np.isfinite(g["entropy"][2][rows]).all()
