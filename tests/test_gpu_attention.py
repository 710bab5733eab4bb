"""GPU parity of the attention with per-sequence causality and a symmetric sliding window
(dg_attention) against the fp64 oracle.

A mixed batch like the pages' example — causal prefills, denoising canvases after a context
(bidirectional), a causal commit pass — with short and long sequences, ragged tails and
grouped key/value heads, with no window and with windows of 0, 1 and 200.  Tolerance, derived
from the arithmetic: every softmax weight goes to the P V product rounded to bf16 (relative
2^-9) while the row sum keeps the unrounded weights, and the output is rounded to bf16, so
|o - ref| <= 2^-9 max|v| + 2^-8 |ref| elementwise, tested with a factor 2 margin; lse from fp32
scores (128-term sums of exact bf16 products) and ex2.approx within 1e-4 + 1e-5 |lse|.  With a
window of 0 a causal query sees only its own key, so its output is that value row bit for bit."""
import numpy as np
import pytest
import torch

import entropy_bounded_denoising_gb300 as dg
from entropy_bounded_denoising_gb300 import synth
import oracle

pytestmark = pytest.mark.gpu
DEV = "cuda"
D = 128

# (q_len, kv_len, causal): prefill, canvas after context, commit, tiny ones, ragged tails
SEQS = [(300, 300, 1), (256, 1256, 0), (256, 1256, 1), (5, 5, 1), (17, 40, 0), (128, 128, 0), (1, 1, 0)]


def _batch(seqs, Hq, Hkv, seed, d=D):
    cu_q = np.cumsum([0] + [s[0] for s in seqs]).astype(np.int32)
    cu_kv = np.cumsum([0] + [s[1] for s in seqs]).astype(np.int32)
    causal = np.array([s[2] for s in seqs], np.uint8)
    q, k, v = synth.attention_inputs(int(cu_q[-1]), int(cu_kv[-1]), Hq, Hkv, d, seed=seed, device=DEV)
    return q, k, v, cu_q, cu_kv, causal


def _run(q, k, v, cu_q, cu_kv, causal, window, max_q=None):
    o = torch.full(q.shape, float("nan"), dtype=torch.bfloat16, device=DEV)
    lse = torch.full(q.shape[:2], float("nan"), dtype=torch.float32, device=DEV)
    t = lambda a: torch.from_numpy(a).to(DEV)
    dg.dg_clear_device_status()
    dg.dg_attention(q, k, v, o, t(cu_q), t(cu_kv), t(causal),
                    int(np.diff(cu_q).max()) if max_q is None else max_q, lse=lse, window=window)
    torch.cuda.synchronize()
    return o, lse


def _check(o, lse, q, k, v, cu_q, cu_kv, causal, window):
    ref_o, ref_lse = oracle.attention(synth.bf16_bits(q), synth.bf16_bits(k), synth.bf16_bits(v), cu_q, cu_kv,
                                      causal, window=window)
    got = o.float().cpu().numpy().astype(np.float64)
    vmax = np.abs(v.float().cpu().numpy()).max()
    err = np.abs(got - ref_o)
    bound = 2 * (2.0 ** -9 * vmax + 2.0 ** -8 * np.abs(ref_o))
    assert np.isfinite(got).all()
    bad = np.argwhere(err > bound)
    assert bad.size == 0, (bad[:5], err.max())
    gl = lse.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(gl - ref_lse) <= 1e-4 + 1e-5 * np.abs(ref_lse)), np.abs(gl - ref_lse).max()
    return float((err / (np.abs(ref_o) + vmax)).max())


@pytest.mark.parametrize("window", [-1, 200, 1])
@pytest.mark.parametrize("Hq,Hkv", [(4, 2), (2, 2)])
def test_attention_mixed_batch(window, Hq, Hkv):
    q, k, v, cu_q, cu_kv, causal = _batch(SEQS, Hq, Hkv, seed=window + 10 * Hq + Hkv)
    o, lse = _run(q, k, v, cu_q, cu_kv, causal, window)
    assert dg.dg_get_device_status() == 0
    print(f"max scaled error {_check(o, lse, q, k, v, cu_q, cu_kv, causal, window):.2e}")


def test_attention_window_zero_returns_the_own_value_row():
    q, k, v, cu_q, cu_kv, causal = _batch(SEQS, 4, 2, seed=3)
    o, lse = _run(q, k, v, cu_q, cu_kv, causal, 0)
    assert dg.dg_get_device_status() == 0
    _check(o, lse, q, k, v, cu_q, cu_kv, causal, 0)
    ob, vb = synth.bf16_bits(o), synth.bf16_bits(v)
    for s, (ql, kl, cz) in enumerate(SEQS):
        for i in range(ql):
            j = cu_kv[s] + kl - ql + i
            for h in range(4):
                if cz:
                    assert np.array_equal(ob[cu_q[s] + i, h], vb[j, h // 2]), (s, i, h)


def test_attention_bad_sequences_raise_status():
    """A sequence with more queries than keys is skipped with DG_DEV_BAD_PARAM; so is a
    max_q_len below a sequence's query count (its later tiles are not computed)."""
    seqs = [(64, 200, 1), (50, 20, 0), (40, 40, 0)]
    q, k, v, cu_q, cu_kv, causal = _batch(seqs, 2, 1, seed=4)
    o, lse = _run(q, k, v, cu_q, cu_kv, causal, -1)
    assert dg.dg_get_device_status() & dg.DG_DEV_BAD_PARAM
    assert torch.isnan(o[cu_q[1]:cu_q[2]].float()).all()
    keep = np.r_[0:cu_q[1], cu_q[2]:cu_q[3]]
    ref_o, _ = oracle.attention(synth.bf16_bits(q), synth.bf16_bits(k), synth.bf16_bits(v), cu_q, cu_kv, causal)
    got = o.float().cpu().numpy()
    vmax = np.abs(v.float().cpu().numpy()).max()
    assert np.all(np.abs(got[keep] - ref_o[keep]) <= 2 * (2.0 ** -9 * vmax + 2.0 ** -8 * np.abs(ref_o[keep])))
    seqs = [(300, 300, 1)]
    q, k, v, cu_q, cu_kv, causal = _batch(seqs, 2, 1, seed=5)
    o, _ = _run(q, k, v, cu_q, cu_kv, causal, -1, max_q=200)
    assert dg.dg_get_device_status() & dg.DG_DEV_BAD_PARAM
    assert torch.isnan(o[256:].float()).all() and not torch.isnan(o[:256].float()).any()
    dg.dg_clear_device_status()


def test_attention_denoising_batch_sampled():
    """The timed shape: 8 canvases of 256 after 2048 context tokens (bidirectional) and 4
    causal prefills of 1024, 16 query heads over 8 key/value heads, with a window of 512 and
    without; sampled query rows against the oracle."""
    seqs = [(256, 2304, 0)] * 8 + [(1024, 1024, 1)] * 4
    q, k, v, cu_q, cu_kv, causal = _batch(seqs, 16, 8, seed=6)
    for window in (-1, 512):
        o, lse = _run(q, k, v, cu_q, cu_kv, causal, window)
        assert dg.dg_get_device_status() == 0
        rng = np.random.default_rng(window + 7)
        pick = [(s, int(rng.integers(0, seqs[s][0]))) for s in rng.choice(len(seqs), 8, replace=False)]
        qb, kb, vb = synth.bf16_bits(q), synth.bf16_bits(k), synth.bf16_bits(v)
        for s, i in pick:
            ql, kl, cz = seqs[s]
            # the sampled query alone, with its whole key range, as a one-query sequence
            qi = qb[cu_q[s] + i:cu_q[s] + i + 1]
            kk, vv = kb[cu_kv[s]:cu_kv[s + 1]], vb[cu_kv[s]:cu_kv[s + 1]]
            # a one-query sequence puts the query at kv_len - 1: cut the keys after its position
            # for a causal sequence, or rebuild its position by a window-exact key range
            pos = kl - ql + i
            ref_o, ref_lse = _one_query(qi, kk, vv, pos, cz, window)
            got = o[cu_q[s] + i].float().cpu().numpy()
            vmax = float(np.abs((vv.astype(np.uint32) << 16).view(np.float32)).max())
            assert np.all(np.abs(got - ref_o) <= 2 * (2.0 ** -9 * vmax + 2.0 ** -8 * np.abs(ref_o))), (s, i, window)
            assert np.allclose(lse[cu_q[s] + i].cpu().numpy(), ref_lse, rtol=1e-5, atol=1e-4), (s, i)


def _one_query(qi, kk, vv, pos, causal, window):
    """Oracle for one query at position `pos` of a sequence with keys kk / vv: the allowed
    keys are gathered into a bidirectional one-query sequence (no further masking)."""
    kl = kk.shape[0]
    keys = [j for j in range(kl) if oracle.attn_allowed(bool(causal), window, pos, j, kl)]
    o, lse = oracle.attention(qi, kk[keys], vv[keys], np.array([0, 1], np.int32),
                              np.array([0, len(keys)], np.int32), np.array([0], np.uint8))
    return o[0], lse[0]


def test_attention_window_wider_than_every_sequence_is_no_window():
    """A window at least as long as every sequence allows what no window allows: the outputs
    are bit-identical (the range arithmetic is 64-bit, so a window near 2^31 cannot wrap)."""
    q, k, v, cu_q, cu_kv, causal = _batch(SEQS, 4, 2, seed=8)
    o1, l1 = _run(q, k, v, cu_q, cu_kv, causal, -1)
    o2, l2 = _run(q, k, v, cu_q, cu_kv, causal, 2 ** 31 - 1)
    assert dg.dg_get_device_status() == 0
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16)) and torch.equal(l1, l2)


@pytest.mark.parametrize("d", [64, 256])
@pytest.mark.parametrize("window", [-1, 200])
def test_attention_other_head_dimensions(d, window):
    """Head dimensions 64 (two CTAs per SM, 192 TMEM columns) and 256 (one CTA per SM, 384)."""
    q, k, v, cu_q, cu_kv, causal = _batch(SEQS, 4, 2, seed=d + window, d=d)
    o, lse = _run(q, k, v, cu_q, cu_kv, causal, window)
    assert dg.dg_get_device_status() == 0
    print(f"D={d}: max scaled error {_check(o, lse, q, k, v, cu_q, cu_kv, causal, window):.2e}")
    if window == -1:   # a window of 0 on the causal sequences: the own value row, bit for bit
        o0, _ = _run(q, k, v, cu_q, cu_kv, causal, 0)
        ob, vb = synth.bf16_bits(o0), synth.bf16_bits(v)
        for s_, (ql, kl, cz) in enumerate(SEQS):
            if cz:
                j = cu_kv[s_] + kl - ql + np.arange(ql)
                for h in range(4):
                    assert np.array_equal(ob[cu_q[s_]:cu_q[s_] + ql, h], vb[j, h // 2]), (s_, h)


@pytest.mark.parametrize("seqs", [[(256, 256, 0)] * 64, [(256, 2304, 0)] * 8 + [(1024, 1024, 1)] * 4],
                         ids=["short_items", "denoising_batch"])
def test_attention_repeated_calls_are_bit_identical(seqs):
    """Repeated calls on the same inputs give the same bits.  Many short items per CTA put the
    softmax warps at different tiles at once; this caught a P barrier shared by both P buffers,
    which a warp a tile ahead could complete for a tile whose P another warp was still
    writing (one warp's rows of one item wrong in a few percent of calls).  Items of one cost
    (the first case) are taken round robin, items of several costs (the second) from the
    counter, whose order differs from call to call."""
    q, k, v, cu_q, cu_kv, causal = _batch(seqs, 16, 8, seed=12)
    o0, l0 = _run(q, k, v, cu_q, cu_kv, causal, -1)
    assert dg.dg_get_device_status() == 0
    _check_rows = np.random.default_rng(3).choice(q.shape[0], 16, replace=False)
    for rep in range(24):
        o, lse = _run(q, k, v, cu_q, cu_kv, causal, -1)
        assert dg.dg_get_device_status() == 0
        assert torch.equal(o.view(torch.int16), o0.view(torch.int16)), rep
        assert torch.equal(lse, l0), rep
    # and the first call is right: sampled rows against the oracle
    qb, kb, vb = synth.bf16_bits(q), synth.bf16_bits(k), synth.bf16_bits(v)
    for qi in _check_rows:
        s = int(np.searchsorted(cu_q, qi, side="right") - 1)
        ql, kl, cz = seqs[s]
        i = int(qi - cu_q[s])
        ref_o, _ = _one_query(qb[qi:qi + 1], kb[cu_kv[s]:cu_kv[s + 1]], vb[cu_kv[s]:cu_kv[s + 1]], kl - ql + i, cz, -1)
        got = o0[qi].float().cpu().numpy()
        vmax = float(np.abs((vb[cu_kv[s]:cu_kv[s + 1]].astype(np.uint32) << 16).view(np.float32)).max())
        assert np.all(np.abs(got - ref_o) <= 2 * (2.0 ** -9 * vmax + 2.0 ** -8 * np.abs(ref_o))), (s, i)
