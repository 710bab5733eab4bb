"""The benchmark's own accounting (CPU): the attention counts behind its TFLOP/s figures
against brute force over the oracle's mask rule, and the step arithmetic of the two step
forms (from logits, from hidden states)."""
import numpy as np
import pytest

import bench
import oracle
from entropy_bounded_denoising_gb300 import synth


def _brute(seqs, W, TQ, TK):
    pairs = tiles = 0
    for ql, kl, c in seqs:
        ok = np.array([[oracle.attn_allowed(bool(c), W, kl - ql + i, j, kl) for j in range(kl)]
                       for i in range(ql)])
        pairs += int(ok.sum())
        for t0 in range(0, ql, TQ):
            blk = ok[t0:t0 + TQ]
            hit = [jt for jt in range(0, kl, TK) if blk[:, jt:jt + TK].any()]
            # the kernel visits the range of tiles from the first to the last that holds a key
            tiles += (hit[-1] - hit[0]) // TK + 1 if hit else 0
    return pairs, tiles


@pytest.mark.parametrize("W", [-1, 0, 5, 40])
def test_attention_counts_match_brute_force(W):
    seqs = [(20, 20, 1), (7, 30, 0), (16, 50, 1), (1, 1, 0), (33, 33, 0)]
    pairs, tiles, tiles_all = bench.attention_counts(seqs, W, TQ=8, TK=4)
    assert (pairs, tiles) == _brute(seqs, W, 8, 4)
    assert tiles_all == sum(-(-kl // 4) * -(-ql // 8) for ql, kl, _ in seqs)


def test_step_arithmetic_from_logits_and_from_hidden():
    wl = synth.WORKLOADS["batched"]
    N = wl.n * wl.L
    a = bench._workload_arith(wl, N, N)
    b = bench._workload_arith(wl, N, N, from_hidden=True)
    assert a["tc_flops"] == 2.0 * N * wl.V * wl.d + 6.0 * N * wl.d * wl.h
    assert b["tc_flops"] == a["tc_flops"] + 2.0 * N * wl.V * wl.d      # the LM head
    # from hidden states the step reads the hidden rows instead of the logits
    assert a["bytes"] - b["bytes"] == 2 * N * wl.V - 2 * N * wl.d


def test_peak_follows_the_timed_window():
    pk = {"bf16_tflops": 1891.2, "bf16_tflops_sustained": 1692.7, "hbm_gbs": 6788.6}
    # a 67 ms window at full clock (the round-end bench line): the burst figure
    assert bench.choose_tc_peak(pk, 0.067, 2070.0, 2070.0) == (1891.2, "burst")
    # a short window is a burst whatever the sampled clock
    assert bench.choose_tc_peak(pk, 0.5, 1600.0, 2070.0) == (1891.2, "burst")
    # seconds under the power cap: the sustained figure
    assert bench.choose_tc_peak(pk, 1.1, 1680.0, 2070.0) == (1692.7, "sustained")
    # seconds at full clock (within 3 %): still the burst figure
    assert bench.choose_tc_peak(pk, 3.0, 2020.0, 2070.0) == (1891.2, "burst")
    assert bench.choose_tc_peak(pk, 3.0, None, None) == (1692.7, "sustained")
