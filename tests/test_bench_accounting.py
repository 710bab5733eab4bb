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
