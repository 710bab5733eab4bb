"""Pins of the oracle's attention with per-sequence causality and a symmetric window (CPU).

The mask rule against hand-written allowed sets for the pages' three-request example (a
causal prefill of 6, a denoising canvas of 4 after 6 context tokens, a causal commit pass of
the same shape), with no window and with W = 2; closed forms (zero queries give the mean of
the allowed values and lse = log of their count; a window of 0 on a causal request leaves
only the query's own key); invariants: permuting the keys of a bidirectional request changes
nothing, the output is linear in V, and grouped key/value heads equal repeating them per
query head (so a wrong head mapping fails)."""
import math

import numpy as np
import torch

import oracle


def _bits(x):
    t = torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _val(b):
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# The pages' figure: request 0 prefills 6 tokens (causal), request 1 denoises a canvas of 4
# after 6 context tokens (bidirectional), request 2 commits that canvas (causal again).
REQ = [(6, 6, True), (4, 10, False), (4, 10, True)]   # (q_len, kv_len, causal)


def _allowed_table(window):
    out = []
    for q_len, kv_len, causal in REQ:
        rows = []
        for i in range(q_len):
            pos = kv_len - q_len + i
            rows.append([j for j in range(kv_len) if oracle.attn_allowed(causal, window, pos, j, kv_len)])
        out.append(rows)
    return out


def test_mask_matches_the_pages_example():
    full = _allowed_table(-1)
    assert full[0] == [list(range(i + 1)) for i in range(6)]               # causal prefill
    assert full[1] == [list(range(10))] * 4                                 # canvas sees all
    assert full[2] == [list(range(7 + i)) for i in range(4)]               # causal commit
    w2 = _allowed_table(2)
    assert w2[0] == [[0], [0, 1], [0, 1, 2], [1, 2, 3], [2, 3, 4], [3, 4, 5]]
    assert w2[1] == [[4, 5, 6, 7, 8], [5, 6, 7, 8, 9], [6, 7, 8, 9], [7, 8, 9]]   # symmetric
    assert w2[2] == [[4, 5, 6], [5, 6, 7], [6, 7, 8], [7, 8, 9]]
    assert not oracle.attn_allowed(False, -1, 3, 10, 10)                    # past the sequence


def _batch(rng, D=8, Hq=2, Hkv=1):
    cu_q = np.cumsum([0] + [r[0] for r in REQ]).astype(np.int32)
    cu_kv = np.cumsum([0] + [r[1] for r in REQ]).astype(np.int32)
    causal = np.array([r[2] for r in REQ], np.uint8)
    q = _bits(rng.normal(0, 1, (cu_q[-1], Hq, D)))
    k = _bits(rng.normal(0, 1, (cu_kv[-1], Hkv, D)))
    v = _bits(rng.normal(0, 1, (cu_kv[-1], Hkv, D)))
    return q, k, v, cu_q, cu_kv, causal


def test_zero_queries_average_the_allowed_values():
    rng = np.random.default_rng(1)
    q, k, v, cu_q, cu_kv, causal = _batch(rng)
    q[:] = 0
    for window in (-1, 2):
        o, lse = oracle.attention(q, k, v, cu_q, cu_kv, causal, window=window)
        table = _allowed_table(window)
        for s, (q_len, kv_len, _) in enumerate(REQ):
            for i in range(q_len):
                keys = table[s][i]
                want = _val(v[cu_kv[s] + np.array(keys), 0]).mean(axis=0)
                for h in range(2):
                    assert np.allclose(o[cu_q[s] + i, h], want, rtol=1e-14, atol=1e-15)
                    assert abs(lse[cu_q[s] + i, h] - math.log(len(keys))) < 1e-14


def test_window_zero_on_a_causal_request_keeps_only_the_own_key():
    rng = np.random.default_rng(2)
    q, k, v, cu_q, cu_kv, causal = _batch(rng)
    o, lse = oracle.attention(q, k, v, cu_q, cu_kv, causal, window=0, scale=0.5)
    for s in (0, 2):
        q_len, kv_len, _ = REQ[s]
        for i in range(q_len):
            j = cu_kv[s] + kv_len - q_len + i
            for h in range(2):
                assert np.array_equal(o[cu_q[s] + i, h], _val(v[j, 0]))
                dot = float(np.dot(_val(q[cu_q[s] + i, h]), _val(k[j, 0])))
                assert abs(lse[cu_q[s] + i, h] - 0.5 * dot) <= 1e-12 * max(1.0, abs(dot))


def test_permuting_the_keys_of_a_bidirectional_request():
    rng = np.random.default_rng(3)
    q, k, v, cu_q, cu_kv, causal = _batch(rng)
    o, lse = oracle.attention(q, k, v, cu_q, cu_kv, causal)
    perm = rng.permutation(10) + cu_kv[1]
    k2, v2 = k.copy(), v.copy()
    k2[cu_kv[1]:cu_kv[2]] = k[perm]
    v2[cu_kv[1]:cu_kv[2]] = v[perm]
    o2, lse2 = oracle.attention(q, k2, v2, cu_q, cu_kv, causal)
    sl = slice(cu_q[1], cu_q[2])
    assert np.allclose(o2[sl], o[sl], rtol=1e-13, atol=1e-14)
    assert np.allclose(lse2[sl], lse[sl], rtol=1e-13, atol=1e-14)
    # the causal requests see different keys after the permutation only if theirs moved
    assert np.array_equal(o2[:cu_q[1]], o[:cu_q[1]])


def test_output_is_linear_in_v():
    rng = np.random.default_rng(4)
    q, k, v, cu_q, cu_kv, causal = _batch(rng)
    va = _bits(rng.integers(-8, 9, v.shape))
    vb = _bits(rng.integers(-8, 9, v.shape))
    vs = _bits(_val(va) + _val(vb))                 # small integers: the sum is exact in bf16
    oa, _ = oracle.attention(q, k, va, cu_q, cu_kv, causal, window=2)
    ob, _ = oracle.attention(q, k, vb, cu_q, cu_kv, causal, window=2)
    os_, _ = oracle.attention(q, k, vs, cu_q, cu_kv, causal, window=2)
    assert np.allclose(os_, oa + ob, rtol=1e-12, atol=1e-12)


def test_grouped_heads_equal_repeated_heads():
    rng = np.random.default_rng(5)
    q, k, v, cu_q, cu_kv, causal = _batch(rng, Hq=4, Hkv=2)
    o, lse = oracle.attention(q, k, v, cu_q, cu_kv, causal)
    k_rep = np.repeat(k, 2, axis=1)                 # query heads 0, 1 -> kv head 0; 2, 3 -> 1
    v_rep = np.repeat(v, 2, axis=1)
    o2, lse2 = oracle.attention(q, k_rep, v_rep, cu_q, cu_kv, causal)
    assert np.array_equal(o, o2) and np.array_equal(lse, lse2)
    k_bad = np.tile(k, (1, 2, 1))                   # the other mapping (h % Hkv) differs
    o3, _ = oracle.attention(q, k_bad, np.tile(v, (1, 2, 1)), cu_q, cu_kv, causal)
    assert not np.allclose(o3, o)
