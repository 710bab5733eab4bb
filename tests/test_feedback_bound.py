"""CPU checks of the comparison rules themselves (no GPU).

* The feedback bound of helpers.delta_elem_excess: a plain PyTorch fp32 emulation of the
  tensor-core path's precision (bf16 P, bf16 pe, bf16 hidden, bf16 delta; fp32 products and
  sums) meets it against the fp64 oracle, while a result with one wholly wrong component
  per row (zeroed) fails it even though it passes the per-row norm, and so does a chunk of
  components stored one column off.
* The acceptance comparison of helpers.compare_step: a mask that differs from the oracle's
  only at positions on a decision boundary passes, one that differs anywhere else fails,
  and so does an accepted count that moves further than the boundary positions allow.
"""
import numpy as np
import pytest
import torch

from entropy_bounded_denoising_gb300 import synth
import oracle

from helpers import DELTA_RTOL, accept_boundary_positions, compare_step, delta_elem_excess, delta_rel_err


def _bf(t):
    return t.to(torch.bfloat16).float()


def _emulate(rows_bits, T, E, Wg, Wu, Wd):
    """Feedback rows at the tensor-core path's precision: fp32 arithmetic with a bf16
    rounding wherever the path stores bf16 (P in shared memory, pe, the MLP hidden, delta)."""
    x = torch.from_numpy((rows_bits.astype(np.uint32) << 16).view(np.float32))
    k = torch.tensor(1.4426950408889634, dtype=torch.float32) / torch.as_tensor(T, dtype=torch.float32)[:, None]
    lse = torch.logsumexp(x.double() / torch.as_tensor(T, dtype=torch.float64)[:, None], 1).float()
    P = _bf(torch.exp2(x * k - (lse * 1.4426950408889634)[:, None]))
    pe = _bf(P @ E.float())
    g = pe @ Wg.float().T
    u = pe @ Wu.float().T
    hid = _bf(torch.nn.functional.gelu(g, approximate="tanh") * u)
    return _bf(hid @ Wd.float().T).double().numpy(), (pe, g, u)


@pytest.fixture(scope="module", params=["tiny", "single"])
def case(request):
    wl = synth.WORKLOADS[request.param]
    rows = 16
    x = synth.logits(1, wl.L, wl.V, seed=wl.seed, step=1, scale=wl.scale, spike_frac=0.25, dtype="bf16")
    hx = synth.host_logits(x)[0][:rows]
    E, Wg, Wu, Wd = synth.weights(wl.V, wl.d, wl.h, seed=wl.seed)
    bits = tuple(synth.bf16_bits(t) for t in (E, Wg, Wu, Wd))
    T = np.linspace(0.5, 1.5, rows)
    ref = oracle.self_cond_rows(hx, T, *bits)
    emu, parts = _emulate(hx, T, E, Wg, Wu, Wd)
    return ref, emu, parts, (E, Wg, Wu, Wd)


def test_emulated_precision_meets_the_bound(case):
    ref, emu, _, _ = case
    assert delta_rel_err(emu, ref).max() <= DELTA_RTOL
    assert delta_elem_excess(emu, ref).max() <= 0.0
    # and with room: the same result still passes with the floor halved
    rms = np.sqrt(np.mean(ref * ref, axis=1, keepdims=True))
    assert (np.abs(emu - ref) <= DELTA_RTOL * np.abs(ref) + 4 * 2.0 ** -8 * rms).all()


def test_a_zeroed_component_fails_only_the_elementwise_check(case):
    ref, emu, _, _ = case
    d = ref.shape[1]
    rows = ref.shape[0]
    for j in (0, d // 2 + 3, d - 1):   # first and last column tiles, one inside
        bad = emu.copy()
        bad[:, j] = 0.0
        ex = delta_elem_excess(bad, ref)
        assert ex.max() > 0.0, j
        if d >= 1024:
            # one column of d moves a row's norm by about 1/sqrt(d) (2.2 % at d = 2048, 1.6 %
            # at 4096): in most rows the per-row check alone passes the mistake
            old_passes = delta_rel_err(bad, ref) <= DELTA_RTOL
            assert (old_passes & (ex > 0.0)).sum() >= rows // 2, (j, old_passes.sum(), (ex > 0).sum())


def test_a_shifted_column_block_fails_the_elementwise_check(case):
    ref, emu, _, _ = case
    d = ref.shape[1]
    bad = emu.copy()
    bad[:, 32:64] = emu[:, 31:63]          # an epilogue chunk stored one column off
    assert delta_elem_excess(bad, ref).max() > 0.0
    bad = emu.copy()
    bad[:, d - 32:] = emu[:, d - 64:d - 32]    # the last chunk holding the one before it
    assert delta_elem_excess(bad, ref).max() > 0.0


def test_nan_fails_the_elementwise_check(case):
    ref, emu, _, _ = case
    bad = emu.copy()
    bad[3, 5] = np.nan
    assert delta_elem_excess(bad, ref)[3] == np.inf


def _one_canvas(H, beta, g_mask, g_n=None, V=64):
    """Compare a made-up GPU accept mask for one canvas with the oracle's decision on the
    entropies H (the other outputs are made consistent so that only the mask differs)."""
    L = len(H)
    seed, req, step = 5, 3, 1
    o_acc = oracle.accept(np.asarray(H, np.float64), beta, 1)
    p = {"temperature": np.ones(1, np.float32), "beta": np.array([beta], np.float32),
         "tau": np.array([0.0], np.float32), "k": np.ones(1, np.int32), "max_steps": np.full(1, 64, np.int32),
         "min_accept": np.ones(1, np.int32), "step": np.array([step], np.int32),
         "request_id": np.array([req], np.uint32), "flags": np.array([oracle.ACTIVE], np.uint32)}
    g_mask = np.asarray(g_mask, np.uint8)
    tok = np.array([oracle.random_token(seed, req, step, i, oracle.STREAM_RENOISE, V) for i in range(L)], np.int32)
    canvas = np.where(g_mask == 1, 7, tok).astype(np.int32)
    sample = np.where(g_mask == 1, 7, -1).astype(np.int32)
    zeros = np.zeros((1, L), np.int32)
    g = {"canvas": canvas[None], "prev": zeros, "stable": np.zeros(1, np.int32), "accept": g_mask[None],
         "argmax": zeros, "sample": sample[None], "entropy": np.asarray(H, np.float32)[None],
         "lse": np.ones((1, L), np.float32), "converged": np.zeros(1, np.uint8),
         "mean_entropy": np.array([np.mean(H)], np.float32),
         "n_accept": np.array([int(g_mask.sum()) if g_n is None else g_n], np.int32)}
    o = {"accept_mask": o_acc["mask"][None], "argmax": zeros, "sample": sample[None],
         "entropy": np.asarray(H, np.float64)[None], "lse": np.ones((1, L)), "converged": np.zeros(1, np.uint8),
         "mean_entropy": np.array([np.mean(H)]), "n_accept": np.array([o_acc["n_accept"]], np.int32),
         "sample_gap": np.full((1, L), np.inf), "cut_gap": np.array([o_acc["cut_gap"]]),
         "budget_gap": np.array([o_acc["budget_gap"]]), "tau_gap": np.array([np.inf]),
         "stable_count": np.zeros(1, np.int32)}
    return compare_step(g, o, p, V, seed, zeros, np.full((1, L), -1, np.int32), np.zeros(1, np.int32))


def test_acceptance_mismatch_only_at_boundary_positions():
    # positions 1 and 4 have entropies 1e-7 apart (relative) across the cut of beta = 2.5
    H = [0.5, 1.0, 0.25, 3.0, 1.0 + 1e-7, 2.0]
    o = oracle.accept(np.asarray(H, np.float64), 2.5, 1)
    assert list(np.nonzero(o["mask"])[0]) == [0, 1, 2]
    near = accept_boundary_positions(np.asarray(H), 2.5, o["n_accept"])
    assert list(np.nonzero(near)[0]) == [1, 4]
    rep = _one_canvas(H, 2.5, [1, 0, 1, 0, 1, 0])         # the two near-equal entropies swapped
    assert rep.accept_mismatch == 2 and rep.accept_boundary_positions == 2
    with pytest.raises(AssertionError):                   # a swap away from the cut
        _one_canvas(H, 2.5, [0, 1, 1, 0, 0, 1])
    with pytest.raises(AssertionError):                   # a count that moves too far
        _one_canvas(H, 2.5, [1, 0, 1, 0, 1, 0], g_n=6)


def test_acceptance_budget_boundary():
    # the running sum reaches beta within 1e-7 relative at the third position
    H = [0.25, 0.5, 1.25 + 2e-7, 2.0]
    o = oracle.accept(np.asarray(H, np.float64), 2.0, 1)
    assert o["n_accept"] == 2
    near = accept_boundary_positions(np.asarray(H), 2.0, o["n_accept"])
    assert list(np.nonzero(near)[0]) == [2]
    rep = _one_canvas(H, 2.0, [1, 1, 1, 0])               # one more accepted at the budget
    assert rep.accept_mismatch == 1
    with pytest.raises(AssertionError):                   # one fewer, at a position off the boundary
        _one_canvas(H, 2.0, [1, 0, 0, 0])
