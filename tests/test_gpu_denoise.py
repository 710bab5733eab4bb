"""GPU parity of the denoise step (K1 statistics + sample, K2 acceptance / renoise /
convergence) against the fp64 oracle, through the C ABI.

Bars: argmax, renoise tokens, prev_argmax and stable counts bit-exact; samples, accept
masks, canvases and convergence bit-exact except positions within 1e-6 relative of a
decision boundary (counted); entropy within 1e-5 relative (+1e-12), lse within 1e-6."""
import numpy as np
import pytest
import torch

import entropy_bounded_denoising_gb300 as dg
from entropy_bounded_denoising_gb300 import synth
import oracle

from helpers import StepBuffers, compare_step, run_step

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _params(n, rng, **kw):
    p = {"temperature": rng.uniform(0.4, 1.6, n).astype(np.float32),
         "beta": rng.uniform(1.0, 40.0, n).astype(np.float32),
         "tau": np.full(n, 0.3, np.float32), "k": rng.integers(1, 4, n).astype(np.int32),
         "max_steps": np.full(n, 64, np.int32), "min_accept": np.ones(n, np.int32),
         "step": rng.integers(0, 5, n).astype(np.int32),
         "request_id": rng.integers(0, 1 << 31, n).astype(np.uint32),
         "flags": np.full(n, dg.DG_ACTIVE, np.uint32)}
    for k, v in kw.items():
        p[k] = np.broadcast_to(np.asarray(v, p[k].dtype), (n,)).copy()
    return p


def _check_case(x, p, seed, V, canvas0=None, prev0=None, stable0=None):
    n, L, ld = x.shape
    canvas0 = np.zeros((n, L), np.int32) if canvas0 is None else canvas0
    prev0 = np.full((n, L), -1, np.int32) if prev0 is None else prev0
    stable0 = np.zeros(n, np.int32) if stable0 is None else stable0
    b = StepBuffers.make(n, L, DEV, canvas0, prev0, stable0)
    dg.dg_clear_device_status()
    run_step(x.to(DEV), dg.params_tensor(p, DEV), seed, b, V=V)
    torch.cuda.synchronize()
    assert dg.dg_get_device_status() == 0
    g = b.host()
    o = oracle.denoise_step(synth.host_logits(x), p, seed, canvas0, prev0, stable0, ld=ld, V=V)
    rep = compare_step(g, o, p, V, seed, canvas0, prev0, stable0)
    print(rep)
    return g, o, rep


@pytest.mark.parametrize("sample_all", [False, True])
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("V,ld", [(5003, 5008), (1024, 1024), (40000, 40000), (70001, 70008)])
def test_step_small_ragged(dtype, V, ld, sample_all):
    """Canvases 0 and 3 draw their samples in opposite ways (every position / accepted
    positions only, after the acceptance); canvas 1 is read-only, canvas 2 inactive."""
    rng = np.random.default_rng(V + (dtype == "fp32"))
    n, L = 4, 200
    x = synth.logits(n, L, V, seed=V, step=1, scale=(0.5, 12.0), spike_frac=0.1, dtype=dtype, ld=ld)
    p = _params(n, rng)
    p["flags"][1] = dg.DG_ACTIVE | dg.DG_READ_ONLY
    p["max_steps"][1] = 1
    p["flags"][2] = 0
    p["flags"][0 if sample_all else 3] |= dg.DG_SAMPLE_ALL
    g, o, _ = _check_case(x, p, 0xDEADBEEF12345, V, canvas0=rng.integers(0, V, (n, L)).astype(np.int32))
    deferred = 3 if sample_all else 0
    assert (g["sample"][deferred][g["accept"][deferred] == 0] == -1).all()
    assert g["accept"][deferred].any()


def test_step_convergence_sequence():
    """A canvas whose logits stop changing converges after k stable steps when its mean
    entropy is below tau (sharp rows), and keeps going otherwise."""
    rng = np.random.default_rng(3)
    n, L, V = 2, 64, 2048
    x = synth.logits(n, L, V, seed=5, step=6, scale=(6.0, 12.0), spike_frac=1.0)
    p = _params(n, rng, k=2, max_steps=64, temperature=1.0)
    p["tau"][:] = [5.0, 1e-9]
    canvas = np.zeros((n, L), np.int32)
    prev = np.full((n, L), -1, np.int32)
    stable = np.zeros(n, np.int32)
    convs = []
    for step in range(3):
        p["step"][:] = step
        g, o, _ = _check_case(x, p, 99, V, canvas, prev, stable)
        canvas, prev, stable = g["canvas"], g["prev"], g["stable"]
        convs.append(list(g["converged"]))
    assert [c[0] for c in convs] == [0, 0, 1]
    assert [c[1] for c in convs] == [0, 0, 0]


def test_accept_hook_golden_and_brute_force():
    """dg_accept_from_entropy on the hand-worked entropy-only cases and on random dyadic
    entropies (exact sums), against the oracle's literal sort-and-scan."""
    import json, os
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "acceptance_4x8.json")))
    cases = [(np.array(c["H"]), c["beta"], c["min_accept"]) for c in g["entropy_only_cases"]]
    rng = np.random.default_rng(4)
    for _ in range(40):
        L = int(rng.integers(1, 300))
        H = rng.integers(0, 64, L) / 16.0
        cases.append((H, float(rng.integers(-2, 300)) / 16.0 + 1.0 / 32, int(rng.integers(0, 2))))
        cases.append((H, float(rng.integers(0, 300)) / 16.0, 1))   # equality cases
    for H, beta, mina in cases:
        L = H.size
        V = 1000
        n = 1
        p = _params(n, rng, beta=beta, min_accept=mina)
        ent = torch.tensor(H, dtype=torch.float32, device=DEV).reshape(1, L)
        smp = torch.arange(L, dtype=torch.int32, device=DEV).reshape(1, L)
        am = torch.zeros((1, L), dtype=torch.int32, device=DEV)
        b = StepBuffers.make(n, L, DEV)
        dg.dg_accept_from_entropy(ent, smp, am, n, L, V, dg.params_tensor(p, DEV), 5, b.canvas, b.prev,
                                  b.stable, b.accept, b.converged, b.mean_entropy, b.n_accept)
        torch.cuda.synchronize()
        r = oracle.accept(H.astype(np.float32).astype(np.float64), beta, mina)
        assert (b.accept.cpu().numpy()[0] == r["mask"]).all(), (H, beta, mina)
        assert int(b.n_accept.cpu()[0]) == r["n_accept"]


def test_canvas_init_matches_oracle():
    rng = np.random.default_rng(6)
    n, L, V = 5, 256, 152064
    p = _params(n, rng)
    p["flags"][3] = 0
    canvas = torch.full((n, L), -5, dtype=torch.int32, device=DEV)
    dg.dg_canvas_init(canvas, n, L, V, dg.params_tensor(p, DEV), 0xABCDEF)
    ref = oracle.canvas_init(n, L, V, p, 0xABCDEF)
    got = canvas.cpu().numpy()
    assert (got[[0, 1, 2, 4]] == ref[[0, 1, 2, 4]]).all()
    assert (got[3] == -5).all()


def test_philox_words_match_oracle():
    n_blocks = 20000
    out = torch.zeros((n_blocks, 4), dtype=torch.int32, device=DEV)
    seed = 0x0123456789ABCDEF
    dg.dg_philox_words(seed, 77, 5, 13, 1, 1000, n_blocks, out)
    got = out.cpu().numpy().view(np.uint32)
    for b in range(0, n_blocks, 97):
        ctr = [1000 + b, 13, 5, 1 | (((seed >> 32) & 0xFFFFFF) << 8)]
        ref = oracle.philox4x32(ctr, [seed & 0xFFFFFFFF, 77])
        assert (got[b] == ref).all(), b


def test_advance_params():
    rng = np.random.default_rng(7)
    n = 6
    p = _params(n, rng)
    p["flags"][5] = 0
    pt = dg.params_tensor(p, DEV)
    conv = torch.tensor([1, 0, 1, 0, 0, 1], dtype=torch.uint8, device=DEV)
    dg.dg_advance_params(pt, conv, n)
    q = dg.unpack_params(pt)
    for c in range(n):
        if c == 5:
            assert q["flags"][c] == 0 and q["step"][c] == p["step"][c]
        elif conv[c]:
            assert not (q["flags"][c] & dg.DG_ACTIVE) and q["step"][c] == p["step"][c]
        else:
            assert q["flags"][c] & dg.DG_ACTIVE and q["step"][c] == p["step"][c] + 1


def test_batch_composition_does_not_change_rows():
    """A canvas gives bit-identical outputs alone and inside a larger, reordered batch."""
    rng = np.random.default_rng(8)
    n, L, V = 4, 128, 65536
    x = synth.logits(n, L, V, seed=8, step=2, scale=(0.5, 12.0))
    p = _params(n, rng)
    outs = []
    for order in ([0, 1, 2, 3], [3, 1, 0, 2]):
        xs = x[order].contiguous()
        ps = {k: v[order] for k, v in p.items()}
        b = StepBuffers.make(n, L, DEV)
        run_step(xs.to(DEV), dg.params_tensor(ps, DEV), 11, b)
        h = b.host()
        inv = np.argsort(order)
        outs.append({k: v[inv] for k, v in h.items()})
    solo = StepBuffers.make(1, L, DEV)
    run_step(x[2:3].contiguous().to(DEV), dg.params_tensor({k: v[2:3] for k, v in p.items()}, DEV), 11, solo)
    s = solo.host()
    for k in ("entropy", "lse", "argmax", "sample", "accept", "canvas", "converged"):
        assert np.array_equal(outs[0][k], outs[1][k]), k
        assert np.array_equal(outs[0][k][2], s[k][0]), k


@pytest.mark.parametrize("sample_all", [False, True])
@pytest.mark.parametrize("pieces", [1, 2, 3, 4, 5, 8, 9])
def test_step_rows_of_many_pieces_with_ragged_ends(pieces, sample_all):
    """Rows of 1-9 16 KB pieces streamed through one CTA's ring.  V = 8192 k - 3 puts a
    ragged end in the last piece; spiked rows put the maximum in any piece.  Against the
    oracle, and with NaN / +inf logits near the row's two ends and an all -inf row (their
    status bits raised, the valid row's argmax and sample still the oracle's)."""
    rng = np.random.default_rng(pieces * 10 + sample_all)
    V = 8192 * pieces - 3
    ld = V + 3  # rows 16-byte aligned
    n, L = 3, 96
    x = synth.logits(n, L, V, seed=pieces, step=1, scale=(0.5, 12.0), spike_frac=0.3, ld=ld)
    p = _params(n, rng)
    if sample_all:
        p["flags"] |= dg.DG_SAMPLE_ALL
    _check_case(x, p, 0x5EED + pieces, V, canvas0=rng.integers(0, V, (n, L)).astype(np.int32))
    # flagged rows: a NaN near the row's end, +inf near its start, a row of -inf
    y = synth.logits(1, 4, V, seed=pieces + 1, step=0, scale=(1.0, 2.0), ld=ld).float()
    y[0, 1, V - 2] = float("nan")
    y[0, 2, 3] = float("inf")
    y[0, 3, :] = float("-inf")
    q = _params(1, rng, temperature=1.0, flags=dg.DG_ACTIVE | dg.DG_SAMPLE_ALL)
    b = StepBuffers.make(1, 4, DEV)
    dg.dg_clear_device_status()
    run_step(y.to(torch.bfloat16).to(DEV), dg.params_tensor(q, DEV), 3, b, V=V)
    st = dg.dg_get_device_status()
    assert st & dg.DG_DEV_NAN_INF_ROW and st & dg.DG_DEV_EMPTY_ROW and not st & dg.DG_DEV_TIMEOUT
    dg.dg_clear_device_status()
    o = oracle.row_stats(synth.host_logits(y.to(torch.bfloat16))[0, 0, :V], T=1.0, seed=3,
                         request_id=int(q["request_id"][0]), step=int(q["step"][0]), position=0)
    assert int(b.argmax[0, 0]) == o["argmax"] and int(b.sample[0, 0]) == o["sample"]


@pytest.mark.parametrize("deferred", [False, True])
def test_nan_and_empty_rows_set_status(deferred):
    """NaN, +inf and all -inf rows raise their status bits and leave the valid rows alone.
    Deferred (no DG_SAMPLE_ALL) with a budget larger than any finite sum: the flagged rows'
    NaN entropies rank after the valid ones, so every slot of the sampler's list is filled."""
    n, L, V = 1, 5, 64
    x = torch.zeros((n, L, V), dtype=torch.float32)
    x[0, 1, 5] = float("nan")
    x[0, 2, :] = float("-inf")
    x[0, 3, 7] = float("inf")
    x[0, 4, 10:20] = float("-inf")      # some -inf entries are fine
    flags = dg.DG_ACTIVE if deferred else dg.DG_ACTIVE | dg.DG_SAMPLE_ALL
    p = _params(n, np.random.default_rng(9), temperature=1.0, flags=flags, beta=1e30)
    b = StepBuffers.make(n, L, DEV)
    dg.dg_clear_device_status()
    run_step(x.to(DEV), dg.params_tensor(p, DEV), 1, b)
    st = dg.dg_get_device_status()
    assert st & dg.DG_DEV_NAN_INF_ROW and st & dg.DG_DEV_EMPTY_ROW
    dg.dg_clear_device_status()
    # the row with a few -inf entries is valid and matches the oracle
    o = oracle.row_stats(x[0, 4].numpy(), T=float(p["temperature"][0]), seed=1,
                         request_id=int(p["request_id"][0]), step=int(p["step"][0]), position=4)
    assert int(b.argmax[0, 4]) == o["argmax"] and int(b.sample[0, 4]) == o["sample"]
    assert abs(float(b.entropy[0, 4]) - o["entropy"]) <= 1e-5 * o["entropy"]
    assert dg.dg_get_device_status() == 0


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_deferred_sampling_every_position_accepted(dtype):
    """A budget that accepts every position: the deferred sampling launch draws every row
    (about ten rows per CTA, flat rows included) and matches the oracle's samples at all of
    them; one canvas samples in the statistics pass instead (DG_SAMPLE_ALL)."""
    rng = np.random.default_rng(12)
    n, L, V = 6, 256, 40000
    x = synth.logits(n, L, V, seed=12, step=0, scale=(0.5, 12.0), spike_frac=0.1, dtype=dtype)
    p = _params(n, rng, beta=1e9)
    p["flags"][4] |= dg.DG_SAMPLE_ALL
    g, o, _ = _check_case(x, p, 77, V)
    assert (g["accept"] == 1).all() and (g["sample"] >= 0).all()
    assert (g["canvas"] == g["sample"]).all()


@pytest.mark.parametrize("sample_all", [False, True])
@pytest.mark.parametrize("dtype,V,ld,L", [("bf16", 2, 8, 33), ("bf16", 7, 8, 1), ("bf16", 9, 16, 64),
                                          ("fp32", 3, 4, 33), ("fp32", 5, 8, 1024), ("bf16", 8200, 8200, 1024)])
def test_step_edge_sizes(dtype, V, ld, L, sample_all):
    """The smallest vocabularies (one partial 16-byte vector per row, most of it padding that
    holds +1000 and must never be read as data), a one-position canvas and the largest canvas
    (L = 1024, one acceptance CTA of 1024 threads), in both sampling modes."""
    rng = np.random.default_rng(V * 7 + L)
    n = 2
    x = synth.logits(n, L, V, seed=V + L, step=1, scale=(0.5, 12.0), spike_frac=0.1, dtype=dtype, ld=ld)
    p = _params(n, rng)
    if sample_all:
        p["flags"] |= dg.DG_SAMPLE_ALL
    _check_case(x, p, 0xE06E + V, V, canvas0=rng.integers(0, V, (n, L)).astype(np.int32))


def test_split_step_on_two_streams_matches_one_call():
    """dg_denoise_stats on one stream and dg_denoise_samples on another (after an event, as
    the benchmark runs them beside the feedback GEMMs) give bit-identical outputs to
    dg_denoise_step, over three steps of a loop with mixed sampling modes."""
    rng = np.random.default_rng(21)
    n, L, V = 5, 256, 70001
    p = _params(n, rng, beta=12.0)
    p["flags"][1] |= dg.DG_SAMPLE_ALL
    p["flags"][3] = dg.DG_ACTIVE | dg.DG_READ_ONLY
    p["max_steps"][3] = 1
    canvas0 = rng.integers(0, V, (n, L)).astype(np.int32)
    one, two = StepBuffers.make(n, L, DEV, canvas0), StepBuffers.make(n, L, DEV, canvas0)
    ws1 = torch.empty(dg.dg_denoise_workspace_bytes(n, L, V), dtype=torch.uint8, device=DEV)
    ws2 = torch.empty_like(ws1)
    main, side = torch.cuda.Stream(), torch.cuda.Stream()
    done = torch.cuda.Event()
    for t in range(3):
        p["step"][:] = t
        pt = dg.params_tensor(p, DEV)
        x = synth.logits(n, L, V, seed=21, step=t, scale=(0.5, 12.0), spike_frac=0.1, ld=70008, device=DEV)
        torch.cuda.synchronize()
        run_step(x, pt, 4242, one, V=V)
        b = two
        dg.dg_denoise_stats(x, pt, 4242, b.canvas, b.prev, b.stable, b.accept, b.argmax, b.sample, b.entropy,
                            b.lse, b.converged, b.mean_entropy, b.n_accept, workspace=ws2, V=V, stream=main)
        done.record(main)
        side.wait_event(done)
        dg.dg_denoise_samples(x, pt, 4242, b.canvas, b.sample, ws2, V=V, stream=side)
        torch.cuda.synchronize()
        h1, h2 = one.host(), two.host()
        for k in h1:
            assert np.array_equal(h1[k], h2[k]), (t, k)
        assert (h2["sample"][0][h2["accept"][0] == 1] >= 0).all()


def test_whole_step_hand_worked_5x4x8():
    """The CUDA step over three steps against the hand-worked whole-step fixture (the same
    values the oracle is pinned to; tests/golden/step_worked_5x4x8.json says how each was
    worked out): entropies 0, ln 2, 2 ln 2 and lse = 0.5/T + ln|support| within fp32
    rounding, everything else exact."""
    from test_oracle_pins import _worked_step, check_worked_step, worked_step_inputs
    g = _worked_step()
    x, p, canvas = worked_step_inputs(g)
    n, L = canvas.shape
    xd = torch.from_numpy(x).to(DEV)
    b = StepBuffers.make(n, L, DEV, canvas)
    dg.dg_clear_device_status()
    for t in range(g["steps"]):
        p["step"][:] = t
        before = b.canvas.cpu().numpy().copy()
        run_step(xd, dg.params_tensor(p, DEV), g["seed"], b)
        torch.cuda.synchronize()
        h = b.host()
        out = {"canvas": h["canvas"], "prev_argmax": h["prev"], "stable_count": h["stable"],
               "accept_mask": h["accept"], "argmax": h["argmax"], "entropy": h["entropy"].astype(np.float64),
               "lse": h["lse"].astype(np.float64), "converged": h["converged"],
               "mean_entropy": h["mean_entropy"].astype(np.float64), "n_accept": h["n_accept"]}
        check_worked_step(g, t, out, before, ent_tol=2e-6, lse_rel=1e-6)
    assert dg.dg_get_device_status() == 0
