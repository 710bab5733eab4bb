"""The overlapped launch schedule of one step against the in-line one, through the C ABI.

In line: dg_denoise_step, then dg_self_cond_logits with the step's converged flags.
Overlapped (what the benchmark runs for small batches): on the main stream
dg_self_cond_prepare with converged = NULL, dg_denoise_row_stats and dg_self_cond_pe; then
dg_denoise_accept and dg_denoise_samples on a second stream while dg_self_cond_mlp runs on the
main one; then, after an event from the second stream, dg_self_cond_zero_converged.  Every
output (canvas, state, statistics, samples, acceptance, convergence and the feedback rows)
must be bit-identical: the schedule moves launches, not arithmetic.  Cases: a mixed batch
(feedback, a canvas converging this step, read-only, inactive and DG_SAMPLE_ALL canvases;
ragged L and V; bf16 and fp32 logits) over two steps, and the single-request size."""
import numpy as np
import pytest
import torch

import entropy_bounded_denoising_gb300 as dg
from entropy_bounded_denoising_gb300 import synth

from helpers import StepBuffers

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _run(x, pt, seed, b, delta, ws_d, ws_s, weights, V, overlapped, main, side):
    n, L, ld = x.shape
    E, Wg, Wu, Wd = weights
    h = Wg.shape[0]
    if not overlapped:
        dg.dg_denoise_step(x, pt, seed, b.canvas, b.prev, b.stable, b.accept, b.argmax, b.sample, b.entropy, b.lse,
                           b.converged, b.mean_entropy, b.n_accept, workspace=ws_d, V=V, stream=main)
        dg.dg_self_cond_logits(x, b.lse, pt, b.converged, E, Wg, Wu, Wd, delta, ws_s, V=V, stream=main)
        return
    dg.dg_self_cond_prepare(pt, None, n, L, delta.shape[2], h, delta, ws_s, stream=main)
    dg.dg_denoise_row_stats(x, pt, seed, b.argmax, b.sample, b.entropy, b.lse, ws_d, V=V, stream=main)
    fork, accept_done = torch.cuda.Event(), torch.cuda.Event()
    dg.dg_self_cond_pe(x, b.lse, pt, E, h, ws_s, V=V, stream=main)
    fork.record(main)
    side.wait_event(fork)
    dg.dg_denoise_accept(b.entropy, b.sample, b.argmax, pt, seed, b.canvas, b.prev, b.stable, b.accept,
                         b.converged, ws_d, V=V, mean_entropy=b.mean_entropy, n_accept=b.n_accept, stream=side)
    dg.dg_denoise_samples(x, pt, seed, b.canvas, b.sample, ws_d, V=V, stream=side)
    accept_done.record(side)
    dg.dg_self_cond_mlp(n, L, Wg, Wu, Wd, delta, ws_s, stream=main)
    main.wait_event(accept_done)
    dg.dg_self_cond_zero_converged(pt, b.converged, delta, stream=main)


def _compare(n, L, V, ld, d, h, p, dtype, steps, seed):
    rng = np.random.default_rng(seed)
    E, Wg, Wu, Wd = (t.to(DEV) for t in synth.weights(V, d, h, seed=seed))
    canvas0 = rng.integers(0, V, (n, L)).astype(np.int32)
    bufs = [StepBuffers.make(n, L, DEV, canvas0) for _ in range(2)]
    deltas = [torch.full((n, L, d), float("nan"), dtype=torch.bfloat16, device=DEV) for _ in range(2)]
    dt = dg.DG_BF16 if dtype == "bf16" else dg.DG_FP32
    ws_d = [torch.empty(dg.dg_denoise_workspace_bytes(n, L, V, dt), dtype=torch.uint8, device=DEV) for _ in range(2)]
    ws_s = [torch.empty(dg.dg_self_cond_workspace_bytes(n, L, d, h), dtype=torch.uint8, device=DEV) for _ in range(2)]
    main, side = torch.cuda.Stream(), torch.cuda.Stream()
    dg.dg_clear_device_status()
    for t in range(steps):
        p["step"][:] = t
        pt = dg.params_tensor(p, DEV)
        x = synth.logits(n, L, V, seed=seed, step=t, scale=(0.5, 12.0), spike_frac=0.2, dtype=dtype, ld=ld,
                         device=DEV)
        torch.cuda.synchronize()
        for k in range(2):
            _run(x, pt, 0xC0FFEE + t, bufs[k], deltas[k], ws_d[k], ws_s[k], (E, Wg, Wu, Wd), V, k == 1, main, side)
        torch.cuda.synchronize()
        assert dg.dg_get_device_status() == 0
        h0, h1 = bufs[0].host(), bufs[1].host()
        for q in h0:
            assert np.array_equal(h0[q], h1[q]), (t, q)
        assert torch.equal(deltas[0], deltas[1]), t
    return bufs[0].host(), deltas[0]


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_overlapped_schedule_mixed_batch(dtype):
    rng = np.random.default_rng(5)
    n, L, V, ld, d, h = 5, 200, 5003, 5008, 192, 320
    p = {"temperature": rng.uniform(0.5, 1.5, n).astype(np.float32), "beta": np.full(n, 6.0, np.float32),
         "tau": np.full(n, 0.3, np.float32), "k": np.full(n, 1, np.int32),
         "max_steps": np.array([64, 1, 64, 64, 64], np.int32), "min_accept": np.ones(n, np.int32),
         "step": np.zeros(n, np.int32), "request_id": np.arange(n, dtype=np.uint32) + 7,
         "flags": np.array([dg.DG_ACTIVE | dg.DG_SELF_COND,
                            dg.DG_ACTIVE | dg.DG_SELF_COND,                       # converges this step
                            dg.DG_ACTIVE | dg.DG_READ_ONLY | dg.DG_SELF_COND,     # read-only: no feedback
                            0,                                                    # inactive
                            dg.DG_ACTIVE | dg.DG_SELF_COND | dg.DG_SAMPLE_ALL], np.uint32)}
    host, delta = _compare(n, L, V, ld, d, h, p, dtype, steps=2, seed=11)
    assert host["converged"][1] == 1 and host["converged"][0] == 0
    got = delta.float().cpu().numpy()
    assert (got[1] == 0).all() and (got[2] == 0).all() and (got[3] == 0).all()
    assert np.abs(got[0]).max() > 0 and np.abs(got[4]).max() > 0


def test_overlapped_schedule_single_request():
    wl = synth.WORKLOADS["single"]
    p = synth.canvas_params(wl, step=0)
    p["flags"] |= dg.DG_SELF_COND
    _compare(wl.n, wl.L, wl.V, wl.V, wl.d, wl.h, p, "bf16", steps=2, seed=wl.seed)
