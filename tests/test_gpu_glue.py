"""GPU parity of the rows around the step, through the C ABI, against the fp64 oracle:

* dg_choice_probs: p = exp(x_tok / T - lse) with the step's own lse from dg_denoise_step;
  relative tolerance 2e-7 |x/T| + 1.5e-6 |lse| + 1e-6 (fp32 scaling and exp, plus the lse's
  own 1e-6 relative bar), absolute 1e-37 for underflow.
* dg_denoise_step_choices (the same gather fused into the statistics pass): the step's outputs
  equal to dg_denoise_step's, the probabilities bit-equal to dg_choice_probs, and the same
  oracle tolerance.
* dg_embed_canvas: bit-exact (the output is a rounded bf16 pattern fixed by its definition).
* dg_commit: exact.
Small ragged cases on every element, the batched workload's full size on sampled rows."""
import numpy as np
import pytest
import torch

import entropy_bounded_denoising_gb300 as dg
from entropy_bounded_denoising_gb300 import synth
import oracle

from helpers import StepBuffers, run_step

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _params(n, rng, flags=None, T=None):
    p = {"temperature": (rng.uniform(0.4, 1.6, n) if T is None else np.full(n, T)).astype(np.float32),
         "beta": np.full(n, 8.0, np.float32), "tau": np.full(n, 0.3, np.float32),
         "k": np.full(n, 2, np.int32), "max_steps": np.full(n, 1, np.int32),
         "min_accept": np.ones(n, np.int32), "step": np.zeros(n, np.int32),
         "request_id": rng.integers(0, 1 << 31, n).astype(np.uint32),
         "flags": np.full(n, dg.DG_ACTIVE | dg.DG_READ_ONLY, np.uint32) if flags is None else flags}
    return p


def _check_probs(got, ref, y, lse):
    tol = 2e-7 * np.abs(y) + 1.5e-6 * np.abs(lse) + 1e-6
    err = np.abs(got - ref)
    ok = (err <= tol * np.abs(ref)) | (err <= 1e-37)
    assert ok.all(), (np.argwhere(~ok)[:5], got[~ok][:5], ref[~ok][:5])


def _logit_values(hx):
    if hx.dtype == np.uint16:
        return (hx.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return hx.astype(np.float64)


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("V,ld", [(5003, 5008), (40000, 40000)])
def test_choice_probs_small(dtype, V, ld):
    rng = np.random.default_rng(V)
    n, L, C = 3, 130, 6
    x = synth.logits(n, L, V, seed=V, step=1, scale=(0.5, 12.0), spike_frac=0.1, dtype=dtype, ld=ld)
    p = _params(n, rng)
    p["flags"][2] = 0                       # inactive: probs untouched
    b = StepBuffers.make(n, L, DEV)
    xd = x.to(DEV)
    pt = dg.params_tensor(p, DEV)
    run_step(xd, pt, 5, b, V=V)
    choices = rng.integers(0, V, (n, L, C)).astype(np.int32)
    choices[:, :, 0] = -1                   # unused slot
    choices[:, :, 1] = V + 3                # out of range
    am = b.argmax.cpu().numpy()
    choices[:, :, 2] = am                   # the argmax token: the largest probability
    probs = torch.full((n, L, C), -5.0, dtype=torch.float32, device=DEV)
    dg.dg_choice_probs(xd, b.lse, pt, torch.from_numpy(choices).to(DEV), probs, V=V)
    torch.cuda.synchronize()
    assert dg.dg_get_device_status() == 0
    got = probs.cpu().numpy()
    hx = synth.host_logits(x)
    assert (got[2] == -5.0).all()
    for c in range(2):
        ref = oracle.choice_probs(hx[c], np.full(L, float(p["temperature"][c])), choices[c], V=V)
        xv = _logit_values(hx[c])
        y = np.take_along_axis(xv, np.clip(choices[c], 0, V - 1), axis=1) / float(p["temperature"][c])
        lse = b.lse.cpu().numpy()[c][:, None]
        _check_probs(got[c], ref, y, lse)
        assert (got[c][:, :2] == 0).all()
        assert (got[c][:, 2] >= got[c][:, 3:].max(axis=1)).all()


def test_choice_probs_batched_full_size():
    wl = synth.WORKLOADS["batched"]
    n, L, V = wl.n, wl.L, wl.V
    rng = np.random.default_rng(11)
    x = synth.logits(n, L, V, seed=wl.seed, step=1, scale=wl.scale, spike_frac=wl.spike_frac, device=DEV)
    p = _params(n, rng, T=1.0)
    pt = dg.params_tensor(p, DEV)
    b = StepBuffers.make(n, L, DEV)
    run_step(x, pt, 5, b)
    C = 4
    choices = rng.integers(0, V, (n, L, C)).astype(np.int32)
    probs = torch.zeros((n, L, C), dtype=torch.float32, device=DEV)
    dg.dg_choice_probs(x, b.lse, pt, torch.from_numpy(choices).to(DEV), probs)
    torch.cuda.synchronize()
    assert dg.dg_get_device_status() == 0
    got = probs.cpu().numpy()
    lse = b.lse.cpu().numpy()
    for (c, i) in [(0, 0), (3, 77), (7, 255)]:
        hx = synth.host_logits(x[c, i:i + 1])
        ref = oracle.choice_probs(hx, [1.0], choices[c, i:i + 1], V=V)
        y = _logit_values(hx)[0][choices[c, i]]
        _check_probs(got[c, i:i + 1], ref, y[None, :], np.array([[lse[c, i]]]))


def _run_choices(xd, pt, seed, b, choices, probs, V):
    n, L, ld = xd.shape
    dg.dg_denoise_step_choices(xd, pt, seed, b.canvas, b.prev, b.stable, b.accept, b.argmax, b.sample,
                               b.entropy, b.lse, b.converged, choices, probs, b.mean_entropy, b.n_accept,
                               V=V, ld=ld)


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("V,ld,C", [(5003, 5008, 6), (40000, 40000, 33), (2, 8, 1)])
def test_step_with_fused_choices(dtype, V, ld, C):
    """dg_denoise_step_choices: every step output equal to dg_denoise_step's on the same
    inputs, the probabilities bit-equal to dg_choice_probs on the step's lse and within the
    oracle tolerance; read-only, normal (deferred and DG_SAMPLE_ALL) and inactive canvases in
    one batch; C = 33 spans two rounds of a warp's lanes."""
    rng = np.random.default_rng(V + C)
    n, L = 4, 70
    x = synth.logits(n, L, V, seed=V + 1, step=1, scale=(0.5, 12.0), spike_frac=0.2, dtype=dtype, ld=ld)
    p = _params(n, rng)
    p["flags"] = np.array([dg.DG_ACTIVE | dg.DG_READ_ONLY, dg.DG_ACTIVE, 0,
                           dg.DG_ACTIVE | dg.DG_SAMPLE_ALL], np.uint32)
    p["max_steps"][:] = 8
    pt = dg.params_tensor(p, DEV)
    xd = x.to(DEV)
    choices = rng.integers(0, V, (n, L, C)).astype(np.int32)
    if C >= 3:
        choices[:, :, 0] = -1
        choices[:, :, 1] = V
    ch = torch.from_numpy(choices).to(DEV)
    canvas0 = rng.integers(0, V, (n, L)).astype(np.int32)
    a = StepBuffers.make(n, L, DEV, canvas=canvas0)
    b = StepBuffers.make(n, L, DEV, canvas=canvas0)
    probs = torch.full((n, L, C), -5.0, dtype=torch.float32, device=DEV)
    _run_choices(xd, pt, 9, a, ch, probs, V)
    run_step(xd, pt, 9, b, V=V)
    ref_g = torch.full((n, L, C), -5.0, dtype=torch.float32, device=DEV)
    dg.dg_choice_probs(xd, b.lse, pt, ch, ref_g, V=V)
    torch.cuda.synchronize()
    assert dg.dg_get_device_status() == 0
    ha, hb = a.host(), b.host()
    for k in ha:
        assert np.array_equal(ha[k], hb[k]), k
    got = probs.cpu().numpy()
    assert np.array_equal(got, ref_g.cpu().numpy())
    assert (got[2] == -5.0).all()
    hx = synth.host_logits(x)
    for c in (0, 1, 3):
        T = float(p["temperature"][c])
        ref = oracle.choice_probs(hx[c], np.full(L, T), choices[c], V=V)
        y = np.take_along_axis(_logit_values(hx[c]), np.clip(choices[c], 0, V - 1), axis=1) / T
        _check_probs(got[c], ref, y, ha["lse"][c][:, None])
        if C >= 3:
            assert (got[c][:, :2] == 0).all()


def test_step_with_fused_choices_batched_full_size():
    """The batched workload (8 x 256, V = 262144) as read-only canvases with 4 choices per
    position, one of them the argmax: probabilities bit-equal to dg_choice_probs everywhere,
    against the oracle on sampled rows, and the argmax slot the largest."""
    wl = synth.WORKLOADS["batched"]
    n, L, V = wl.n, wl.L, wl.V
    rng = np.random.default_rng(12)
    x = synth.logits(n, L, V, seed=wl.seed, step=1, scale=wl.scale, spike_frac=wl.spike_frac, device=DEV)
    p = _params(n, rng)
    pt = dg.params_tensor(p, DEV)
    C = 4
    b = StepBuffers.make(n, L, DEV)
    run_step(x, pt, 5, b)
    choices = rng.integers(0, V, (n, L, C)).astype(np.int32)
    choices[:, :, 3] = b.argmax.cpu().numpy()
    ch = torch.from_numpy(choices).to(DEV)
    a = StepBuffers.make(n, L, DEV)
    probs = torch.zeros((n, L, C), dtype=torch.float32, device=DEV)
    _run_choices(x, pt, 5, a, ch, probs, V)
    ref_g = torch.zeros((n, L, C), dtype=torch.float32, device=DEV)
    dg.dg_choice_probs(x, a.lse, pt, ch, ref_g)
    torch.cuda.synchronize()
    assert dg.dg_get_device_status() == 0
    assert torch.equal(a.lse, b.lse) and torch.equal(a.entropy, b.entropy)
    got = probs.cpu().numpy()
    assert np.array_equal(got, ref_g.cpu().numpy())
    assert (got[:, :, 3] >= got[:, :, :3].max(axis=2)).all()
    lse = a.lse.cpu().numpy()
    for (c, i) in [(0, 0), (2, 131), (5, 64), (7, 255)]:
        T = float(p["temperature"][c])
        hx = synth.host_logits(x[c, i:i + 1])
        ref = oracle.choice_probs(hx, [T], choices[c, i:i + 1], V=V)
        y = _logit_values(hx)[0][choices[c, i]] / T
        _check_probs(got[c, i:i + 1], ref, y[None, :], np.array([[lse[c, i]]]))


def _bits(t):
    return synth.bf16_bits(t)


@pytest.mark.parametrize("scale", [1.0, 64.0, 0.70710677])
@pytest.mark.parametrize("with_delta", [True, False])
def test_embed_canvas_small_bit_exact(scale, with_delta):
    rng = np.random.default_rng(int(scale * 10) + with_delta)
    V, d, rows = 1000, 72, 600
    E = (torch.randn(V, d) * 0.5).to(torch.bfloat16).to(DEV)
    delta = (torch.randn(rows, d) * 0.1).to(torch.bfloat16).to(DEV) if with_delta else None
    canvas = rng.integers(0, V, rows).astype(np.int32)
    out = torch.full((rows, d), 7, dtype=torch.bfloat16, device=DEV)
    dg.dg_clear_device_status()
    dg.dg_embed_canvas(torch.from_numpy(canvas).to(DEV), E, delta, out, scale)
    torch.cuda.synchronize()
    assert dg.dg_get_device_status() == 0
    ref = oracle.embed_canvas(canvas, _bits(E), None if delta is None else _bits(delta), scale)
    assert np.array_equal(_bits(out), ref)


def test_embed_canvas_invalid_tokens():
    V, d = 16, 8
    E = torch.ones(V, d, dtype=torch.bfloat16, device=DEV)
    canvas = torch.tensor([3, -1, 16, 0], dtype=torch.int32, device=DEV)
    out = torch.full((4, d), 5, dtype=torch.bfloat16, device=DEV)
    dg.dg_clear_device_status()
    dg.dg_embed_canvas(canvas, E, None, out)
    st = dg.dg_get_device_status()
    dg.dg_clear_device_status()
    assert st & dg.DG_DEV_BAD_PARAM
    o = out.float().cpu().numpy()
    assert (o[0] == 1).all() and (o[1] == 0).all() and (o[2] == 0).all() and (o[3] == 1).all()


def test_embed_canvas_batched_full_size():
    wl = synth.WORKLOADS["batched"]
    n, L, V, d = wl.n, wl.L, wl.V, wl.d
    rng = np.random.default_rng(12)
    E = synth.weights(V, d, 8, seed=wl.seed, device=DEV)[0]
    delta = (torch.randn(n * L, d, device=DEV) * 0.02).to(torch.bfloat16)
    canvas = torch.from_numpy(rng.integers(0, V, n * L).astype(np.int32)).to(DEV)
    out = torch.empty((n * L, d), dtype=torch.bfloat16, device=DEV)
    dg.dg_embed_canvas(canvas, E, delta, out, 64.0)
    torch.cuda.synchronize()
    rows = [0, 1, 777, n * L - 1]
    cv = canvas.cpu().numpy()
    Eb = _bits(E)
    ref = oracle.embed_canvas(cv[rows], Eb, _bits(delta)[rows], 64.0)
    assert np.array_equal(_bits(out)[rows], ref)


def test_commit_matches_oracle():
    rng = np.random.default_rng(13)
    n, L = 40, 256
    p = _params(n, rng, flags=rng.choice([0, dg.DG_ACTIVE], n).astype(np.uint32))
    conv = rng.integers(0, 2, n).astype(np.uint8)
    argmax = rng.integers(0, 1000, (n, L)).astype(np.int32)
    tokens = np.full((n, L), -9, np.int32)
    prev = rng.integers(0, 1000, (n, L)).astype(np.int32)
    stable = rng.integers(0, 5, n).astype(np.int32)
    t = {k: torch.from_numpy(v).to(DEV) for k, v in
         dict(conv=conv, argmax=argmax, tokens=tokens, prev=prev, stable=stable).items()}
    committed = torch.full((n,), 7, dtype=torch.uint8, device=DEV)
    dg.dg_commit(dg.params_tensor(p, DEV), t["conv"], t["argmax"], t["tokens"], t["prev"], t["stable"], committed)
    torch.cuda.synchronize()
    r = oracle.commit(conv, (p["flags"] & dg.DG_ACTIVE).astype(np.uint8), argmax, tokens, prev, stable)
    assert np.array_equal(committed.cpu().numpy(), r["committed"])
    assert np.array_equal(t["tokens"].cpu().numpy(), r["tokens"])
    assert np.array_equal(t["prev"].cpu().numpy(), r["prev_argmax"])
    assert np.array_equal(t["stable"].cpu().numpy(), r["stable_count"])


def test_block_loop_prefill_denoise_commit():
    """Prefill -> denoise steps with feedback embeddings -> commit, against the oracle's loop:
    committed tokens equal the oracle's argmax canvas at the converging step."""
    rng = np.random.default_rng(14)
    wl = synth.WORKLOADS["tiny"]
    n, L, V, d, h = wl.n, wl.L, wl.V, wl.d, wl.h
    seed = 77
    base = synth.canvas_params(wl, step=0)
    E, Wg, Wu, Wd = synth.weights(V, d, h, seed=wl.seed, device=DEV)
    pt = dg.params_tensor(base, DEV)
    b = StepBuffers.make(n, L, DEV)
    dg.dg_canvas_init(b.canvas, n, L, V, pt, seed)
    o_canvas = oracle.canvas_init(n, L, V, base, seed)
    o_prev, o_stable = np.full((n, L), -1, np.int32), np.zeros(n, np.int32)
    delta = torch.zeros((n, L, d), dtype=torch.bfloat16, device=DEV)
    ws = torch.empty(dg.dg_self_cond_workspace_bytes(n, L, d, h), dtype=torch.uint8, device=DEV)
    emb = torch.empty((n * L, d), dtype=torch.bfloat16, device=DEV)
    tokens = torch.full((n, L), -1, dtype=torch.int32, device=DEV)
    committed = torch.zeros((n,), dtype=torch.uint8, device=DEV)
    done = False
    for t in range(int(base["max_steps"].max())):
        # the next pass's input embeddings: canvas tokens plus the stored feedback
        dg.dg_embed_canvas(b.canvas, E, delta if t > 0 else None, emb)
        ref_emb = oracle.embed_canvas(b.canvas.cpu().numpy(), _bits(E), _bits(delta).reshape(n * L, d) if t > 0 else None)
        torch.cuda.synchronize()
        assert np.array_equal(_bits(emb), ref_emb)
        p = synth.params_with(base, step=t)
        pt = dg.params_tensor(p, DEV)
        x = synth.logits(n, L, V, seed=wl.seed, step=t, scale=wl.scale, spike_frac=wl.spike_frac, dtype=wl.dtype)
        xd = x.to(DEV)
        run_step(xd, pt, seed, b, V=V)
        dg.dg_self_cond_logits(xd, b.lse, pt, b.converged, E, Wg, Wu, Wd, delta, ws, V=V)
        dg.dg_commit(pt, b.converged, b.argmax, tokens, b.prev, b.stable, committed)
        torch.cuda.synchronize()
        o = oracle.denoise_step(synth.host_logits(x), p, seed, o_canvas, o_prev, o_stable)
        o_canvas, o_prev, o_stable = o["canvas"], o["prev_argmax"], o["stable_count"]
        if o["converged"][0]:
            assert committed.cpu().numpy()[0] == 1
            assert np.array_equal(tokens.cpu().numpy()[0], o["argmax"][0])
            assert (b.prev.cpu().numpy()[0] == -1).all() and int(b.stable.cpu()[0]) == 0
            done = True
            break
        assert committed.cpu().numpy()[0] == 0
    assert done
