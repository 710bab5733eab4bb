"""GPU parity of the tensor-core path: the GEMM engine on plain operands (against fp32
matmuls of the same bf16 inputs), and the self-conditioning feedback
delta = W_down (gelu(W_gate pe) * (W_up pe)), pe = P . E, against the fp64 oracle
(per-row relative error <= 2e-2 and the elementwise bound of helpers.delta_elem_excess:
bf16 tensor-core operands, fp32 accumulation)."""
import numpy as np
import pytest
import torch

import entropy_bounded_denoising_gb300 as dg
from entropy_bounded_denoising_gb300 import synth
import oracle

from helpers import StepBuffers, check_delta, run_step

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _gemm_case(M, N, K, mn_major, seed=0):
    g = torch.Generator(device="cpu").manual_seed(seed)
    A = torch.randn((M, K), generator=g).to(torch.bfloat16)
    B = torch.randn((K, N) if mn_major else (N, K), generator=g).to(torch.bfloat16)
    ref = A.float() @ (B.float() if mn_major else B.float().T)
    C = torch.full((M, N), float("nan"), device=DEV)
    ws = torch.empty(max(1, dg.dg_gemm_workspace_bytes(M, N)), dtype=torch.uint8, device=DEV)
    dg.dg_clear_device_status()
    dg.dg_gemm_bf16(A.to(DEV), B.to(DEV), C, mn_major, ws)
    torch.cuda.synchronize()
    assert dg.dg_get_device_status() == 0
    got = C.cpu()
    err = (got - ref).abs().max().item() / ref.abs().max().item()
    assert torch.isfinite(got).all()
    assert err < 2e-3, (M, N, K, mn_major, err)


@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (300, 700, 1000), (1, 9, 8), (513, 260, 4104)])
def test_gemm_k_major(M, N, K):
    _gemm_case(M, N, K, False)


@pytest.mark.parametrize("M,N,K", [(128, 512, 32), (300, 1104, 3000), (5, 64, 40), (256, 600, 65536)])
def test_gemm_mn_major(M, N, K):
    _gemm_case(M, N, K, True)


def _weights(V, d, h, seed):
    E, Wg, Wu, Wd = synth.weights(V, d, h, seed=seed)
    return (E, Wg, Wu, Wd), tuple(synth.bf16_bits(t) for t in (E, Wg, Wu, Wd))


@pytest.mark.parametrize("V,d,h", [(1000, 64, 128), (5003, 192, 320), (4096, 512, 1024)])
def test_self_cond_probs(V, d, h):
    rng = np.random.default_rng(V)
    n_rows = 150
    ld = (V + 7) // 8 * 8
    P = np.zeros((n_rows, ld), np.float32)
    hot = rng.integers(0, V, n_rows)
    P[: n_rows // 2][np.arange(n_rows // 2), hot[: n_rows // 2]] = 1.0           # one-hot rows
    P[n_rows // 2:, :V] = rng.dirichlet(np.full(V, 0.05), n_rows - n_rows // 2)   # peaked rows
    Pb = torch.from_numpy(P).to(torch.bfloat16)
    (E, Wg, Wu, Wd), bits = _weights(V, d, h, seed=V)
    delta = torch.full((n_rows, d), float("nan"), dtype=torch.bfloat16, device=DEV)
    ws = torch.empty(dg.dg_self_cond_probs_workspace_bytes(n_rows, d, h), dtype=torch.uint8, device=DEV)
    dg.dg_clear_device_status()
    dg.dg_self_cond_probs(Pb.to(DEV), E.to(DEV), Wg.to(DEV), Wu.to(DEV), Wd.to(DEV), delta, ws, V=V)
    torch.cuda.synchronize()
    assert dg.dg_get_device_status() == 0
    Pw = Pb.float().numpy().astype(np.float64)[:, :V]
    pe = oracle.pe_from_probs(Pw, bits[0])
    one_hot_pe = (bits[0][hot[: n_rows // 2]].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert np.array_equal(pe[: n_rows // 2], one_hot_pe)       # P.E = E[argmax] for one-hot P
    ref = oracle.gated_mlp(pe, *bits[1:])
    check_delta(delta.float().cpu().numpy(), ref, (V, d, h))


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("V,ld,d,h,L", [(5003, 5008, 192, 320, 200), (2048, 2048, 512, 256, 128),
                                        (1024, 1032, 64, 128, 16)])
def test_self_cond_logits(dtype, V, ld, d, h, L):
    rng = np.random.default_rng(V + d)
    n = 4
    x = synth.logits(n, L, V, seed=d, step=1, scale=(0.5, 8.0), spike_frac=0.1, dtype=dtype, ld=ld)
    p = {"temperature": rng.uniform(0.5, 1.5, n).astype(np.float32), "beta": np.full(n, 4.0, np.float32),
         "tau": np.full(n, 0.3, np.float32), "k": np.full(n, 2, np.int32),
         "max_steps": np.array([64, 64, 64, 1], np.int32), "min_accept": np.ones(n, np.int32),
         "step": np.zeros(n, np.int32), "request_id": np.arange(n, dtype=np.uint32),
         "flags": np.array([dg.DG_ACTIVE | dg.DG_SELF_COND, dg.DG_ACTIVE, dg.DG_ACTIVE | dg.DG_SELF_COND,
                            dg.DG_ACTIVE | dg.DG_SELF_COND], np.uint32)}
    # canvas 3 converges this step (step cap 1), so its feedback is zero
    (E, Wg, Wu, Wd), bits = _weights(V, d, h, seed=d)
    xd = x.to(DEV)
    pt = dg.params_tensor(p, DEV)
    b = StepBuffers.make(n, L, DEV)
    run_step(xd, pt, 3, b, V=V)
    delta = torch.full((n, L, d), float("nan"), dtype=torch.bfloat16, device=DEV)
    ws = torch.empty(dg.dg_self_cond_workspace_bytes(n, L, d, h), dtype=torch.uint8, device=DEV)
    dg.dg_clear_device_status()
    dg.dg_self_cond_logits(xd, b.lse, pt, b.converged, E.to(DEV), Wg.to(DEV), Wu.to(DEV), Wd.to(DEV), delta,
                           ws, V=V)
    torch.cuda.synchronize()
    assert dg.dg_get_device_status() == 0
    got = delta.float().cpu().numpy()
    conv = b.converged.cpu().numpy()
    assert conv[3] == 1 and conv[0] == 0 and conv[2] == 0
    for c in (1, 3):
        assert (got[c] == 0).all(), c
    hx = synth.host_logits(x)
    for c in (0, 2):
        ref = oracle.self_cond_rows(hx[c], np.full(L, p["temperature"][c], np.float64), *bits, V=V)
        check_delta(got[c], ref, c)


@pytest.mark.parametrize("n,L,V,d,h", [(3, 256, 32768, 1024, 2048), (1, 200, 5003, 192, 320)])
def test_feedback_is_deterministic(n, L, V, d, h):
    """The feedback depends only on its inputs: two runs give bit-identical delta_emb (the
    split-K partials are added in slice order by one thread per column; no float atomics).
    A race in the GEMM engine's pipeline would show here as a bit difference."""
    rng = np.random.default_rng(n + L)
    ld = (V + 7) // 8 * 8  # rows 16-byte aligned
    x = synth.logits(n, L, V, seed=n * 7 + L, step=1, scale=(0.5, 12.0), spike_frac=0.1, ld=ld, device=DEV)
    (E, Wg, Wu, Wd), _ = _weights(V, d, h, seed=3)
    E, Wg, Wu, Wd = (t.to(DEV) for t in (E, Wg, Wu, Wd))
    p = {"temperature": rng.uniform(0.5, 1.5, n).astype(np.float32), "beta": np.full(n, 8.0, np.float32),
         "tau": np.full(n, 0.3, np.float32), "k": np.full(n, 2, np.int32), "max_steps": np.full(n, 64, np.int32),
         "min_accept": np.ones(n, np.int32), "step": np.ones(n, np.int32),
         "request_id": np.arange(n, dtype=np.uint32), "flags": np.full(n, dg.DG_ACTIVE | dg.DG_SELF_COND, np.uint32)}
    pt = dg.params_tensor(p, DEV)
    b = StepBuffers.make(n, L, DEV)
    run_step(x, pt, 5, b, V=V)
    ws = torch.empty(dg.dg_self_cond_workspace_bytes(n, L, d, h), dtype=torch.uint8, device=DEV)
    outs = []
    for _ in range(2):
        delta = torch.full((n, L, d), float("nan"), dtype=torch.bfloat16, device=DEV)
        dg.dg_self_cond_logits(x, b.lse, pt, b.converged, E, Wg, Wu, Wd, delta, ws, V=V)
        torch.cuda.synchronize()
        outs.append(delta.view(torch.int16).cpu())
    assert dg.dg_get_device_status() == 0
    assert torch.equal(outs[0], outs[1])
    assert torch.isfinite(outs[0].view(torch.bfloat16).float()).all()


def test_feedback_with_few_active_canvases_replans_on_device():
    """Six canvases of which only one has feedback on: the host plans P.E's k-slices for
    twelve m-tiles, the device for the two that are active (a different split of K); the
    feedback rows match the oracle and every other canvas's rows are zero."""
    n, L, V, d, h = 6, 256, 32768, 1024, 2048
    x = synth.logits(n, L, V, seed=61, step=1, scale=(0.5, 12.0), spike_frac=0.1, device=DEV)
    (E, Wg, Wu, Wd), bits = _weights(V, d, h, seed=4)
    E, Wg, Wu, Wd = (t.to(DEV) for t in (E, Wg, Wu, Wd))
    p = {"temperature": np.full(n, 0.9, np.float32), "beta": np.full(n, 8.0, np.float32),
         "tau": np.full(n, 0.3, np.float32), "k": np.full(n, 2, np.int32), "max_steps": np.full(n, 64, np.int32),
         "min_accept": np.ones(n, np.int32), "step": np.ones(n, np.int32),
         "request_id": np.arange(n, dtype=np.uint32), "flags": np.full(n, dg.DG_ACTIVE, np.uint32)}
    p["flags"][2] |= dg.DG_SELF_COND
    pt = dg.params_tensor(p, DEV)
    b = StepBuffers.make(n, L, DEV)
    run_step(x, pt, 9, b)
    ws = torch.empty(dg.dg_self_cond_workspace_bytes(n, L, d, h), dtype=torch.uint8, device=DEV)
    delta = torch.full((n, L, d), float("nan"), dtype=torch.bfloat16, device=DEV)
    dg.dg_clear_device_status()
    dg.dg_self_cond_logits(x, b.lse, pt, b.converged, E, Wg, Wu, Wd, delta, ws)
    torch.cuda.synchronize()
    assert dg.dg_get_device_status() == 0
    dh = delta.float().cpu().numpy()
    for c in range(n):
        if c != 2:
            assert (dh[c] == 0).all(), c
    rows = [0, 77, 255]
    ref = oracle.self_cond_rows(synth.host_logits(x[2, rows]), np.full(len(rows), 0.9), *bits, V=V)
    check_delta(dh[2, rows], ref)


def test_feedback_plan_beyond_the_host_table():
    """More than 256 canvases with feedback: the k-slice count is then evaluated on the device
    (the host tabulates it only up to 256 listed canvases).  300 canvases of 8 positions
    (each its own 128-row m-tile), all with feedback, against the oracle on sampled rows; and a
    second call with 200 of them listed (the table) on the same inputs, checked the same way."""
    n, L, V, d, h = 300, 8, 4096, 256, 512
    x = synth.logits(n, L, V, seed=71, step=1, scale=(0.5, 12.0), spike_frac=0.1, device=DEV)
    (E, Wg, Wu, Wd), bits = _weights(V, d, h, seed=5)
    E, Wg, Wu, Wd = (t.to(DEV) for t in (E, Wg, Wu, Wd))
    T = np.linspace(0.6, 1.4, n).astype(np.float32)
    p = {"temperature": T, "beta": np.full(n, 4.0, np.float32), "tau": np.full(n, 0.3, np.float32),
         "k": np.full(n, 2, np.int32), "max_steps": np.full(n, 64, np.int32), "min_accept": np.ones(n, np.int32),
         "step": np.ones(n, np.int32), "request_id": np.arange(n, dtype=np.uint32),
         "flags": np.full(n, dg.DG_ACTIVE | dg.DG_SELF_COND, np.uint32)}
    ws = torch.empty(dg.dg_self_cond_workspace_bytes(n, L, d, h), dtype=torch.uint8, device=DEV)
    hx = synth.host_logits(x)
    for listed in (n, 200):
        q = dict(p)
        q["flags"] = p["flags"].copy()
        q["flags"][listed:] = dg.DG_ACTIVE
        pt = dg.params_tensor(q, DEV)
        b = StepBuffers.make(n, L, DEV)
        run_step(x, pt, 9, b)
        delta = torch.full((n, L, d), float("nan"), dtype=torch.bfloat16, device=DEV)
        dg.dg_clear_device_status()
        dg.dg_self_cond_logits(x, b.lse, pt, b.converged, E, Wg, Wu, Wd, delta, ws)
        torch.cuda.synchronize()
        assert dg.dg_get_device_status() == 0
        dh = delta.float().cpu().numpy()
        assert np.isfinite(dh).all()
        if listed < n:
            assert (dh[listed:] == 0).all()
        for c in (0, 137, listed - 1):
            ref = oracle.self_cond_rows(hx[c], np.full(L, float(T[c]), np.float64), *bits, V=V)
            check_delta(dh[c], ref, (listed, c))

