"""dg_gemm_bf16_noalloc: the GEMM engine for callers that cannot allocate device memory
(a plugin handed only its input and output buffers, or a path where an allocation and its
implicit synchronisation are not allowed).  Its split-K partial tiles live in a fixed
8 MiB array inside the library instead of a caller workspace.

Checked through the C ABI on two calls in a row with different inputs: bit for bit
against dg_gemm_bf16 (which takes a workspace and plans the same k-slices, so it adds the
same partial tiles in the same order), so a stale partial tile left by the first call would
show in the second; and against an fp32 torch matmul of the same bf16 inputs within the
GEMM engine tests' tolerance.  Plus the host-side rejection of problems that need more
scratch than the array holds.  This file runs last so that a stop-at-first-failure run has
done every other test."""
import numpy as np
import pytest
import torch

import entropy_bounded_denoising_gb300 as dg

pytestmark = pytest.mark.gpu
DEV = "cuda"
REL_TOL = 2e-3   # the tolerance of the GEMM engine tests


def _inputs(M, N, K, mn_major, seed):
    g = torch.Generator(device="cpu").manual_seed(seed)
    A = torch.randn((M, K), generator=g).to(torch.bfloat16).to(DEV)
    B = torch.randn((K, N) if mn_major else (N, K), generator=g).to(torch.bfloat16).to(DEV)
    return A, B


@pytest.mark.parametrize("M,N,K,mn_major", [(256, 512, 65536, True), (128, 256, 65536, False),
                                            (300, 700, 1000, False)])
def test_noalloc_matches_workspace_gemm_twice(M, N, K, mn_major):
    dg.dg_clear_device_status()
    ws = torch.empty(max(1, dg.dg_gemm_workspace_bytes(M, N)), dtype=torch.uint8, device=DEV)
    for call, seed in enumerate((11, 12)):
        A, B = _inputs(M, N, K, mn_major, seed)
        ref = torch.full((M, N), float("nan"), device=DEV)
        dg.dg_gemm_bf16(A, B, ref, mn_major, ws)
        got = torch.full((M, N), float("nan"), device=DEV)
        dg.dg_gemm_bf16_noalloc(A, B, got, mn_major)
        torch.cuda.synchronize()
        assert dg.dg_get_device_status() == 0
        assert torch.isfinite(got).all(), call
        assert torch.equal(got, ref), (call, (got - ref).abs().max().item())
        exact = A.float() @ (B.float() if mn_major else B.float().T)
        err = (got - exact).abs().max().item() / exact.abs().max().item()
        assert err <= REL_TOL, (call, err)


def test_noalloc_rejects_problems_beyond_its_scratch():
    # 32 output tiles over a 262144-deep contraction split into many k-slices: the partial
    # tiles would need far more than the fixed array
    M, N, K = 1024, 2048, 262144
    A = torch.zeros((M, 64), dtype=torch.bfloat16, device=DEV)
    B = torch.zeros((64, N), dtype=torch.bfloat16, device=DEV)
    C = torch.zeros((M, N), device=DEV)
    rc = dg.dg_gemm_bf16_noalloc(A, B, C, True, K=64, check=False)
    assert rc == dg.DG_OK
    A = torch.zeros((M, K), dtype=torch.bfloat16, device=DEV)
    B = torch.zeros((K, N), dtype=torch.bfloat16, device=DEV)
    C.fill_(5.0)
    rc = dg.dg_gemm_bf16_noalloc(A, B, C, True, check=False)
    torch.cuda.synchronize()
    assert rc == dg.DG_ERR_UNSUPPORTED
    assert (C == 5.0).all()          # nothing was launched
