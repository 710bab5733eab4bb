"""The kernels' bounded waits, made to expire on purpose (no GPU fault involved).

Every mbarrier wait in the library's kernels polls a bounded number of times; on expiry the
kernel raises DG_DEV_TIMEOUT in the device status word, unwinds and returns, so the
context stays usable.  dg_probe_bounded_wait runs those same wait routines on a
shared-memory barrier that nothing arrives on, with a short limit: the waits must return,
report expiry and raise the bit, and a wait on a barrier that did complete must succeed.
(The unwinding of a GEMM with copies and MMAs still in flight is not exercised: that would
need a wait inside a running GEMM that never completes.)"""
import numpy as np
import pytest
import torch

import entropy_bounded_denoising_gb300 as dg
from entropy_bounded_denoising_gb300 import synth

from helpers import StepBuffers, run_step

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("polls", [1, 1000])
def test_expired_wait_returns_and_raises_timeout(polls):
    dg.dg_clear_device_status()
    assert dg.dg_get_device_status() == 0
    r = torch.full((3,), 7, dtype=torch.int32, device=DEV)
    dg.dg_probe_bounded_wait(polls, r)
    torch.cuda.synchronize()
    assert r.cpu().tolist() == [0, 0, 1]
    assert dg.dg_get_device_status() == dg.DG_DEV_TIMEOUT
    dg.dg_clear_device_status()
    assert dg.dg_get_device_status() == 0


def test_context_stays_usable_after_an_expired_wait():
    r = torch.zeros(3, dtype=torch.int32, device=DEV)
    dg.dg_probe_bounded_wait(64, r)
    dg.dg_clear_device_status()
    n, L, V = 2, 64, 4096
    x = synth.logits(n, L, V, seed=3, step=1, scale=(0.5, 8.0), device=DEV)
    p = {"temperature": np.ones(n, np.float32), "beta": np.full(n, 4.0, np.float32),
         "tau": np.full(n, 0.3, np.float32), "k": np.full(n, 2, np.int32), "max_steps": np.full(n, 8, np.int32),
         "min_accept": np.ones(n, np.int32), "step": np.ones(n, np.int32),
         "request_id": np.arange(n, dtype=np.uint32), "flags": np.full(n, dg.DG_ACTIVE, np.uint32)}
    b = StepBuffers.make(n, L, DEV)
    run_step(x, dg.params_tensor(p, DEV), 5, b)
    torch.cuda.synchronize()
    assert dg.dg_get_device_status() == 0
    assert (b.argmax.cpu() == x.float().argmax(-1).int().cpu()).all()
