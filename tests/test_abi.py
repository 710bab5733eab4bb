"""The C ABI: the library builds for sm_103a on this host (cross-compiled), loads, and
exports every entry point include/dg.h declares; host-side validation rejects bad
arguments without touching the GPU."""
import os
import re

import pytest

import entropy_bounded_denoising_gb300 as dg
from entropy_bounded_denoising_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    txt = open(os.path.join(ROOT, "include", "dg.h")).read()
    return sorted(set(re.findall(r"^DG_API [^()]*?\b(dg_\w+)\(", txt, flags=re.M)))


def test_header_declares_the_boundary():
    names = _declared()
    for required in ("dg_denoise_step", "dg_self_cond_logits", "dg_self_cond_probs",
                     "dg_canvas_init", "dg_accept_from_entropy", "dg_get_device_status"):
        assert required in names


def test_library_builds_loads_and_exports_all():
    build.build()
    lib = dg.load()
    for name in _declared():
        assert hasattr(lib, name), name
    assert dg.version() >= 100
    assert dg.status_string(dg.DG_ERR_WORKSPACE) == "DG_ERR_WORKSPACE"


def test_host_validation_without_gpu():
    lib = dg.load()
    # null / out-of-range arguments are refused before any CUDA call
    assert lib.dg_denoise_step(None, 0, 8, 1, 16, 8, None, 0, *([None] * 11), None, 0, None) == dg.DG_ERR_INVALID_ARG
    assert lib.dg_denoise_step(None, 0, 8, 1, 0, 8, None, 0, *([None] * 11), None, 0, None) == dg.DG_ERR_INVALID_ARG
    assert lib.dg_denoise_step(None, 0, 8, 1, 2000, 8, None, 0, *([None] * 11), None, 0, None) == dg.DG_ERR_INVALID_ARG
    assert lib.dg_denoise_step(None, 7, 8, 1, 16, 8, None, 0, *([None] * 11), None, 0, None) == dg.DG_ERR_INVALID_ARG
    # ld < V
    assert lib.dg_denoise_step(16, 0, 4, 1, 16, 8, 16, 0, *([16] * 11), None, 0, None) == dg.DG_ERR_INVALID_ARG
    # misaligned logits / row stride
    assert lib.dg_denoise_step(18, 0, 8, 1, 16, 8, 16, 0, *([16] * 11), None, 0, None) == dg.DG_ERR_ALIGNMENT
    assert lib.dg_denoise_step(16, 0, 12, 1, 16, 12, 16, 0, *([16] * 11), None, 0, None) == dg.DG_ERR_ALIGNMENT
    # a row that does not fit the on-chip plan
    assert lib.dg_denoise_step(16, 1, 1 << 29, 1, 16, 1 << 29, 16, 0, *([16] * 11), None, 0, None) == dg.DG_ERR_UNSUPPORTED
    # the deferred-sampling list needs a workspace of 256 + 24 bytes per position, 256-byte
    # granular and 8-byte aligned
    assert lib.dg_denoise_step(16, 0, 8, 1, 16, 8, 16, 0, *([16] * 11), None, 0, None) == dg.DG_ERR_WORKSPACE
    assert lib.dg_denoise_step(16, 0, 8, 1, 16, 8, 16, 0, *([16] * 11), 256, 640, None) == dg.DG_ERR_WORKSPACE
    assert lib.dg_denoise_step(16, 0, 8, 1, 16, 8, 16, 0, *([16] * 11), 260, 768, None) == dg.DG_ERR_ALIGNMENT
    # the two halves of the step validate like the whole
    assert lib.dg_denoise_stats(16, 0, 8, 1, 16, 8, None, 0, *([16] * 11), 256, 768, None) == dg.DG_ERR_INVALID_ARG
    assert lib.dg_denoise_stats(16, 0, 8, 1, 16, 8, 16, 0, *([16] * 11), None, 0, None) == dg.DG_ERR_WORKSPACE
    assert lib.dg_denoise_samples(16, 0, 8, 1, 16, 8, 16, 0, None, 16, 256, 768, None) == dg.DG_ERR_INVALID_ARG
    assert lib.dg_denoise_samples(16, 0, 8, 1, 16, 8, 16, 0, 16, 16, 256, 640, None) == dg.DG_ERR_WORKSPACE
    assert lib.dg_denoise_samples(18, 0, 8, 1, 16, 8, 16, 0, 16, 16, 256, 768, None) == dg.DG_ERR_ALIGNMENT
    # the step with the fused choice gather: C within 1..1024, choices and probs given, then
    # the step's own checks
    assert lib.dg_denoise_step_choices(16, 0, 8, 1, 16, 8, 16, 0, *([16] * 11), 16, 0, 16, 256, 768, None) == dg.DG_ERR_INVALID_ARG
    assert lib.dg_denoise_step_choices(16, 0, 8, 1, 16, 8, 16, 0, *([16] * 11), 16, 1025, 16, 256, 768, None) == dg.DG_ERR_INVALID_ARG
    assert lib.dg_denoise_step_choices(16, 0, 8, 1, 16, 8, 16, 0, *([16] * 11), None, 4, 16, 256, 768, None) == dg.DG_ERR_INVALID_ARG
    assert lib.dg_denoise_step_choices(16, 0, 8, 1, 16, 8, 16, 0, *([16] * 11), 16, 4, None, 256, 768, None) == dg.DG_ERR_INVALID_ARG
    assert lib.dg_denoise_step_choices(18, 0, 8, 1, 16, 8, 16, 0, *([16] * 11), 16, 4, 16, 256, 768, None) == dg.DG_ERR_ALIGNMENT
    assert lib.dg_denoise_step_choices(16, 0, 8, 1, 16, 8, 16, 0, *([16] * 11), 16, 4, 16, None, 0, None) == dg.DG_ERR_WORKSPACE
    assert lib.dg_denoise_step_choices(None, 0, 8, 0, 16, 8, None, 0, *([None] * 11), None, 4, None, None, 0, None) == dg.DG_OK
    # the staged statistics / acceptance calls and the converged-row zeroing
    assert lib.dg_denoise_row_stats(16, 0, 8, 1, 16, 8, 16, 0, 16, 16, 16, None, 256, 768, None) == dg.DG_ERR_INVALID_ARG
    assert lib.dg_denoise_row_stats(18, 0, 8, 1, 16, 8, 16, 0, 16, 16, 16, 16, 256, 768, None) == dg.DG_ERR_ALIGNMENT
    assert lib.dg_denoise_row_stats(16, 0, 8, 1, 16, 8, 16, 0, 16, 16, 16, 16, 256, 640, None) == dg.DG_ERR_WORKSPACE
    assert lib.dg_denoise_row_stats(None, 0, 8, 0, 16, 8, None, 0, None, None, None, None, None, 0, None) == dg.DG_OK
    assert lib.dg_denoise_accept(16, 16, 16, 1, 16, 8, 16, 0, *([16] * 4), None, None, None, 256, 768, None) == dg.DG_ERR_INVALID_ARG
    assert lib.dg_denoise_accept(16, 16, 16, 1, 16, 8, 16, 0, *([16] * 5), None, None, 256, 640, None) == dg.DG_ERR_WORKSPACE
    assert lib.dg_denoise_accept(16, 16, 16, 1, 16, 8, 16, 0, *([16] * 5), None, None, 260, 768, None) == dg.DG_ERR_ALIGNMENT
    assert lib.dg_denoise_accept(16, 16, 16, 1, 2000, 8, 16, 0, *([16] * 5), None, None, 256, 768, None) == dg.DG_ERR_INVALID_ARG
    assert lib.dg_self_cond_zero_converged(16, 16, 1, 16, 12, 16, None) == dg.DG_ERR_INVALID_ARG
    assert lib.dg_self_cond_zero_converged(16, None, 1, 16, 16, 16, None) == dg.DG_ERR_INVALID_ARG
    assert lib.dg_self_cond_zero_converged(16, 16, 1, 16, 16, 18, None) == dg.DG_ERR_ALIGNMENT
    assert lib.dg_self_cond_zero_converged(None, None, 0, 16, 16, None, None) == dg.DG_OK
    # the bounded-wait probe: poll limits outside 1..65536, a null or misaligned result
    assert lib.dg_probe_bounded_wait(0, 16, None) == dg.DG_ERR_INVALID_ARG
    assert lib.dg_probe_bounded_wait(65537, 16, None) == dg.DG_ERR_INVALID_ARG
    assert lib.dg_probe_bounded_wait(100, None, None) == dg.DG_ERR_INVALID_ARG
    assert lib.dg_probe_bounded_wait(100, 18, None) == dg.DG_ERR_ALIGNMENT
    assert lib.dg_denoise_samples(None, 0, 8, 0, 16, 8, None, 0, None, None, None, 0, None) == dg.DG_OK
    # empty batch is a no-op
    assert lib.dg_denoise_step(None, 0, 8, 0, 16, 8, None, 0, *([None] * 11), None, 0, None) == dg.DG_OK
    assert lib.dg_denoise_workspace_bytes(8, 256, 262144, 0) == 256 + 24 * 8 * 256
    assert lib.dg_denoise_workspace_bytes(1, 16, 1024, 1) == 768
    # self-conditioning: sizes and alignment
    assert lib.dg_self_cond_logits(16, 0, 64, 16, 16, None, 1, 16, 64, 12, 128, 16, 16, 16, 16, 16, 16, 1 << 30, None) == dg.DG_ERR_INVALID_ARG
    assert lib.dg_self_cond_logits(16, 0, 64, 16, 16, None, 1, 16, 64, 64, 128, 18, 16, 16, 16, 16, 16, 1 << 30, None) == dg.DG_ERR_ALIGNMENT
    assert lib.dg_self_cond_probs(16, 64, 4, 64, 64, 128, 16, 16, 16, 16, 16, None, 0, None) == dg.DG_ERR_WORKSPACE
    assert lib.dg_gemm_bf16(16, 8, 16, 8, 0, 16, 8, 4, 4, 0, None, 0, None) == dg.DG_ERR_INVALID_ARG
    assert lib.dg_philox_words(0, 0, 0, 0, 300, 0, 4, 16, None) == dg.DG_ERR_INVALID_ARG
    assert lib.dg_canvas_init(None, 1, 16, 8, None, 0, None) == dg.DG_ERR_INVALID_ARG
    assert lib.dg_advance_params(None, None, -1, None) == dg.DG_ERR_INVALID_ARG


def test_lm_head_validation_without_gpu():
    lib = dg.load()
    # workspace: deferred list (256 + 24 per position), canvas list, 20 bytes per position and tile
    assert dg.dg_lm_head_workspace_bytes(2, 16, 1000) == 1024 + 256 + 32 * 4 * 20
    assert dg.dg_lm_head_workspace_bytes(8, 256, 262144) == \
        (256 + 24 * 2048 + 255) // 256 * 256 + 256 + 2048 * 1024 * 20
    ws = dg.dg_lm_head_workspace_bytes(1, 16, 64)

    def call(h=16, ldh=64, W=16, ldw=64, n=1, L=16, V=64, d=64, logits=16, ld=64, w=256, wb=None):
        return lib.dg_lm_head_logits(h, ldh, W, ldw, n, L, V, d, 16, logits, ld, w, ws if wb is None else wb, None)

    assert call(d=60, ldh=60, ldw=60) == dg.DG_ERR_INVALID_ARG      # d % 8
    assert call(ldh=32) == dg.DG_ERR_INVALID_ARG                    # ldh < d
    assert call(ld=56) == dg.DG_ERR_INVALID_ARG                     # ld < V
    assert call(V=1 << 30, ld=1 << 30) == dg.DG_ERR_INVALID_ARG     # V >= 2^30
    assert call(L=0) == dg.DG_ERR_INVALID_ARG
    assert call(h=None) == dg.DG_ERR_INVALID_ARG
    assert call(h=24) == dg.DG_ERR_ALIGNMENT
    assert call(ldw=68) == dg.DG_ERR_ALIGNMENT
    assert call(ld=68) == dg.DG_ERR_ALIGNMENT
    assert call(wb=ws - 1) == dg.DG_ERR_WORKSPACE
    assert call(w=None) == dg.DG_ERR_WORKSPACE
    assert call(w=264) == dg.DG_ERR_ALIGNMENT
    assert call(n=0) == dg.DG_OK
    step = lib.dg_lm_head_denoise_step
    args = [16, 64, 16, 64, 1, 16, 64, 64, 16, 0, 16, 64]
    assert step(*args, *([16] * 11), 256, ws - 1, None) == dg.DG_ERR_WORKSPACE
    assert step(*args, None, *([16] * 10), 256, ws, None) == dg.DG_ERR_INVALID_ARG   # canvas
    assert step(*args[:4], 0, *args[5:], *([None] * 11), None, 0, None) == dg.DG_OK


def test_attention_validation_without_gpu():
    lib = dg.load()

    assert dg.dg_attention_workspace_bytes(3, 300) == 256      # 16 + 3 x 3 x 8 bytes, rounded
    assert dg.dg_attention_workspace_bytes(100, 1024) == (16 + 100 * 8 * 8 + 255) // 256 * 256

    def call(q=16, k=16, v=16, o=16, n=1, mq=4, tq=4, tk=8, Hq=2, Hkv=1, D=128, W=-1, scale=0.1, ws=256, wsb=256):
        return lib.dg_attention(q, k, v, o, None, 16, 16, 16, n, mq, tq, tk, Hq, Hkv, D, W, scale, ws, wsb, None)

    assert call(D=96) == dg.DG_ERR_UNSUPPORTED
    assert call(D=512) == dg.DG_ERR_UNSUPPORTED
    assert call(Hq=3, Hkv=2) == dg.DG_ERR_INVALID_ARG
    assert call(W=-2) == dg.DG_ERR_INVALID_ARG
    assert call(scale=float("nan")) == dg.DG_ERR_INVALID_ARG
    assert call(mq=0) == dg.DG_ERR_INVALID_ARG
    assert call(tk=0) == dg.DG_ERR_INVALID_ARG
    assert call(q=None) == dg.DG_ERR_INVALID_ARG
    assert call(o=24) == dg.DG_ERR_ALIGNMENT
    assert call(ws=None) == dg.DG_ERR_WORKSPACE
    assert call(wsb=0) == dg.DG_ERR_WORKSPACE
    assert call(ws=264) == dg.DG_ERR_ALIGNMENT
    assert call(n=0, q=None) == dg.DG_OK


def test_params_record_layout():
    import numpy as np
    p = {"temperature": np.float32([0.5]), "beta": np.float32([2.0]), "tau": np.float32([0.25]),
         "k": np.int32([3]), "max_steps": np.int32([9]), "min_accept": np.int32([1]),
         "step": np.int32([4]), "request_id": np.uint32([77]), "flags": np.uint32([5])}
    raw = dg.pack_params(p)
    assert len(raw) == dg.PARAM_BYTES == 36
    import torch
    back = dg.unpack_params(torch.frombuffer(bytearray(raw), dtype=torch.uint8))
    for k, v in p.items():
        assert back[k][0] == v[0]
