"""ctypes binding of libdg (include/dg.h): argument marshalling only.

Every function here has the name of the C entry point it calls and forwards torch tensors
as raw device pointers on the current (or given) CUDA stream.  All arithmetic runs in the
library's kernels; there is no fallback.  Loading fails loudly when the library has not been
built (run ``entropy_bounded_denoising_gb300.build.build()``).
"""
from __future__ import annotations

import ctypes
import os
import struct

import numpy as np
import torch

from . import build as _build

DG_OK, DG_ERR_INVALID_ARG, DG_ERR_ALIGNMENT, DG_ERR_WORKSPACE, DG_ERR_UNSUPPORTED, DG_ERR_CUDA = 0, -1, -2, -3, -4, -5
DG_BF16, DG_FP32 = 0, 1
DG_ACTIVE, DG_READ_ONLY, DG_SELF_COND, DG_SAMPLE_ALL = 1, 2, 4, 8
DG_DEV_NAN_INF_ROW, DG_DEV_EMPTY_ROW, DG_DEV_TIMEOUT, DG_DEV_BAD_PARAM = 1, 2, 4, 8

PARAM_FIELDS = ("temperature", "beta", "tau", "k", "max_steps", "min_accept", "step",
                "request_id", "flags")
_PARAM_FMT = "<fffiiiiII"
PARAM_BYTES = struct.calcsize(_PARAM_FMT)   # 36, sizeof(dg_canvas_params)

_lib = None


class DGError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} failed: {status_string(code)} ({code})")
        self.code = code


def library_path() -> str:
    return _build.LIB


def load(path: str | None = None):
    """Load libdg.so (built in-tree).  Raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or _build.LIB
    if not os.path.exists(path):
        raise RuntimeError(f"libdg.so not found at {path}: build it with "
                           "entropy_bounded_denoising_gb300.build.build()")
    lib = ctypes.CDLL(path)
    P, i32, i64, u32, u64, sz = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32,
                                  ctypes.c_uint64, ctypes.c_size_t)
    st = ctypes.c_int
    sig = {
        "dg_denoise_workspace_bytes": (sz, [i64, i32, i64, ctypes.c_int]),
        "dg_denoise_step": (st, [P, ctypes.c_int, i64, i64, i32, i64, P, u64] + [P] * 11 + [P, sz, P]),
        "dg_denoise_stats": (st, [P, ctypes.c_int, i64, i64, i32, i64, P, u64] + [P] * 11 + [P, sz, P]),
        "dg_denoise_samples": (st, [P, ctypes.c_int, i64, i64, i32, i64, P, u64, P, P, P, sz, P]),
        "dg_denoise_row_stats": (st, [P, ctypes.c_int, i64, i64, i32, i64, P, u64, P, P, P, P, P, sz, P]),
        "dg_denoise_accept": (st, [P, P, P, i64, i32, i64, P, u64] + [P] * 7 + [P, sz, P]),
        "dg_self_cond_zero_converged": (st, [P, P, i64, i32, i32, P, P]),
        "dg_denoise_step_choices": (st, [P, ctypes.c_int, i64, i64, i32, i64, P, u64] + [P] * 11
                                    + [P, i32, P] + [P, sz, P]),
        "dg_accept_from_entropy": (st, [P, P, P, i64, i32, i64, P, u64] + [P] * 7 + [P]),
        "dg_lm_head_workspace_bytes": (sz, [i64, i32, i64]),
        "dg_lm_head_logits": (st, [P, i64, P, i64, i64, i32, i64, i32, P, P, i64, P, sz, P]),
        "dg_lm_head_denoise_step": (st, [P, i64, P, i64, i64, i32, i64, i32, P, u64, P, i64]
                                    + [P] * 11 + [P, sz, P]),
        "dg_canvas_init": (st, [P, i64, i32, i64, P, u64, P]),
        "dg_advance_params": (st, [P, P, i64, P]),
        "dg_self_cond_workspace_bytes": (sz, [i64, i32, i32, i32]),
        "dg_self_cond_logits": (st, [P, ctypes.c_int, i64, P, P, P, i64, i32, i64, i32, i32,
                                     P, P, P, P, P, P, sz, P]),
        "dg_self_cond_prepare": (st, [P, P, i64, i32, i32, i32, P, P, sz, P]),
        "dg_self_cond_pe": (st, [P, ctypes.c_int, i64, P, P, i64, i32, i64, i32, i32, P, P, sz, P]),
        "dg_self_cond_mlp": (st, [i64, i32, i32, i32, P, P, P, P, P, sz, P]),
        "dg_self_cond_probs_workspace_bytes": (sz, [i64, i32, i32]),
        "dg_self_cond_probs": (st, [P, i64, i64, i64, i32, i32, P, P, P, P, P, P, sz, P]),
        "dg_gemm_workspace_bytes": (sz, [i64, i64]),
        "dg_gemm_bf16": (st, [P, i64, P, i64, ctypes.c_int, P, i64, i64, i64, i64, P, sz, P]),
        "dg_gemm_bf16_noalloc": (st, [P, i64, P, i64, ctypes.c_int, P, i64, i64, i64, i64, P]),
        "dg_choice_probs": (st, [P, ctypes.c_int, i64, P, P, i64, i32, i64, P, i32, P, P]),
        "dg_attention_workspace_bytes": (sz, [i32, i32]),
        "dg_attention": (st, [P, P, P, P, P, P, P, P, i32, i32, i64, i64, i32, i32, i32, i32, ctypes.c_float,
                              P, sz, P]),
        "dg_embed_canvas": (st, [P, i64, i64, P, i32, P, ctypes.c_float, P, P]),
        "dg_commit": (st, [P, P, P, i64, i32, P, P, P, P, P]),
        "dg_philox_words": (st, [u64, u32, u32, u32, u32, u32, i64, P, P]),
        "dg_get_device_status": (st, [P, ctypes.POINTER(u32)]),
        "dg_clear_device_status": (st, [P]),
        "dg_probe_bounded_wait": (st, [u32, P, P]),
        "dg_status_string": (ctypes.c_char_p, [st]),
        "dg_version": (i32, []),
        "dg_launch_count": (u64, []),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _lib = lib
    return lib


def exported_symbols() -> list[str]:
    lib = load()
    return [n for n in ("dg_denoise_workspace_bytes", "dg_denoise_step", "dg_denoise_stats",
                        "dg_denoise_samples", "dg_denoise_step_choices", "dg_denoise_row_stats", "dg_denoise_accept",
                        "dg_self_cond_zero_converged", "dg_accept_from_entropy", "dg_lm_head_workspace_bytes",
                        "dg_lm_head_logits", "dg_lm_head_denoise_step",
                        "dg_canvas_init", "dg_advance_params", "dg_self_cond_workspace_bytes",
                        "dg_self_cond_logits", "dg_self_cond_prepare", "dg_self_cond_pe",
                        "dg_self_cond_mlp", "dg_self_cond_probs_workspace_bytes",
                        "dg_self_cond_probs", "dg_gemm_workspace_bytes", "dg_gemm_bf16",
                        "dg_gemm_bf16_noalloc", "dg_choice_probs", "dg_embed_canvas", "dg_commit", "dg_attention",
                        "dg_attention_workspace_bytes",
                        "dg_philox_words", "dg_get_device_status", "dg_clear_device_status",
                        "dg_probe_bounded_wait",
                        "dg_status_string", "dg_version", "dg_launch_count") if hasattr(lib, n)]


# ------------------------------------------------------------------ marshalling helpers
def _p(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise ValueError("device tensor expected")
    return t.data_ptr()


def _s(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check(fn: str, code: int) -> None:
    if code != DG_OK:
        raise DGError(fn, code)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return DG_BF16
    if t.dtype == torch.float32:
        return DG_FP32
    raise TypeError("logits must be bfloat16 or float32")


def status_string(code: int) -> str:
    return load().dg_status_string(int(code)).decode()


def version() -> int:
    return int(load().dg_version())


def dg_launch_count() -> int:
    return int(load().dg_launch_count())


def pack_params(p: dict) -> bytes:
    """Pack per-canvas parameter arrays into dg_canvas_params records (host bytes)."""
    n = len(p["flags"])
    return b"".join(struct.pack(_PARAM_FMT, *(np.asarray(p[f])[i].item() for f in PARAM_FIELDS))
                    for i in range(n))


def params_tensor(p: dict, device="cuda") -> torch.Tensor:
    """Per-canvas parameters as a device uint8 tensor [n * 36]."""
    raw = np.frombuffer(pack_params(p), dtype=np.uint8).copy()
    return torch.from_numpy(raw).to(device)


def unpack_params(t: torch.Tensor) -> dict:
    raw = t.detach().cpu().numpy().tobytes()
    n = len(raw) // PARAM_BYTES
    rows = [struct.unpack_from(_PARAM_FMT, raw, i * PARAM_BYTES) for i in range(n)]
    return {f: np.array([r[j] for r in rows]) for j, f in enumerate(PARAM_FIELDS)}


# ------------------------------------------------------------------ entry points
def dg_denoise_workspace_bytes(n_canvas: int, L: int, V: int, dtype: int = DG_BF16) -> int:
    return int(load().dg_denoise_workspace_bytes(n_canvas, L, V, dtype))


def _denoise_dims(logits, n_canvas, L, V, ld):
    n, Lx, ldx = logits.shape if logits.dim() == 3 else (n_canvas, L, ld)
    n_canvas = n if n_canvas is None else n_canvas
    L = Lx if L is None else L
    ld = ldx if ld is None else ld
    V = ld if V is None else V
    return n_canvas, L, V, ld


def _denoise_ws(workspace, logits, n_canvas, L, V):
    if workspace is None:  # the caller gave none: one sized by the library, on the logits' device
        workspace = torch.empty(dg_denoise_workspace_bytes(n_canvas, L, V, _dtype_code(logits)),
                                dtype=torch.uint8, device=logits.device)
    return workspace, workspace.numel() * workspace.element_size()


def _denoise_full(fn, logits, params, seed, canvas, prev_argmax, stable_count, accept_mask, argmax,
                  sample, entropy, lse, converged, mean_entropy, n_accept, workspace, n_canvas, L, V,
                  ld, stream, check):
    n_canvas, L, V, ld = _denoise_dims(logits, n_canvas, L, V, ld)
    workspace, ws_bytes = _denoise_ws(workspace, logits, n_canvas, L, V)
    rc = getattr(load(), fn)(_p(logits), _dtype_code(logits), ld, n_canvas, L, V, _p(params),
                             int(seed) & 0xFFFFFFFFFFFFFFFF, _p(canvas), _p(prev_argmax),
                             _p(stable_count), _p(accept_mask), _p(argmax), _p(sample), _p(entropy),
                             _p(lse), _p(converged), _p(mean_entropy), _p(n_accept),
                             _p(workspace), ws_bytes, _s(stream))
    if check:
        _check(fn, rc)
    return rc


def dg_denoise_step(logits, params, seed, canvas, prev_argmax, stable_count, accept_mask, argmax,
                    sample, entropy, lse, converged, mean_entropy=None, n_accept=None,
                    workspace=None, *, n_canvas=None, L=None, V=None, ld=None, stream=None,
                    check=True) -> int:
    return _denoise_full("dg_denoise_step", logits, params, seed, canvas, prev_argmax, stable_count,
                         accept_mask, argmax, sample, entropy, lse, converged, mean_entropy, n_accept,
                         workspace, n_canvas, L, V, ld, stream, check)


def dg_denoise_step_choices(logits, params, seed, canvas, prev_argmax, stable_count, accept_mask,
                            argmax, sample, entropy, lse, converged, choices, probs, mean_entropy=None,
                            n_accept=None, workspace=None, *, n_canvas=None, L=None, V=None, ld=None,
                            stream=None, check=True) -> int:
    """dg_denoise_step plus probs[c, i, k] = exp(logits[c, i, choices[c, i, k]] / T - lse[c, i])
    gathered in the statistics pass; choices [n, L, C] int32, probs [n, L, C] float32."""
    n_canvas, L, V, ld = _denoise_dims(logits, n_canvas, L, V, ld)
    workspace, ws_bytes = _denoise_ws(workspace, logits, n_canvas, L, V)
    C = choices.shape[-1]
    rc = load().dg_denoise_step_choices(_p(logits), _dtype_code(logits), ld, n_canvas, L, V, _p(params),
                                        int(seed) & 0xFFFFFFFFFFFFFFFF, _p(canvas), _p(prev_argmax),
                                        _p(stable_count), _p(accept_mask), _p(argmax), _p(sample),
                                        _p(entropy), _p(lse), _p(converged), _p(mean_entropy), _p(n_accept),
                                        _p(choices), C, _p(probs), _p(workspace), ws_bytes, _s(stream))
    if check:
        _check("dg_denoise_step_choices", rc)
    return rc


def dg_denoise_stats(logits, params, seed, canvas, prev_argmax, stable_count, accept_mask, argmax,
                     sample, entropy, lse, converged, mean_entropy=None, n_accept=None,
                     workspace=None, *, n_canvas=None, L=None, V=None, ld=None, stream=None,
                     check=True) -> int:
    """The statistics / acceptance half of dg_denoise_step (pass the same workspace to
    dg_denoise_samples afterwards)."""
    if workspace is None:
        raise ValueError("dg_denoise_stats needs the workspace that dg_denoise_samples will read")
    return _denoise_full("dg_denoise_stats", logits, params, seed, canvas, prev_argmax, stable_count,
                         accept_mask, argmax, sample, entropy, lse, converged, mean_entropy, n_accept,
                         workspace, n_canvas, L, V, ld, stream, check)


def dg_denoise_row_stats(logits, params, seed, argmax, sample, entropy, lse, workspace, *, n_canvas=None,
                         L=None, V=None, ld=None, stream=None, check=True) -> int:
    """K1 alone: per-position statistics (and DG_SAMPLE_ALL samples) into the given buffers;
    the workspace then goes to dg_denoise_accept and dg_denoise_samples."""
    n_canvas, L, V, ld = _denoise_dims(logits, n_canvas, L, V, ld)
    ws_bytes = workspace.numel() * workspace.element_size()
    rc = load().dg_denoise_row_stats(_p(logits), _dtype_code(logits), ld, n_canvas, L, V, _p(params),
                                     int(seed) & 0xFFFFFFFFFFFFFFFF, _p(argmax), _p(sample), _p(entropy),
                                     _p(lse), _p(workspace), ws_bytes, _s(stream))
    if check:
        _check("dg_denoise_row_stats", rc)
    return rc


def dg_denoise_accept(entropy, sample, argmax, params, seed, canvas, prev_argmax, stable_count, accept_mask,
                      converged, workspace, *, V, mean_entropy=None, n_accept=None, stream=None,
                      check=True) -> int:
    """Acceptance, renoise, convergence and the sampler's list after dg_denoise_row_stats."""
    n_canvas, L = entropy.shape
    ws_bytes = workspace.numel() * workspace.element_size()
    rc = load().dg_denoise_accept(_p(entropy), _p(sample), _p(argmax), n_canvas, L, V, _p(params),
                                  int(seed) & 0xFFFFFFFFFFFFFFFF, _p(canvas), _p(prev_argmax), _p(stable_count),
                                  _p(accept_mask), _p(converged), _p(mean_entropy), _p(n_accept),
                                  _p(workspace), ws_bytes, _s(stream))
    if check:
        _check("dg_denoise_accept", rc)
    return rc


def dg_denoise_samples(logits, params, seed, canvas, sample, workspace, *, n_canvas=None, L=None,
                       V=None, ld=None, stream=None, check=True) -> int:
    n_canvas, L, V, ld = _denoise_dims(logits, n_canvas, L, V, ld)
    ws_bytes = workspace.numel() * workspace.element_size()
    rc = load().dg_denoise_samples(_p(logits), _dtype_code(logits), ld, n_canvas, L, V, _p(params),
                                   int(seed) & 0xFFFFFFFFFFFFFFFF, _p(canvas), _p(sample),
                                   _p(workspace), ws_bytes, _s(stream))
    if check:
        _check("dg_denoise_samples", rc)
    return rc


def dg_accept_from_entropy(entropy, sample, argmax, n_canvas, L, V, params, seed, canvas,
                           prev_argmax, stable_count, accept_mask, converged, mean_entropy=None,
                           n_accept=None, stream=None, check=True) -> int:
    rc = load().dg_accept_from_entropy(_p(entropy), _p(sample), _p(argmax), n_canvas, L, V,
                                       _p(params), int(seed) & 0xFFFFFFFFFFFFFFFF, _p(canvas),
                                       _p(prev_argmax), _p(stable_count), _p(accept_mask),
                                       _p(converged), _p(mean_entropy), _p(n_accept), _s(stream))
    if check:
        _check("dg_accept_from_entropy", rc)
    return rc


def dg_lm_head_workspace_bytes(n_canvas: int, L: int, V: int) -> int:
    return int(load().dg_lm_head_workspace_bytes(n_canvas, L, V))


def _lm_dims(hidden, W_lm, logits, V):
    n, L, ldh = hidden.shape
    d = W_lm.shape[1] if W_lm.dim() == 2 else None
    if hidden.stride(2) != 1 or W_lm.stride(1) != 1 or logits.stride(2) != 1:
        raise ValueError("rows must be contiguous")
    if hidden.stride(0) != L * hidden.stride(1) or logits.stride(0) != L * logits.stride(1):
        raise ValueError("canvases must follow each other at L row strides")
    V = W_lm.shape[0] if V is None else V
    return n, L, V, d, hidden.stride(1), W_lm.stride(0), logits.stride(1)


def dg_lm_head_logits(hidden, W_lm, params, logits, workspace=None, *, V=None, stream=None,
                      check=True) -> int:
    """logits[n, L, ld] = bf16(hidden[n, L, d] . W_lm[V, d]^T) for the active canvases."""
    n, L, V, d, ldh, ldw, ld = _lm_dims(hidden, W_lm, logits, V)
    if workspace is None:
        workspace = torch.empty(dg_lm_head_workspace_bytes(n, L, V), dtype=torch.uint8, device=hidden.device)
    rc = load().dg_lm_head_logits(_p(hidden), ldh, _p(W_lm), ldw, n, L, V, d, _p(params), _p(logits), ld,
                                  _p(workspace), workspace.numel(), _s(stream))
    if check:
        _check("dg_lm_head_logits", rc)
    return rc


def dg_lm_head_denoise_step(hidden, W_lm, params, seed, logits, canvas, prev_argmax, stable_count,
                            accept_mask, argmax, sample, entropy, lse, converged, mean_entropy=None,
                            n_accept=None, workspace=None, *, V=None, stream=None, check=True) -> int:
    """The LM head (logits stored into ``logits``) and one denoising step on its logits."""
    n, L, V, d, ldh, ldw, ld = _lm_dims(hidden, W_lm, logits, V)
    if workspace is None:
        workspace = torch.empty(dg_lm_head_workspace_bytes(n, L, V), dtype=torch.uint8, device=hidden.device)
    rc = load().dg_lm_head_denoise_step(_p(hidden), ldh, _p(W_lm), ldw, n, L, V, d, _p(params),
                                        int(seed) & 0xFFFFFFFFFFFFFFFF, _p(logits), ld, _p(canvas),
                                        _p(prev_argmax), _p(stable_count), _p(accept_mask), _p(argmax),
                                        _p(sample), _p(entropy), _p(lse), _p(converged), _p(mean_entropy),
                                        _p(n_accept), _p(workspace), workspace.numel(), _s(stream))
    if check:
        _check("dg_lm_head_denoise_step", rc)
    return rc


def dg_canvas_init(canvas, n_canvas, L, V, params, seed, stream=None, check=True) -> int:
    rc = load().dg_canvas_init(_p(canvas), n_canvas, L, V, _p(params),
                               int(seed) & 0xFFFFFFFFFFFFFFFF, _s(stream))
    if check:
        _check("dg_canvas_init", rc)
    return rc


def dg_advance_params(params, converged, n_canvas, stream=None, check=True) -> int:
    rc = load().dg_advance_params(_p(params), _p(converged), n_canvas, _s(stream))
    if check:
        _check("dg_advance_params", rc)
    return rc


def dg_choice_probs(logits, lse, params, choices, probs, *, V=None, stream=None, check=True) -> int:
    """probs[c, i, k] = exp(logits[c, i, choices[c, i, k]] / T - lse[c, i]); logits [n, L, ld]."""
    n, L, ld = logits.shape
    C = choices.shape[-1]
    rc = load().dg_choice_probs(_p(logits), _dtype_code(logits), ld, _p(lse), _p(params), n, L,
                                ld if V is None else V, _p(choices), C, _p(probs), _s(stream))
    if check:
        _check("dg_choice_probs", rc)
    return rc


def dg_attention_workspace_bytes(n_seq: int, max_q_len: int) -> int:
    return int(load().dg_attention_workspace_bytes(n_seq, max_q_len))


def dg_attention(q, k, v, o, cu_q, cu_kv, causal, max_q_len: int, *, lse=None, window: int = -1,
                 scale: float | None = None, workspace=None, stream=None, check=True) -> int:
    """o = attention over the allowed keys (per-sequence causality, optional symmetric window);
    q [total_q, Hq, D], k / v [total_kv, Hkv, D], o like q (bf16); cu_q / cu_kv [n + 1] int32 and
    causal [n] uint8 on the device."""
    total_q, Hq, D = q.shape
    total_kv, Hkv, _ = k.shape
    for t in (q, k, v, o):
        if not t.is_contiguous():
            raise ValueError("q, k, v and o must be contiguous")
    n = causal.numel()
    scale = 1.0 / float(D) ** 0.5 if scale is None else float(scale)
    if workspace is None:
        workspace = torch.empty(max(1, dg_attention_workspace_bytes(n, int(max_q_len))), dtype=torch.uint8,
                                device=q.device)
    rc = load().dg_attention(_p(q), _p(k), _p(v), _p(o), _p(lse), _p(cu_q), _p(cu_kv), _p(causal), n,
                             int(max_q_len), total_q, total_kv, Hq, Hkv, D, int(window), scale, _p(workspace),
                             workspace.numel(), _s(stream))
    if check:
        _check("dg_attention", rc)
    return rc


def dg_embed_canvas(canvas, E, delta_emb, out, scale: float = 1.0, stream=None, check=True) -> int:
    """out = bf16(fma(scale, E[canvas], delta_emb)); canvas [..] int32, E [V, d], out [.., d]."""
    V, d = E.shape
    rc = load().dg_embed_canvas(_p(canvas), canvas.numel(), V, _p(E), d, _p(delta_emb), float(scale),
                                _p(out), _s(stream))
    if check:
        _check("dg_embed_canvas", rc)
    return rc


def dg_commit(params, converged, argmax, tokens, prev_argmax, stable_count, committed, stream=None,
              check=True) -> int:
    n, L = argmax.shape
    rc = load().dg_commit(_p(params), _p(converged), _p(argmax), n, L, _p(tokens), _p(prev_argmax),
                          _p(stable_count), _p(committed), _s(stream))
    if check:
        _check("dg_commit", rc)
    return rc


def dg_self_cond_workspace_bytes(n_canvas: int, L: int, d: int, h: int) -> int:
    return int(load().dg_self_cond_workspace_bytes(n_canvas, L, d, h))


def dg_self_cond_logits(logits, lse, params, converged, E, W_gate, W_up, W_down, delta_emb,
                        workspace, *, n_canvas=None, L=None, V=None, ld=None, stream=None,
                        check=True) -> int:
    n, Lx, ldx = logits.shape if logits.dim() == 3 else (n_canvas, L, ld)
    n_canvas = n if n_canvas is None else n_canvas
    L = Lx if L is None else L
    ld = ldx if ld is None else ld
    V = ld if V is None else V
    d = E.shape[1]
    h = W_gate.shape[0]
    ws_bytes = workspace.numel() * workspace.element_size()
    rc = load().dg_self_cond_logits(_p(logits), _dtype_code(logits), ld, _p(lse), _p(params),
                                    _p(converged), n_canvas, L, V, d, h, _p(E), _p(W_gate),
                                    _p(W_up), _p(W_down), _p(delta_emb), _p(workspace), ws_bytes,
                                    _s(stream))
    if check:
        _check("dg_self_cond_logits", rc)
    return rc


def dg_self_cond_prepare(params, converged, n_canvas, L, d, h, delta_emb, workspace, stream=None,
                         check=True) -> int:
    ws_bytes = workspace.numel() * workspace.element_size()
    rc = load().dg_self_cond_prepare(_p(params), _p(converged), n_canvas, L, d, h, _p(delta_emb),
                                     _p(workspace), ws_bytes, _s(stream))
    if check:
        _check("dg_self_cond_prepare", rc)
    return rc


def dg_self_cond_pe(logits, lse, params, E, h, workspace, *, n_canvas=None, L=None, V=None, ld=None,
                    stream=None, check=True) -> int:
    n, Lx, ldx = logits.shape if logits.dim() == 3 else (n_canvas, L, ld)
    n_canvas = n if n_canvas is None else n_canvas
    L = Lx if L is None else L
    ld = ldx if ld is None else ld
    V = ld if V is None else V
    ws_bytes = workspace.numel() * workspace.element_size()
    rc = load().dg_self_cond_pe(_p(logits), _dtype_code(logits), ld, _p(lse), _p(params), n_canvas, L, V,
                                E.shape[1], h, _p(E), _p(workspace), ws_bytes, _s(stream))
    if check:
        _check("dg_self_cond_pe", rc)
    return rc


def dg_self_cond_mlp(n_canvas, L, W_gate, W_up, W_down, delta_emb, workspace, stream=None,
                     check=True) -> int:
    d = W_gate.shape[1]
    h = W_gate.shape[0]
    ws_bytes = workspace.numel() * workspace.element_size()
    rc = load().dg_self_cond_mlp(n_canvas, L, d, h, _p(W_gate), _p(W_up), _p(W_down), _p(delta_emb),
                                 _p(workspace), ws_bytes, _s(stream))
    if check:
        _check("dg_self_cond_mlp", rc)
    return rc


def dg_self_cond_zero_converged(params, converged, delta_emb, stream=None, check=True) -> int:
    """Zero the feedback rows of canvases that got feedback and converged (delta_emb [n, L, d])."""
    n_canvas, L, d = delta_emb.shape
    rc = load().dg_self_cond_zero_converged(_p(params), _p(converged), n_canvas, L, d, _p(delta_emb), _s(stream))
    if check:
        _check("dg_self_cond_zero_converged", rc)
    return rc


def dg_self_cond_probs_workspace_bytes(n_rows: int, d: int, h: int) -> int:
    return int(load().dg_self_cond_probs_workspace_bytes(n_rows, d, h))


def dg_self_cond_probs(P, E, W_gate, W_up, W_down, delta_emb, workspace, *, V=None, stream=None,
                       check=True) -> int:
    n_rows, ld = P.shape
    V = ld if V is None else V
    d = E.shape[1]
    h = W_gate.shape[0]
    ws_bytes = workspace.numel() * workspace.element_size()
    rc = load().dg_self_cond_probs(_p(P), ld, n_rows, V, d, h, _p(E), _p(W_gate), _p(W_up),
                                   _p(W_down), _p(delta_emb), _p(workspace), ws_bytes, _s(stream))
    if check:
        _check("dg_self_cond_probs", rc)
    return rc


def dg_gemm_workspace_bytes(M: int, N: int) -> int:
    return int(load().dg_gemm_workspace_bytes(M, N))


def dg_gemm_bf16(A, B, C, b_mn_major: bool, workspace, *, M=None, N=None, K=None, stream=None,
                 check=True) -> int:
    M = A.shape[0] if M is None else M
    K = A.shape[1] if K is None else K
    N = (B.shape[1] if b_mn_major else B.shape[0]) if N is None else N
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load().dg_gemm_bf16(_p(A), A.stride(0), _p(B), B.stride(0), int(bool(b_mn_major)), _p(C),
                             C.stride(0), M, N, K, _p(workspace), ws_bytes, _s(stream))
    if check:
        _check("dg_gemm_bf16", rc)
    return rc


def dg_gemm_bf16_noalloc(A, B, C, b_mn_major: bool, *, M=None, N=None, K=None, stream=None,
                         check=True) -> int:
    M = A.shape[0] if M is None else M
    K = A.shape[1] if K is None else K
    N = (B.shape[1] if b_mn_major else B.shape[0]) if N is None else N
    rc = load().dg_gemm_bf16_noalloc(_p(A), A.stride(0), _p(B), B.stride(0), int(bool(b_mn_major)), _p(C),
                                     C.stride(0), M, N, K, _s(stream))
    if check:
        _check("dg_gemm_bf16_noalloc", rc)
    return rc


def dg_philox_words(seed, request_id, step, position, stream_id, block0, n_blocks, out,
                    stream=None, check=True) -> int:
    rc = load().dg_philox_words(int(seed) & 0xFFFFFFFFFFFFFFFF, request_id, step, position,
                                stream_id, block0, n_blocks, _p(out), _s(stream))
    if check:
        _check("dg_philox_words", rc)
    return rc


def dg_get_device_status(stream=None) -> int:
    v = ctypes.c_uint32(0)
    _check("dg_get_device_status", load().dg_get_device_status(_s(stream), ctypes.byref(v)))
    return int(v.value)


def dg_clear_device_status(stream=None) -> None:
    _check("dg_clear_device_status", load().dg_clear_device_status(_s(stream)))


def dg_probe_bounded_wait(polls, result, stream=None, check=True) -> int:
    rc = load().dg_probe_bounded_wait(int(polls), _p(result), _s(stream))
    if check:
        _check("dg_probe_bounded_wait", rc)
    return rc
