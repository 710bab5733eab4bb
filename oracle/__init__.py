"""fp64 CPU oracle of the entropy-bounded denoising step (ctypes front end).

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` are the only callers.  The oracle shares no code with the CUDA
library; both read the same seeded inputs from ``entropy_bounded_denoising_gb300.synth``.

The arithmetic lives in ``dg_oracle.c`` (plain fp64 C, one row at a time, OpenMP only
across independent rows).  This module compiles it with gcc on first use (or via
``build()``) and marshals numpy arrays.  Every function cites its source in the C file:
the DiffusionGemma vLLM page ("DiffusionGemma: vLLM이 네이티브로 지원하는 최초의 디퓨전
언어 모델(dLLM)"), sections "엔트로피 기반 디노이징", "자기 조건화" and
"DiffusionGemmaModelState와 DiffusionSampler".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dg_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libdg_oracle.so")
_lock = threading.Lock()
_lib = None

ACTIVE, READ_ONLY, SELF_COND = 1, 2, 4
STREAM_GUMBEL, STREAM_RENOISE, STREAM_INIT = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/libdg_oracle.so`` (plain gcc, fp64, no fast-math)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=gnu11", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P, i32, i64, u32, u64, dbl = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64,
                                       ctypes.c_uint32, ctypes.c_uint64, ctypes.c_double)
        lib.orc_philox4x32.argtypes = [P, P, ctypes.c_int, P]
        lib.orc_uniform.argtypes = [u32]
        lib.orc_uniform.restype = dbl
        lib.orc_token.argtypes = [u32, u32, u32]
        lib.orc_token.restype = u32
        lib.orc_gumbel.argtypes = [u64, u32, u32, u32, u32]
        lib.orc_gumbel.restype = dbl
        lib.orc_random_token.argtypes = [u64, u32, u32, u32, u32, u32]
        lib.orc_random_token.restype = u32
        lib.orc_row_stats.argtypes = [P, ctypes.c_int, i64, dbl, u64, u32, u32, u32, ctypes.c_int, P]
        lib.orc_accept.argtypes = [P, i32, dbl, i32, P, P, P, P]
        lib.orc_accept.restype = i32
        lib.orc_denoise_step.argtypes = [P, ctypes.c_int, i64, i64, i32, i64] + [P] * 9 + [u64] + [P] * 15 + [ctypes.c_int]
        lib.orc_canvas_init.argtypes = [P, i64, i32, i64, P, P, P, u64]
        lib.orc_gelu_tanh.argtypes = [dbl]
        lib.orc_gelu_tanh.restype = dbl
        lib.orc_pe_from_probs.argtypes = [P, i64, i64, i32, P, P, ctypes.c_int]
        lib.orc_gated_mlp.argtypes = [P, i64, i32, i32, P, P, P, P, ctypes.c_int]
        lib.orc_probs_from_logits.argtypes = [P, ctypes.c_int, i64, i64, i64, P, P, ctypes.c_int]
        lib.orc_choice_probs.argtypes = [P, ctypes.c_int, i64, i64, i64, P, P, i32, P, ctypes.c_int]
        lib.orc_bf16_round.argtypes = [ctypes.c_float]
        lib.orc_bf16_round.restype = ctypes.c_uint16
        lib.orc_embed_canvas.argtypes = [P, i64, i64, P, i32, P, ctypes.c_float, P]
        lib.orc_commit.argtypes = [P, P, P, i64, i32, P, P, P, P]
        lib.orc_bf16_round_f64.argtypes = [dbl]
        lib.orc_bf16_round_f64.restype = ctypes.c_uint16
        lib.orc_lm_head_logits.argtypes = [P, i64, i32, i64, P, i64, i64, P, i64, P, P, ctypes.c_int]
        lib.orc_attn_allowed.argtypes = [ctypes.c_int, i64, i64, i64, i64]
        lib.orc_attn_allowed.restype = ctypes.c_int
        lib.orc_attention.argtypes = [P, P, P, P, P, P, i32, i32, i32, i32, i64, dbl, P, P, ctypes.c_int]
        lib.orc_max_threads.restype = ctypes.c_int
        _lib = lib
        return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def max_threads() -> int:
    return int(_load().orc_max_threads())


# ---------------------------------------------------------------- random numbers
def philox4x32(ctr, key, rounds: int = 10) -> np.ndarray:
    lib = _load()
    c = _c(ctr, np.uint32)
    k = _c(key, np.uint32)
    out = np.zeros(4, np.uint32)
    lib.orc_philox4x32(_ptr(c), _ptr(k), int(rounds), _ptr(out))
    return out


def uniform(w: int) -> float:
    return float(_load().orc_uniform(int(w) & 0xFFFFFFFF))


def token(w0: int, w1: int, V: int) -> int:
    return int(_load().orc_token(int(w0) & 0xFFFFFFFF, int(w1) & 0xFFFFFFFF, int(V)))


def gumbel(seed: int, request_id: int, step: int, position: int, v: int) -> float:
    return float(_load().orc_gumbel(int(seed), int(request_id), int(step), int(position), int(v)))


def random_token(seed: int, request_id: int, step: int, position: int, stream: int, V: int) -> int:
    return int(_load().orc_random_token(int(seed), int(request_id), int(step), int(position),
                                        int(stream), int(V)))


# ---------------------------------------------------------------- per-row statistics
class _RowResult(ctypes.Structure):
    _fields_ = [("entropy", ctypes.c_double), ("entropy_alt", ctypes.c_double),
                ("lse", ctypes.c_double), ("score1", ctypes.c_double), ("score2", ctypes.c_double),
                ("argmax", ctypes.c_int32), ("sample", ctypes.c_int32),
                ("nonfinite", ctypes.c_int32), ("pad", ctypes.c_int32)]


def _dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.uint16:   # bf16 bit patterns
        return 0
    if a.dtype == np.float32:
        return 1
    raise TypeError("logits must be bf16 bit patterns (uint16) or float32")


def row_stats(row, T: float = 1.0, seed: int = 0, request_id: int = 0, step: int = 0,
              position: int = 0, sample: bool = True) -> dict:
    """Statistics of one canvas position (entropy, lse, argmax, Gumbel-max sample)."""
    lib = _load()
    r = np.ascontiguousarray(row)
    res = _RowResult()
    lib.orc_row_stats(_ptr(r), _dtype_code(r), r.shape[-1], float(T), int(seed), int(request_id),
                      int(step), int(position), int(bool(sample)), ctypes.byref(res))
    return {f: getattr(res, f) for f, _ in _RowResult._fields_ if f != "pad"}


def accept(H, beta: float, min_accept: int = 1) -> dict:
    """Entropy-bound acceptance on given entropies (fp64)."""
    lib = _load()
    h = _c(H, np.float64)
    L = h.shape[0]
    mask = np.zeros(L, np.uint8)
    order = np.zeros(L, np.int32)
    cg = ctypes.c_double()
    bg = ctypes.c_double()
    n = lib.orc_accept(_ptr(h), L, float(beta), int(min_accept), _ptr(mask), _ptr(order),
                       ctypes.byref(cg), ctypes.byref(bg))
    return {"n_accept": int(n), "mask": mask, "order": order,
            "cut_gap": cg.value, "budget_gap": bg.value}


# ---------------------------------------------------------------- one denoise step
def denoise_step(logits, params: dict, seed: int, canvas, prev_argmax, stable_count,
                 ld: int | None = None, V: int | None = None, n_threads: int = 0) -> dict:
    """One denoise step over n canvases.

    logits: [n, L, ld] uint16 (bf16 bits) or float32.  params: dict of per-canvas arrays
    temperature, beta, tau (float), k, max_steps, min_accept, step (int32),
    request_id, flags (uint32).  canvas / prev_argmax [n, L] int32 and stable_count [n]
    int32 are updated in place (on copies returned in the result)."""
    lib = _load()
    x = np.ascontiguousarray(logits)
    n, L, ldx = x.shape
    ld = ldx if ld is None else ld
    V = ld if V is None else V
    dt = _dtype_code(x)
    T = _c(params["temperature"], np.float32)
    beta = _c(params["beta"], np.float32)
    tau = _c(params["tau"], np.float32)
    k = _c(params["k"], np.int32)
    S = _c(params["max_steps"], np.int32)
    mina = _c(params["min_accept"], np.int32)
    step = _c(params["step"], np.int32)
    req = _c(params["request_id"], np.uint32)
    flags = _c(params["flags"], np.uint32)
    canvas = _c(canvas, np.int32).copy()
    prev = _c(prev_argmax, np.int32).copy()
    stable = _c(stable_count, np.int32).copy()
    out = {
        "accept_mask": np.zeros((n, L), np.uint8), "argmax": np.zeros((n, L), np.int32),
        "sample": np.zeros((n, L), np.int32), "entropy": np.zeros((n, L), np.float64),
        "lse": np.zeros((n, L), np.float64), "converged": np.zeros(n, np.uint8),
        "mean_entropy": np.zeros(n, np.float64), "n_accept": np.zeros(n, np.int32),
        "sample_gap": np.full((n, L), np.inf), "cut_gap": np.full(n, np.inf),
        "budget_gap": np.full(n, np.inf), "tau_gap": np.full(n, np.inf),
    }
    lib.orc_denoise_step(_ptr(x), dt, ld, n, L, V, _ptr(T), _ptr(beta), _ptr(tau), _ptr(k),
                         _ptr(S), _ptr(mina), _ptr(step), _ptr(req), _ptr(flags), int(seed),
                         _ptr(canvas), _ptr(prev), _ptr(stable),
                         _ptr(out["accept_mask"]), _ptr(out["argmax"]), _ptr(out["sample"]),
                         _ptr(out["entropy"]), _ptr(out["lse"]), _ptr(out["converged"]),
                         _ptr(out["mean_entropy"]), _ptr(out["n_accept"]),
                         _ptr(out["sample_gap"]), _ptr(out["cut_gap"]), _ptr(out["budget_gap"]),
                         _ptr(out["tau_gap"]), int(n_threads))
    out.update(canvas=canvas, prev_argmax=prev, stable_count=stable)
    return out


def canvas_init(n: int, L: int, V: int, params: dict, seed: int) -> np.ndarray:
    lib = _load()
    canvas = np.zeros((n, L), np.int32)
    step = _c(params["step"], np.int32)
    req = _c(params["request_id"], np.uint32)
    flags = _c(params["flags"], np.uint32)
    lib.orc_canvas_init(_ptr(canvas), n, L, V, _ptr(step), _ptr(req), _ptr(flags), int(seed))
    return canvas


# ---------------------------------------------------------------- self-conditioning
def gelu_tanh(z: float) -> float:
    return float(_load().orc_gelu_tanh(float(z)))


def probs_from_logits(rows, T_rows, V: int | None = None, n_threads: int = 0) -> np.ndarray:
    """P = softmax(x / T) per row, fp64.  rows: [r, ld] bf16 bits or float32."""
    lib = _load()
    x = np.ascontiguousarray(rows)
    r, ld = x.shape
    V = ld if V is None else V
    T = _c(np.broadcast_to(np.asarray(T_rows, np.float64), (r,)), np.float64)
    P = np.zeros((r, V), np.float64)
    lib.orc_probs_from_logits(_ptr(x), _dtype_code(x), ld, r, V, _ptr(T), _ptr(P), int(n_threads))
    return P


def pe_from_probs(P, E_bf16, n_threads: int = 0) -> np.ndarray:
    """pe = P . E with E given as bf16 bit patterns [V, d]."""
    lib = _load()
    p = _c(P, np.float64)
    E = _c(E_bf16, np.uint16)
    r, V = p.shape
    d = E.shape[1]
    assert E.shape[0] == V
    pe = np.zeros((r, d), np.float64)
    lib.orc_pe_from_probs(_ptr(p), r, V, d, _ptr(E), _ptr(pe), int(n_threads))
    return pe


def gated_mlp(pe, W_gate, W_up, W_down, n_threads: int = 0) -> np.ndarray:
    """delta = W_down (gelu_tanh(W_gate pe) * (W_up pe)); W as bf16 bits, [h,d],[h,d],[d,h]."""
    lib = _load()
    z = _c(pe, np.float64)
    r, d = z.shape
    Wg = _c(W_gate, np.uint16)
    Wu = _c(W_up, np.uint16)
    Wd = _c(W_down, np.uint16)
    h = Wg.shape[0]
    assert Wg.shape == (h, d) and Wu.shape == (h, d) and Wd.shape == (d, h)
    out = np.zeros((r, d), np.float64)
    lib.orc_gated_mlp(_ptr(z), r, d, h, _ptr(Wg), _ptr(Wu), _ptr(Wd), _ptr(out), int(n_threads))
    return out


def self_cond_rows(rows, T_rows, E_bf16, W_gate, W_up, W_down, V: int | None = None,
                   n_threads: int = 0) -> np.ndarray:
    """Self-conditioning delta for logit rows: gated MLP of softmax(x / T) . E."""
    P = probs_from_logits(rows, T_rows, V=V, n_threads=n_threads)
    return gated_mlp(pe_from_probs(P, E_bf16, n_threads), W_gate, W_up, W_down, n_threads)


# ---------------------------------------------------------------- single-pass reads
def choice_probs(rows, T_rows, choices, V: int | None = None, n_threads: int = 0) -> np.ndarray:
    """p = exp(x_tok / T - lse) for caller-given tokens per row (fp64); tokens outside
    [0, V) give 0.  rows: [r, ld] bf16 bits or float32; choices: [r, C] int32."""
    lib = _load()
    x = np.ascontiguousarray(rows)
    r, ld = x.shape
    V = ld if V is None else V
    T = _c(np.broadcast_to(np.asarray(T_rows, np.float64), (r,)), np.float64)
    ch = _c(choices, np.int32)
    C = ch.shape[1]
    assert ch.shape[0] == r
    out = np.zeros((r, C), np.float64)
    lib.orc_choice_probs(_ptr(x), _dtype_code(x), ld, r, V, _ptr(T), _ptr(ch), C, _ptr(out), int(n_threads))
    return out


# ---------------------------------------------------------------- step-after glue
def bf16_round(f: float) -> int:
    """Round-to-nearest-even of an fp32 value to a bf16 bit pattern."""
    return int(_load().orc_bf16_round(float(np.float32(f))))


def embed_canvas(canvas, E_bf16, delta_bf16=None, scale: float = 1.0) -> np.ndarray:
    """emb = bf16(fma(scale, E[canvas], delta)) as bf16 bit patterns [rows, d]."""
    lib = _load()
    cv = _c(canvas, np.int32).reshape(-1)
    E = _c(E_bf16, np.uint16)
    V, d = E.shape
    dl = None if delta_bf16 is None else _c(delta_bf16, np.uint16).reshape(-1, d)
    out = np.zeros((cv.shape[0], d), np.uint16)
    lib.orc_embed_canvas(_ptr(cv), cv.shape[0], V, _ptr(E), d, _ptr(dl), float(scale), _ptr(out))
    return out


def commit(converged, active, argmax, tokens, prev_argmax, stable_count) -> dict:
    """Commit of converged active canvases: tokens = argmax, state reset (copies returned)."""
    lib = _load()
    cv = _c(converged, np.uint8)
    ac = _c(active, np.uint8)
    am = _c(argmax, np.int32)
    n, L = am.shape
    tok = _c(tokens, np.int32).copy()
    prev = _c(prev_argmax, np.int32).copy()
    st = _c(stable_count, np.int32).copy()
    committed = np.zeros(n, np.uint8)
    lib.orc_commit(_ptr(cv), _ptr(ac), _ptr(am), n, L, _ptr(tok), _ptr(prev), _ptr(st), _ptr(committed))
    return {"tokens": tok, "prev_argmax": prev, "stable_count": st, "committed": committed}


# ---------------------------------------------------------------- LM head
def bf16_round_f64(x: float) -> int:
    """The bf16 bit pattern nearest to a double (ties to even), rounded once."""
    return int(_load().orc_bf16_round_f64(float(x)))


def lm_head_logits(hidden_bf16, W_bf16, V: int | None = None, ld: int | None = None,
                   exact: bool = False, n_threads: int = 0):
    """logits = bf16(hidden . W^T): hidden [rows, d] and W [V, d] as bf16 bit patterns.
    Returns the logits as bf16 bits [rows, ld] (columns past V are 0); with exact=True also
    the unrounded fp64 dot products and sum_j |h_j W_vj|, each [rows, V]."""
    lib = _load()
    h = _c(hidden_bf16, np.uint16)
    W = _c(W_bf16, np.uint16)
    rows, d = h.shape
    V = W.shape[0] if V is None else V
    assert W.shape[1] == d and W.shape[0] >= V
    ld = V if ld is None else ld
    out = np.zeros((rows, ld), np.uint16)
    ex = np.zeros((rows, V), np.float64) if exact else None
    ab = np.zeros((rows, V), np.float64) if exact else None
    lib.orc_lm_head_logits(_ptr(h), rows, d, d, _ptr(W), V, d, _ptr(out), ld, _ptr(ex), _ptr(ab), int(n_threads))
    return (out, ex, ab) if exact else out


# ---------------------------------------------------------------- attention
def attn_allowed(causal: bool, window: int, pos: int, j: int, kv_len: int) -> bool:
    """Whether query position `pos` may attend to key j (window < 0: no window)."""
    return bool(_load().orc_attn_allowed(int(bool(causal)), int(window), int(pos), int(j), int(kv_len)))


def attention(q_bf16, k_bf16, v_bf16, cu_q, cu_kv, causal, window: int = -1, scale: float | None = None,
              n_threads: int = 0):
    """Attention with per-sequence causality and an optional symmetric window (fp64).
    q [total_q, Hq, D], k / v [total_kv, Hkv, D] as bf16 bit patterns; cu_q / cu_kv [n + 1]
    int32 offsets; causal [n] flags.  Returns (o [total_q, Hq, D], lse [total_q, Hq])."""
    lib = _load()
    q = _c(q_bf16, np.uint16)
    k = _c(k_bf16, np.uint16)
    v = _c(v_bf16, np.uint16)
    total_q, Hq, D = q.shape
    Hkv = k.shape[1]
    assert k.shape == v.shape and k.shape[2] == D and Hq % Hkv == 0
    cq = _c(cu_q, np.int32)
    ck = _c(cu_kv, np.int32)
    cz = _c(causal, np.uint8)
    n = cz.shape[0]
    scale = 1.0 / np.sqrt(D) if scale is None else float(scale)
    o = np.zeros((total_q, Hq, D), np.float64)
    lse = np.zeros((total_q, Hq), np.float64)
    lib.orc_attention(_ptr(q), _ptr(k), _ptr(v), _ptr(cq), _ptr(ck), _ptr(cz), n, Hq, Hkv, D, int(window),
                      scale, _ptr(o), _ptr(lse), int(n_threads))
    return o, lse
