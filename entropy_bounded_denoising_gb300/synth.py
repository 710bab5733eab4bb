"""Seeded synthetic inputs for the denoising step: logits, embedding table, MLP weights and
per-canvas parameters.

This module holds none of the method's arithmetic.  Both the CUDA path and the fp64 oracle
read the bytes it produces, so it is the only code the two sides share.

Workload recipe (the pages publish no logit statistics, so the shapes follow the five
workloads this library is measured on):
  * base_v = s_i * z_v with z ~ N(0, 1) per vocabulary entry and a per-position scale
    s_i ~ U[lo, hi] that spreads the entropies from near-uniform to near-one-hot;
  * step t (0-based) sees logits base * (1 + 0.5 t) + 0.1 * n_t, n_t ~ N(0, 1) fresh per
    step, so the distributions sharpen and the canvas converges;
  * optionally a fraction of positions is made near one-hot by setting one random token
    to (row max + 20) after the step's logits are formed;
  * computed in fp32 and rounded to bf16 (or kept fp32);
  * E, W_gate, W_up, W_down ~ N(0, 0.02^2), rounded to bf16;
  * for the LM head, hidden states h_i = s_i z / (0.02 sqrt(d)) with z ~ N(0, 1), so that
    hidden . E^T has the same per-position spread s_i; or small-integer operands (k / 8,
    |k| <= 12 for hidden, <= 4 for W) whose dot products fp32 sums exactly;
  * for attention, q ~ N(0, s_t^2) per token with s_t ~ U[0.5, 4] (scores from flat to peaked
    at the scale 1/sqrt(D)), k and v ~ N(0, 1), all bf16.
Every draw comes from a torch generator seeded from (seed, purpose, canvas), so the bytes
do not depend on how canvases are chunked; CPU and CUDA generators give different (each
reproducible) streams, and a test always hands the same bytes to both sides.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

ACTIVE, READ_ONLY, SELF_COND, SAMPLE_ALL = 1, 2, 4, 8

# purposes for seeding (arbitrary distinct constants)
_P_BASE, _P_SCALE, _P_NOISE, _P_SPIKE, _P_WEIGHT, _P_PARAMS, _P_HIDDEN, _P_ATTN = 11, 23, 37, 41, 53, 67, 79, 83


def _gen(device, *parts: int) -> torch.Generator:
    seed = 0x9E3779B97F4A7C15
    for p in parts:
        seed = (seed * 6364136223846793005 + (int(p) & 0xFFFFFFFFFFFFFFFF) + 1442695040888963407) \
            & 0xFFFFFFFFFFFFFFFF
    g = torch.Generator(device=device)
    g.manual_seed(seed & 0x7FFFFFFFFFFFFFFF)
    return g


@dataclasses.dataclass
class Workload:
    name: str
    n: int
    L: int
    V: int
    d: int
    h: int
    dtype: str               # "bf16" or "fp32"
    scale: tuple             # (lo, hi) of s_i
    seed: int
    spike_frac: float = 0.0  # fraction of near-one-hot positions (+20 over the row max)
    full_loop: bool = True
    steps: int = 1           # step cap S for normal canvases


WORKLOADS = {
    "tiny": Workload("tiny", 1, 16, 1024, 64, 128, "fp32", (0.5, 8.0), 0, steps=8),
    "single": Workload("single", 1, 256, 32768, 2048, 8192, "bf16", (0.5, 12.0), 1, steps=32),
    "batched": Workload("batched", 8, 256, 262144, 4096, 16384, "bf16", (0.5, 12.0), 2,
                        spike_frac=0.10, full_loop=False, steps=64),
    "sweep": Workload("sweep", 64, 256, 262144, 4096, 16384, "bf16", (0.5, 12.0), 3, steps=64),
    "ragged": Workload("ragged", 32, 256, 152064, 3584, 18944, "bf16", (0.5, 12.0), 4,
                       full_loop=False, steps=64),
    # reduced case for profiler captures: the batched kernels' shapes with half the
    # vocabulary and half the canvases (inputs still larger than L2, ~1.5 GB on the device)
    "profile": Workload("profile", 4, 256, 131072, 4096, 16384, "bf16", (0.5, 12.0), 5,
                        spike_frac=0.10, full_loop=False, steps=64),
}


def logits(n: int, L: int, V: int, *, seed: int, step: int = 0, scale=(0.5, 8.0),
           spike_frac: float = 0.0, dtype: str = "bf16", ld: int | None = None,
           device="cpu", canvases=None) -> torch.Tensor:
    """Logits [n, L, ld] for one step (ld >= V; padding columns hold +1000, never valid data).

    ``canvases`` (optional list of canvas indices) generates only those canvases, with the
    same bytes they have in the full tensor."""
    ld = V if ld is None else ld
    assert ld >= V
    idx = list(range(n)) if canvases is None else list(canvases)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    out = torch.empty((len(idx), L, ld), dtype=tdt, device=device)
    if ld > V:
        out[:, :, V:] = 1000.0
    for j, c in enumerate(idx):
        z = torch.randn((L, V), generator=_gen(device, seed, _P_BASE, c), device=device)
        s = torch.empty((L, 1), device=device).uniform_(scale[0], scale[1],
                                                        generator=_gen(device, seed, _P_SCALE, c))
        x = z.mul_(s).mul_(1.0 + 0.5 * step)
        x.add_(torch.randn((L, V), generator=_gen(device, seed, _P_NOISE, c, step), device=device),
               alpha=0.1)
        if spike_frac > 0.0:
            g = _gen(device, seed, _P_SPIKE, c)
            pick = torch.rand((L,), generator=g, device=device) < spike_frac
            tok = torch.randint(0, V, (L,), generator=g, device=device)
            rows = torch.nonzero(pick).flatten()
            if rows.numel():
                rmax = x[rows].amax(dim=1)
                x[rows, tok[rows]] = rmax + 20.0
        out[j, :, :V] = x.to(tdt)
        del x, z
    return out


def weights(V: int, d: int, h: int, *, seed: int, device="cpu"):
    """E [V, d], W_gate [h, d], W_up [h, d], W_down [d, h] in bf16, entries ~ N(0, 0.02^2)."""
    def w(shape, purpose):
        t = torch.randn(shape, generator=_gen(device, seed, _P_WEIGHT, purpose), device=device)
        return t.mul_(0.02).to(torch.bfloat16)
    return w((V, d), 1), w((h, d), 2), w((h, d), 3), w((d, h), 4)


def hidden_states(n: int, L: int, d: int, *, seed: int, scale=(0.5, 12.0), kind: str = "normal",
                  ld: int | None = None, device="cpu") -> torch.Tensor:
    """Last hidden states [n, L, ld] bf16 for the LM head (columns past d are 0).

    kind "normal": s_i z / (0.02 sqrt(d)), z ~ N(0, 1), s_i ~ U[scale] per position (with
    N(0, 0.02^2) weights the logits spread like the logits workload's); kind "int": k m_i / 8
    with k uniform in [-4, 4] and m_i in {1, 2, 3} per position."""
    ld = d if ld is None else ld
    assert ld >= d and kind in ("normal", "int")
    out = torch.zeros((n, L, ld), dtype=torch.bfloat16, device=device)
    for c in range(n):
        g = _gen(device, seed, _P_HIDDEN, c)
        if kind == "normal":
            z = torch.randn((L, d), generator=g, device=device)
            s = torch.empty((L, 1), device=device).uniform_(scale[0], scale[1],
                                                            generator=_gen(device, seed, _P_SCALE, c))
            out[c, :, :d] = (z * s / (0.02 * math.sqrt(d))).to(torch.bfloat16)
        else:
            k = torch.randint(-4, 5, (L, d), generator=g, device=device).float()
            m = torch.randint(1, 4, (L, 1), generator=g, device=device).float()
            out[c, :, :d] = (k * m / 8.0).to(torch.bfloat16)
    return out


def lm_head_weights_int(V: int, d: int, *, seed: int, device="cpu") -> torch.Tensor:
    """W_lm [V, d] bf16 with entries k / 8, k uniform in [-4, 4]."""
    k = torch.randint(-4, 5, (V, d), generator=_gen(device, seed, _P_WEIGHT, 5), device=device).float()
    return (k / 8.0).to(torch.bfloat16)


def attention_inputs(total_q: int, total_kv: int, Hq: int, Hkv: int, D: int, *, seed: int, device="cpu"):
    """q [total_q, Hq, D], k and v [total_kv, Hkv, D] in bf16 (see the module recipe)."""
    g = _gen(device, seed, _P_ATTN, 0)
    s = torch.empty((total_q, 1, 1), device=device).uniform_(0.5, 4.0, generator=g)
    q = (torch.randn((total_q, Hq, D), generator=g, device=device) * s).to(torch.bfloat16)
    k = torch.randn((total_kv, Hkv, D), generator=g, device=device).to(torch.bfloat16)
    v = torch.randn((total_kv, Hkv, D), generator=g, device=device).to(torch.bfloat16)
    return q, k, v


def canvas_params(wl: Workload, step: int = 0):
    """Per-canvas parameters for a workload, as a dict of numpy arrays (host)."""
    n = wl.n
    rng = np.random.default_rng(np.random.SeedSequence([wl.seed, _P_PARAMS]))
    p = {
        "temperature": np.ones(n, np.float32), "beta": np.zeros(n, np.float32),
        "tau": np.zeros(n, np.float32), "k": np.zeros(n, np.int32),
        "max_steps": np.zeros(n, np.int32), "min_accept": np.ones(n, np.int32),
        "step": np.full(n, step, np.int32), "request_id": np.arange(n, dtype=np.uint32) + 1000,
        "flags": np.full(n, ACTIVE, np.uint32),
    }
    if wl.name == "tiny":
        p["beta"][:] = 2.0; p["tau"][:] = 0.5; p["k"][:] = 2; p["max_steps"][:] = 8
    elif wl.name == "single":
        p["beta"][:] = 8.0; p["tau"][:] = 0.3; p["k"][:] = 2; p["max_steps"][:] = 32
    elif wl.name == "batched":
        p["beta"][:] = rng.uniform(4.0, 16.0, n); p["tau"][:] = 0.3; p["k"][:] = 2
        p["max_steps"][:] = 64; p["flags"][:] = ACTIVE | SELF_COND
    elif wl.name == "profile":
        p["beta"][:] = rng.uniform(4.0, 16.0, n); p["tau"][:] = 0.3; p["k"][:] = 2
        p["max_steps"][:] = 64; p["flags"][:] = ACTIVE | SELF_COND
    elif wl.name == "sweep":
        p["beta"][:] = 8.0; p["tau"][:] = 0.3; p["k"][:] = 3; p["max_steps"][:] = 64
    elif wl.name == "ragged":
        p["temperature"][:] = rng.uniform(0.3, 1.5, n); p["beta"][:] = rng.uniform(2.0, 24.0, n)
        p["tau"][:] = 0.3; p["k"][:] = rng.integers(1, 4, n)
        roles = rng.permutation(n)
        q = n // 4
        conv, ro, normal = roles[:q], roles[q:2 * q], roles[2 * q:]
        p["flags"][conv] = 0                      # already converged: masked, never read
        p["flags"][ro] = ACTIVE | READ_ONLY       # single-pass read
        p["max_steps"][ro] = 1
        p["flags"][normal] = ACTIVE | SELF_COND
        p["max_steps"][normal] = rng.choice(np.array([8, 64], np.int32), normal.size)
        p["max_steps"][conv] = 64
    else:
        raise KeyError(wl.name)
    return p


def params_with(base: dict, **kw) -> dict:
    """Copy of a parameter dict with some arrays replaced or scalars broadcast."""
    out = {k: v.copy() for k, v in base.items()}
    for k, v in kw.items():
        out[k] = np.broadcast_to(np.asarray(v, dtype=out[k].dtype), out[k].shape).copy()
    return out


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 bit patterns (host)."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def host_logits(t: torch.Tensor) -> np.ndarray:
    """Logits tensor -> numpy array the oracle reads (uint16 bf16 bits or float32)."""
    if t.dtype == torch.bfloat16:
        return bf16_bits(t)
    return t.detach().contiguous().cpu().numpy()
