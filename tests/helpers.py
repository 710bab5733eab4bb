"""Shared test utilities: device buffers for one step, and the parity comparison with the
oracle under the counted-boundary rules (exact everywhere except positions within 1e-6
relative of a decision boundary, which are counted and reported)."""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

import entropy_bounded_denoising_gb300 as dg
from entropy_bounded_denoising_gb300 import synth
import oracle

BOUNDARY = 1e-6      # relative margin that makes a decision "near a boundary"
H_RTOL, H_ATOL = 1e-5, 1e-12
LSE_RTOL, LSE_ATOL = 1e-6, 1e-12
DELTA_RTOL = 2e-2
DELTA_ELEM_C = 8.0   # elementwise floor of the feedback check, in units of 2^-8 of the row's RMS


@dataclasses.dataclass
class StepBuffers:
    canvas: torch.Tensor
    prev: torch.Tensor
    stable: torch.Tensor
    accept: torch.Tensor
    argmax: torch.Tensor
    sample: torch.Tensor
    entropy: torch.Tensor
    lse: torch.Tensor
    converged: torch.Tensor
    mean_entropy: torch.Tensor
    n_accept: torch.Tensor

    @staticmethod
    def make(n, L, dev, canvas=None, prev=None, stable=None):
        z = lambda shape, dt, v=0: torch.full(shape, v, dtype=dt, device=dev)
        b = StepBuffers(z((n, L), torch.int32), z((n, L), torch.int32, -1), z((n,), torch.int32),
                        z((n, L), torch.uint8, 7), z((n, L), torch.int32, -7), z((n, L), torch.int32, -7),
                        z((n, L), torch.float32, -1.0), z((n, L), torch.float32, -1.0),
                        z((n,), torch.uint8, 7), z((n,), torch.float32, -1.0), z((n,), torch.int32, -7))
        if canvas is not None:
            b.canvas.copy_(torch.as_tensor(canvas, dtype=torch.int32))
        if prev is not None:
            b.prev.copy_(torch.as_tensor(prev, dtype=torch.int32))
        if stable is not None:
            b.stable.copy_(torch.as_tensor(stable, dtype=torch.int32))
        return b

    def host(self):
        return {k: getattr(self, k).cpu().numpy() for k in
                ("canvas", "prev", "stable", "accept", "argmax", "sample", "entropy", "lse",
                 "converged", "mean_entropy", "n_accept")}


def run_step(x_dev, params_dev, seed, bufs: StepBuffers, V=None, stream=None):
    n, L, ld = x_dev.shape
    dg.dg_denoise_step(x_dev, params_dev, seed, bufs.canvas, bufs.prev, bufs.stable, bufs.accept,
                       bufs.argmax, bufs.sample, bufs.entropy, bufs.lse, bufs.converged,
                       bufs.mean_entropy, bufs.n_accept, V=V if V is not None else ld, ld=ld,
                       stream=stream)


@dataclasses.dataclass
class Report:
    positions: int = 0
    sample_boundary: int = 0
    accept_boundary_canvases: int = 0
    accept_boundary_positions: int = 0
    accept_mismatch: int = 0
    tau_boundary: int = 0
    max_h_rel: float = 0.0

    def __str__(self):
        return (f"positions={self.positions} sample_boundary={self.sample_boundary} "
                f"accept_boundary_canvases={self.accept_boundary_canvases} "
                f"accept_boundary_positions={self.accept_boundary_positions} "
                f"accept_mismatch={self.accept_mismatch} tau_boundary={self.tau_boundary} "
                f"max_entropy_rel={self.max_h_rel:.2e}")


def accept_boundary_positions(H: np.ndarray, beta: float, n_acc: int) -> np.ndarray:
    """Positions of one canvas whose acceptance sits on a decision boundary of the
    entropy-bound rule (DiffusionGemma vLLM page, "엔트로피 기반 디노이징": order by ascending
    entropy, accept the prefix whose running sum stays within beta), given the oracle's fp64
    entropies H [L] and its accepted count n_acc:

    * sort boundary: an accepted position whose entropy lies within 1e-6 relative of the
      first rejected entropy, or a rejected one within 1e-6 of the last accepted entropy (a
      swap across the cut is then a rounding question);
    * budget boundary: the running sum up to and including the position, in the (H, index)
      order, lies within 1e-6 relative of beta (one more or one fewer accepted).

    Below 1e-12 nats entropies are compared absolutely (the entropy check's floor), so the
    sort margin carries that floor too.  Returns a boolean mask [L]."""
    H = np.asarray(H, np.float64)
    L = H.shape[0]
    order = np.lexsort((np.arange(L), H))
    Hs = H[order]
    near = np.zeros(L, bool)
    if 0 < n_acc < L:
        acc = np.zeros(L, bool)
        acc[order[:n_acc]] = True
        h_last, h_first = Hs[n_acc - 1], Hs[n_acc]
        near |= acc & (H >= h_first - (BOUNDARY * abs(h_first) + H_ATOL))
        near |= ~acc & (H <= h_last + (BOUNDARY * abs(h_last) + H_ATOL))
    S = np.cumsum(Hs)   # sequential running sums in the rule's order
    near[order[np.abs(S - beta) <= BOUNDARY * max(abs(beta), 1e-300)]] = True
    return near


def compare_step(g: dict, o: dict, p: dict, V: int, seed: int, canvas_in: np.ndarray,
                 prev_in: np.ndarray, stable_in: np.ndarray, rows=None, g_in: dict | None = None) -> Report:
    """Compare GPU outputs `g` (StepBuffers.host()) with oracle outputs `o`.

    `rows` (optional) restricts the per-position checks to these (canvas, position) pairs and
    skips the per-canvas checks (for sampled parity at full size).  `g_in` (optional) holds
    the GPU buffers before the step; inactive canvases must keep them (else the buffers'
    initial fill values)."""
    rep = Report()
    flags = np.asarray(p["flags"])
    n, L = g["argmax"].shape
    for c in range(n):
        if not (flags[c] & oracle.ACTIVE):
            # inactive: nothing written
            assert (g["canvas"][c] == canvas_in[c]).all()
            assert (g["prev"][c] == prev_in[c]).all() and g["stable"][c] == stable_in[c]
            if g_in is None:
                assert (g["accept"][c] == 7).all() and (g["argmax"][c] == -7).all()
                assert g["converged"][c] == 7
            else:
                for k in ("accept", "argmax", "sample", "entropy", "lse", "converged"):
                    assert np.array_equal(g[k][c], g_in[k][c]), k
            continue
        pos = range(L) if rows is None else [i for (cc, i) in rows if cc == c]
        ro = bool(flags[c] & oracle.READ_ONLY)
        sample_all = bool(flags[c] & synth.SAMPLE_ALL)
        for i in pos:
            rep.positions += 1
            assert g["argmax"][c, i] == o["argmax"][c, i], (c, i)
            h, hr = float(g["entropy"][c, i]), float(o["entropy"][c, i])
            assert abs(h - hr) <= H_RTOL * abs(hr) + H_ATOL, (c, i, h, hr)
            if hr > 1e-9:   # below, the oracle's own -p log p carries ~1e-16 absolute rounding
                rep.max_h_rel = max(rep.max_h_rel, abs(h - hr) / hr)
            l, lr = float(g["lse"][c, i]), float(o["lse"][c, i])
            assert abs(l - lr) <= LSE_RTOL * abs(lr) + LSE_ATOL, (c, i, l, lr)
            if ro or (not sample_all and not g["accept"][c, i]):
                # read-only canvases draw nothing; other canvases without DG_SAMPLE_ALL draw
                # only at accepted positions (a rejected sample is renoised in the same step)
                assert g["sample"][c, i] == -1, (c, i, g["sample"][c, i])
            elif g["sample"][c, i] != o["sample"][c, i]:
                assert o["sample_gap"][c, i] < BOUNDARY, (c, i, g["sample"][c, i], o["sample"][c, i])
                rep.sample_boundary += 1
        if rows is not None:
            continue
        # per-canvas decisions: the accept mask is exact except at positions that sit on a
        # decision boundary themselves, and the accepted count moves by at most their number
        if not ro:
            near = accept_boundary_positions(o["entropy"][c], float(p["beta"][c]), int(o["n_accept"][c]))
            diff = g["accept"][c] != o["accept_mask"][c]
            assert not (diff & ~near).any(), (c, np.nonzero(diff & ~near), np.nonzero(near))
            assert abs(int(g["n_accept"][c]) - int(o["n_accept"][c])) <= int(near.sum()), (c, g["n_accept"][c],
                                                                                           o["n_accept"][c])
            if (o["cut_gap"][c] <= BOUNDARY) or (o["budget_gap"][c] <= BOUNDARY):
                rep.accept_boundary_canvases += 1
            rep.accept_boundary_positions += int(near.sum())
            rep.accept_mismatch += int(diff.sum())
        else:
            assert (g["accept"][c] == 0).all() and g["n_accept"][c] == o["n_accept"][c]
        for i in range(L):
            if ro:
                assert g["canvas"][c, i] == canvas_in[c, i] and g["accept"][c, i] == 0
            elif g["accept"][c, i]:
                assert g["canvas"][c, i] == g["sample"][c, i]
            else:
                tok = oracle.random_token(seed, int(p["request_id"][c]), int(p["step"][c]), i,
                                          oracle.STREAM_RENOISE, V)
                assert g["canvas"][c, i] == tok, (c, i)
        assert (g["prev"][c] == o["argmax"][c]).all()
        assert g["stable"][c] == o["stable_count"][c]
        if g["converged"][c] != o["converged"][c]:
            assert o["tau_gap"][c] <= BOUNDARY, (c, o["mean_entropy"][c], p["tau"][c])
            rep.tau_boundary += 1
        assert abs(g["mean_entropy"][c] - o["mean_entropy"][c]) <= 1e-5 * abs(o["mean_entropy"][c]) + 1e-12
    return rep


def delta_rel_err(got: np.ndarray, ref: np.ndarray) -> np.ndarray:
    """Per-row ||got - ref|| / ||ref|| (rows with ref = 0 compare the absolute norm)."""
    num = np.linalg.norm(got - ref, axis=-1)
    den = np.linalg.norm(ref, axis=-1)
    return np.where(den > 0, num / np.maximum(den, 1e-300), num)


def delta_elem_excess(got: np.ndarray, ref: np.ndarray) -> np.ndarray:
    """Elementwise check of the self-conditioning feedback (DiffusionGemma vLLM page,
    "자기 조건화": every component of delta = W_down (gelu(W_gate pe) * (W_up pe)), pe = P . E).

    Bound per component j of a row:  |got_j - ref_j| <= 2e-2 |ref_j| + c 2^-8 rms(ref row),
    c = DELTA_ELEM_C = 8.  Returned: the largest excess over the bound per row, in units of
    the row's RMS (<= 0 passes).

    Derivation.  The tensor-core path rounds to bf16 (relative error <= 2^-9) four times: the
    softmax P fed to P . E, pe, the MLP's hidden gelu(g) * u, and delta itself; it
    accumulates in fp32 (relative ~1e-7 per sum, negligible).  The last rounding is a
    relative error of the component (<= 2^-9, inside the 2e-2 term).  The three inner
    roundings enter through linear maps with random weights, so each leaves an error of
    about 2^-9 / sqrt(3) of the row's RMS per component, sqrt(2) larger through the product
    gelu(g) * u (both factors move): a standard deviation of about sqrt(5/3) 2^-9 = 0.65 2^-8
    of the RMS, plus a part proportional to |ref_j| (a sharp P's rounding scales the whole
    row), which the relative term absorbs.  A CPU emulation of the same roundings in torch
    (tests/test_feedback_bound.py) leaves at most 3.8 2^-8 RMS beyond 2e-2 |ref_j| on the
    batched shapes; c = 8 doubles that.  A component that is wholly wrong (zero, another
    column's value, a gate/up mix-up) misses by |ref_j|, which exceeds the bound wherever
    |ref_j| > 3.2 % of the RMS, i.e. in almost every row, while it moves the row's norm by
    only ~1/sqrt(d) (1.6 % at d = 4096, under the per-row 2e-2)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    rms = np.sqrt(np.mean(ref * ref, axis=-1, keepdims=True))
    bound = DELTA_RTOL * np.abs(ref) + DELTA_ELEM_C * 2.0 ** -8 * rms
    ex = np.abs(got - ref) - bound
    ex = np.where(np.isnan(ex), np.inf, ex)
    return np.max(ex / np.where(rms > 0, rms, 1.0), axis=-1)


def check_delta(got: np.ndarray, ref: np.ndarray, ctx=None) -> None:
    """Feedback rows against the oracle: the per-row norm (2e-2) and every component
    (delta_elem_excess <= 0)."""
    got = np.asarray(got, np.float64).reshape(-1, ref.shape[-1])
    ref = np.asarray(ref, np.float64).reshape(-1, ref.shape[-1])
    err = delta_rel_err(got, ref)
    assert err.max() <= DELTA_RTOL, (ctx, "row norm", err.max())
    ex = delta_elem_excess(got, ref)
    assert ex.max() <= 0.0, (ctx, "elementwise", int(np.argmax(ex)), ex.max())
