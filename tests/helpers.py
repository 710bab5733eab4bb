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
LSE_RTOL = 1e-6
DELTA_RTOL = 2e-2


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
    accept_mismatch: int = 0
    tau_boundary: int = 0
    max_h_rel: float = 0.0

    def __str__(self):
        return (f"positions={self.positions} sample_boundary={self.sample_boundary} "
                f"accept_boundary_canvases={self.accept_boundary_canvases} "
                f"accept_mismatch_at_boundary={self.accept_mismatch} tau_boundary={self.tau_boundary} "
                f"max_entropy_rel={self.max_h_rel:.2e}")


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
            assert abs(l - lr) <= LSE_RTOL * max(abs(lr), 1.0), (c, i, l, lr)
            if ro or (not sample_all and not g["accept"][c, i]):
                # read-only canvases draw nothing; other canvases without DG_SAMPLE_ALL draw
                # only at accepted positions (a rejected sample is renoised in the same step)
                assert g["sample"][c, i] == -1, (c, i, g["sample"][c, i])
            elif g["sample"][c, i] != o["sample"][c, i]:
                assert o["sample_gap"][c, i] < BOUNDARY, (c, i, g["sample"][c, i], o["sample"][c, i])
                rep.sample_boundary += 1
        if rows is not None:
            continue
        # per-canvas decisions
        boundary = (o["cut_gap"][c] <= BOUNDARY) or (o["budget_gap"][c] <= BOUNDARY)
        mism = int((g["accept"][c] != o["accept_mask"][c]).sum())
        if boundary:
            rep.accept_boundary_canvases += 1
            rep.accept_mismatch += mism
        else:
            assert mism == 0, (c, np.nonzero(g["accept"][c] != o["accept_mask"][c]))
            assert g["n_accept"][c] == o["n_accept"][c]
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
