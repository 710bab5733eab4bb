"""Benchmark of the entropy-bounded denoising step on GB300.

One step = the whole hot path over one batch: the denoise step (per-position softmax /
entropy / argmax / Gumbel-max sample, entropy-bound acceptance, renoise, convergence) and the
self-conditioning feedback (P.E on tensor cores with the softmax fused into the operand load,
then the gated MLP).  Default workload: 8 canvases x 256 positions, V = 262144, d = 4096,
h = 16384, bf16 logits (the batched full-vocabulary step).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload batched|sweep|ragged|single]
    python bench.py --workload sweep --loop --warmup 1   # the whole loop to convergence
    python bench.py --impl reference ...   # the fp64 CPU oracle on the host cores

Prints one JSON line (rank 0).  Under torchrun every rank runs an independent replica on its
own GPU (the path has no exchange step), the timed region is bracketed by barriers and the
slowest rank's time counts.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "canvas positions/s per denoise step (V=262144, d=4096); % of HBM/TC roofline"
UNIT = "positions/s"


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            pk = json.load(f)
        return {"hbm_gbs": pk["hbm_gbs"], "bf16_tflops": pk["bf16_tflops"],
                "bf16_tflops_sustained": pk.get("bf16_tflops_sustained", pk["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def choose_tc_peak(pk: dict, window_s: float, sm_mhz, sm_max_mhz):
    """The bf16 tensor peak that matches the timed window: the burst figure (cuBLAS timed
    alone, at full clock) when the window is short (under a second) or the SM clock stayed
    within 3 % of its maximum, else the sustained figure (cuBLAS over seconds under the
    power cap).  Returns (peak TFLOP/s, which)."""
    full_clock = bool(sm_mhz and sm_max_mhz and sm_mhz >= 0.97 * sm_max_mhz)
    if window_s < 1.0 or full_clock:
        return pk["bf16_tflops"], "burst"
    return pk["bf16_tflops_sustained"], "sustained"


def max_over_ranks(x: float, device=None) -> float:
    """The largest of the ranks' values (the slowest rank's time); x itself on one rank."""
    import torch
    import torch.distributed as tdist
    if not (tdist.is_available() and tdist.is_initialized()) or tdist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    tdist.all_reduce(t, op=tdist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(positions_per_rank: int, world: int, steps: int, elapsed_ms: float) -> float:
    """Whole-job positions/s: every rank's positions over the slowest rank's time."""
    return positions_per_rank * world * steps / (elapsed_ms / 1e3)


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, which):
        setattr(self, which, time.time())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        """Median SM clock and throttle reasons over the samples taken inside the timed
        region (all samples if none fell inside)."""
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        t0, t1 = getattr(self, "t_start", None), getattr(self, "t_end", None)
        rows = self.lines
        if t0 is not None and t1 is not None:
            inside = [r for r in rows if t0 <= r[0] <= t1 + 0.25]
            rows = inside or rows
        for _, ln in rows:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def _workload_arith(wl, n_sc_rows, n_read_rows, from_hidden=False):
    """Algorithmic bytes and tensor-core FLOPs of one step.  From hidden states the step
    reads the hidden rows instead of the logits and adds the LM head's contraction (its
    weights are the embedding table, already counted); the logits are an intermediate."""
    N = wl.n * wl.L
    logits_b = 2 * n_read_rows * wl.V
    e_b = 2 * wl.V * wl.d
    w_b = 6 * wl.d * wl.h
    out_b = 17 * N + 2 * N * wl.d
    pe_flops = 2.0 * n_sc_rows * wl.V * wl.d
    mlp_flops = 6.0 * n_sc_rows * wl.d * wl.h
    lm_flops = 2.0 * n_read_rows * wl.V * wl.d if from_hidden else 0.0
    in_b = 2 * n_read_rows * wl.d if from_hidden else logits_b
    return {"bytes": in_b + e_b + w_b + out_b, "logits_bytes": logits_b, "pe_flops": pe_flops,
            "mlp_flops": mlp_flops, "lm_flops": lm_flops, "tc_flops": pe_flops + mlp_flops + lm_flops}


def _profile_traffic(kernel_tag: str):
    """Per-launch DRAM bytes recorded from an ncu capture in profiles/, if the kernel sources
    it was taken on (the files its `csrc_files:` line lists) are unchanged (else None)."""
    path = os.path.join(ROOT, "profiles", f"{kernel_tag}.md")
    if not os.path.exists(path):
        return None
    txt = open(path).read()
    src = os.path.join(ROOT, "entropy_bounded_denoising_gb300", "csrc")
    f = re.search(r"csrc_files:\s*([^\n]+)", txt)
    files = f.group(1).split() if f else sorted(x for x in os.listdir(src) if x.endswith((".cu", ".cuh")))
    h = hashlib.sha256()
    for name in files:
        with open(os.path.join(src, name), "rb") as fh:
            h.update(fh.read())
    digest = h.hexdigest()[:16]
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", txt)
    s = re.search(r"csrc_sha256_16:\s*([0-9a-f]{16})", txt)
    if m and s and s.group(1) == digest:
        return float(m.group(1))
    return None


# --------------------------------------------------------------------------- CPU oracle
def _oracle_sample(wl, x_host, weights_host, p, n_sc_rows: int, threads: int):
    """Time the fp64 oracle's denoise step on every canvas of x_host [n, L, V] and its
    self-conditioning on n_sc_rows rows; returns seconds per canvas position (denoise time per
    active position + feedback time per row) and the two times."""
    import oracle
    n, L = x_host.shape[0], wl.L
    active = int(((np.asarray(p["flags"]) & 1) != 0).sum()) * L
    t0 = time.perf_counter()
    oracle.denoise_step(x_host, p, 7, np.zeros((n, L), np.int32), np.full((n, L), -1, np.int32),
                        np.zeros(n, np.int32), n_threads=threads)
    t_dn = time.perf_counter() - t0
    t_sc = 0.0
    if n_sc_rows:
        E, Wg, Wu, Wd = weights_host
        rows = x_host.reshape(n * L, -1)[:n_sc_rows]
        t0 = time.perf_counter()
        oracle.self_cond_rows(rows, np.full(n_sc_rows, float(p["temperature"][0])), E, Wg, Wu, Wd, V=wl.V,
                              n_threads=threads)
        t_sc = time.perf_counter() - t0
    per_pos = t_dn / max(1, active) + (t_sc / n_sc_rows if n_sc_rows else 0.0)
    return per_pos, t_dn, t_sc


def run_reference(args):
    """The oracle as it stands, on the host cores, as the comparison arm.

    One step = the oracle's denoise step on a slice of positions of canvas 0 plus, in every
    m-th step, its self-conditioning on one position per host thread (the oracle runs rows
    in parallel); m and the slice are set from the warm-up timings so that the K timed steps
    take about two minutes.  The value is positions/s with the per-position cost =
    (denoise time / positions) + (feedback time / feedback rows) over the timed steps."""
    ws, rank, _ = _dist()
    if rank != 0:
        return 0
    import oracle
    from entropy_bounded_denoising_gb300 import synth
    wl = synth.WORKLOADS[args.workload]
    oracle.build()
    threads = oracle.max_threads()
    p = synth.canvas_params(wl, step=1)
    x = synth.logits(1, wl.L, wl.V, seed=wl.seed, step=1, scale=wl.scale, spike_frac=wl.spike_frac,
                     dtype=wl.dtype, canvases=[0])
    xh = synth.host_logits(x)[0]
    E, Wg, Wu, Wd = synth.weights(wl.V, wl.d, wl.h, seed=wl.seed)
    wh = tuple(synth.bf16_bits(t) for t in (E, Wg, Wu, Wd))
    p1 = {k: v[:1].copy() for k, v in p.items()}

    def denoise(rows):
        t0 = time.perf_counter()
        oracle.denoise_step(xh[None, :rows], p1, 7, np.zeros((1, rows), np.int32), np.full((1, rows), -1, np.int32),
                            np.zeros(1, np.int32), n_threads=threads)
        return time.perf_counter() - t0

    n_fb = min(wl.L, max(1, threads))  # feedback rows per call: one per host thread

    def feedback():
        t0 = time.perf_counter()
        oracle.self_cond_rows(xh[:n_fb], np.full(n_fb, float(p["temperature"][0])), *wh, V=wl.V, n_threads=threads)
        return time.perf_counter() - t0

    # warm-up: unit costs
    rows = min(wl.L, max(1, threads))
    c_dn, c_sc = denoise(rows) / rows, feedback()
    for _ in range(max(0, args.warmup - 1)):
        c_dn = denoise(rows) / rows
    budget = 120.0 / max(1, args.steps)               # seconds per timed step
    rows = int(min(wl.L, max(1, (0.5 * budget) / max(c_dn, 1e-9))))
    every = max(1, int(np.ceil(c_sc / max(0.5 * budget, 1e-9))))
    t_dn = t_sc = 0.0
    n_dn = n_sc = 0
    wall0 = time.perf_counter()
    for k in range(args.steps):
        t_dn += denoise(rows)
        n_dn += rows
        if k % every == 0:
            t_sc += feedback()
            n_sc += n_fb
    wall = time.perf_counter() - wall0
    per_pos = t_dn / n_dn + t_sc / max(1, n_sc)
    value = 1.0 / per_pos
    sample = (f"per step: oracle denoise on {rows} positions of canvas 0 (V={wl.V}); oracle self-conditioning "
              f"on {n_fb} positions every {every} step(s) ({n_sc} rows in total); per-position cost = denoise "
              f"time / positions + feedback time / feedback rows")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": wall / max(1, args.steps) * 1e3,
            "value_note": (f"value extrapolated from the sample: 1 / (denoise time per position + feedback time per "
                           f"row); a whole {wl.n} x {wl.L} step would take about "
                           f"{per_pos * wl.n * wl.L:.0f} s on these cores; ms_per_step is the wall time of one "
                           f"sampled step"),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": _config(wl),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def _config(wl, from_hidden=False):
    src = ("from bf16 hidden states: LM head (tied to E) fused with the step's statistics"
           if from_hidden else f"{wl.dtype} logits")
    return {"workload": (f"{wl.name}: {wl.n} canvases x {wl.L} positions, V={wl.V}, d={wl.d}, h={wl.h}, "
                         f"{src}"),
            "n_canvas": wl.n, "L": wl.L, "V": wl.V, "d": wl.d, "h": wl.h,
            "l2": "no flush: each step reads inputs larger than L2 (logits + embedding table)",
            "parallelism": "replicas (canvases independent, no exchange step)"}


# --------------------------------------------------------------------------- GPU arm
def run_ours(args):
    import torch
    import entropy_bounded_denoising_gb300 as dg
    from entropy_bounded_denoising_gb300 import synth, build

    ws, rank, local = _dist()
    if ws > 1:
        import torch.distributed as tdist
        torch.cuda.set_device(local)
        tdist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if rank == 0:
        build.build()
    if ws > 1:
        tdist.barrier()
    dg.load()

    def barrier():
        if ws > 1:
            tdist.barrier()

    wl = synth.WORKLOADS[args.workload]
    n, L, V, d, h = wl.n, wl.L, wl.V, wl.d, wl.h
    p = synth.canvas_params(wl, step=1)
    if wl.name in ("sweep", "single", "profile"):
        p["flags"] |= dg.DG_SELF_COND
    x = synth.logits(n, L, V, seed=wl.seed + 1000 * rank, step=1, scale=wl.scale, spike_frac=wl.spike_frac,
                     dtype=wl.dtype, device=dev)
    E, Wg, Wu, Wd = synth.weights(V, d, h, seed=wl.seed, device=dev)
    params = dg.params_tensor(p, dev)

    def z(shape, dt, v=0):
        return torch.full(shape, v, dtype=dt, device=dev)

    canvas, prev, stable = z((n, L), torch.int32), z((n, L), torch.int32, -1), z((n,), torch.int32)
    acc, am, smp = z((n, L), torch.uint8), z((n, L), torch.int32), z((n, L), torch.int32)
    ent, lse, conv = z((n, L), torch.float32), z((n, L), torch.float32), z((n,), torch.uint8)
    delta = torch.empty((n, L, d), dtype=torch.bfloat16, device=dev)
    wsp = torch.empty(dg.dg_self_cond_workspace_bytes(n, L, d, h), dtype=torch.uint8, device=dev)
    dws = torch.empty(dg.dg_denoise_workspace_bytes(n, L, V, dg.DG_BF16 if wl.dtype == "bf16" else dg.DG_FP32),
                      dtype=torch.uint8, device=dev)
    # --from-hidden: the step starts from the last hidden states; the LM head (tied to E) writes
    # the logits the feedback reads and the step's statistics come from its epilogue
    fh = args.from_hidden
    if fh:
        hid = synth.hidden_states(n, L, d, seed=wl.seed + 1000 * rank, kind="normal", device=dev)
        xs = torch.empty((n, L, V), dtype=torch.bfloat16, device=dev)
        lws = torch.empty(dg.dg_lm_head_workspace_bytes(n, L, V), dtype=torch.uint8, device=dev)
    else:
        xs = x
    # --graph captures the step once as a CUDA graph (on a side stream, as capture requires)
    # and times its replays; otherwise every step is enqueued call by call.
    stream = torch.cuda.Stream(device=dev) if args.graph else torch.cuda.current_stream()
    stream.wait_stream(torch.cuda.current_stream())
    seed = 0x5EED0000 + rank
    # Small batches (a single request) run the overlapped schedule: the feedback, which needs
    # only the step's lse, starts right after the statistics pass; the acceptance and the
    # deferred samples run on a second stream beside the MLP GEMMs; the rows of canvases that
    # converged are zeroed at the end (bit-identical outputs, tests/test_gpu_schedule.py).  Larger batches keep every launch
    # on one stream (measured faster: the second stream's sampler slows P.E more than it saves).
    overlap = not fh and n * L <= 512
    side = torch.cuda.Stream(device=dev) if overlap else None
    ev_fork, ev_join = torch.cuda.Event(), torch.cuda.Event()

    def step_calls(xin, ev=None):
        if ev:
            ev[0].record(stream)
        if fh:
            dg.dg_lm_head_denoise_step(hid, E, params, seed, xs, canvas, prev, stable, acc, am, smp, ent, lse,
                                       conv, workspace=lws, stream=stream)
        elif overlap:
            # the feedback plan needs no statistics: first, so that P.E follows the statistics
            # pass directly (its CTAs take the SMs the pass leaves free and bring their first
            # embedding tiles into L2 while it runs)
            dg.dg_self_cond_prepare(params, None, n, L, d, h, delta, wsp, stream=stream)
            dg.dg_denoise_row_stats(xin, params, seed, am, smp, ent, lse, dws, stream=stream)
        else:
            dg.dg_denoise_step(xin, params, seed, canvas, prev, stable, acc, am, smp, ent, lse, conv,
                               workspace=dws, stream=stream)
        if not overlap:
            dg.dg_self_cond_prepare(params, conv, n, L, d, h, delta, wsp, stream=stream)
        if ev:
            ev[1].record(stream)
        dg.dg_self_cond_pe(xs if fh else xin, lse, params, E, h, wsp, stream=stream)
        if overlap:
            # forked once P.E is done: the acceptance and the samples then share the SMs with
            # the MLP GEMMs (which leave some idle) instead of taking an SM that P.E needs
            ev_fork.record(stream)
            side.wait_event(ev_fork)
            dg.dg_denoise_accept(ent, smp, am, params, seed, canvas, prev, stable, acc, conv, dws, V=V, stream=side)
            dg.dg_denoise_samples(xin, params, seed, canvas, smp, dws, stream=side)
            ev_join.record(side)
        if ev:
            ev[2].record(stream)
        dg.dg_self_cond_mlp(n, L, Wg, Wu, Wd, delta, wsp, stream=stream)
        if overlap:
            stream.wait_event(ev_join)
            dg.dg_self_cond_zero_converged(params, conv, delta, stream=stream)
        if ev:
            ev[3].record(stream)

    def step(ev=None):
        step_calls(x, ev)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    dg.dg_clear_device_status()
    graph = None
    launches_per_step = 0
    if args.graph:
        graph = torch.cuda.CUDAGraph()
        c0 = dg.dg_launch_count()
        with torch.cuda.graph(graph, stream=stream):
            step()
        launches_per_step = dg.dg_launch_count() - c0
        with torch.cuda.stream(stream):
            for _ in range(3):
                graph.replay()
        torch.cuda.synchronize()

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        time.sleep(0.3)  # let nvidia-smi start sampling before the timed region
        clk.mark("t_start")
        launches0 = dg.dg_launch_count()
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(stream)
        if graph is not None:
            with torch.cuda.stream(stream):
                for k in range(args.steps):
                    graph.replay()
        else:
            for k in range(args.steps):
                step(evs[k])
        end.record(stream)
        launches = dg.dg_launch_count() - launches0
        torch.cuda.synchronize()
        clk.mark("t_end")
    barrier()
    elapsed_ms = start.elapsed_time(end)
    status = dg.dg_get_device_status()
    if status:
        raise RuntimeError(f"device status {status:#x} after the timed region")
    n_conv = int(conv.sum().item())
    flags = p["flags"]
    active = (flags & dg.DG_ACTIVE) != 0
    sc_on = active & ((flags & dg.DG_SELF_COND) != 0) & ((flags & dg.DG_READ_ONLY) == 0)
    conv_h = conv.cpu().numpy().astype(bool)
    n_sc_rows = int((sc_on & ~conv_h).sum()) * L
    n_read_rows = int(active.sum()) * L
    positions = n_read_rows
    elapsed_ms = max_over_ranks(elapsed_ms, dev)
    ms_step = elapsed_ms / args.steps
    value = job_throughput(positions, ws, args.steps, elapsed_ms)

    if graph is not None:
        # the per-phase split from eager steps (the replays carry no events); launches per
        # replay are the captured step's
        launches = launches_per_step * args.steps
        for k in range(min(20, args.steps)):
            step(evs[k])
        torch.cuda.synchronize()
        evs = evs[:min(20, args.steps)]
    t_dn = float(np.mean([e[0].elapsed_time(e[1]) for e in evs]))
    t_pe = float(np.mean([e[1].elapsed_time(e[2]) for e in evs]))
    t_mlp = float(np.mean([e[2].elapsed_time(e[3]) for e in evs]))
    ar = _workload_arith(wl, n_sc_rows, n_read_rows, from_hidden=fh)
    pk = _peaks()
    clocks = clk.summary()
    window_s = elapsed_ms * 1e-3
    peak_tc, peak_kind = choose_tc_peak(pk, window_s, clocks.get("sm_mhz"), clocks.get("sm_max_mhz"))
    peak_alone = pk["bf16_tflops"]   # rows timed alone, in short bursts
    pe_tflops = ar["pe_flops"] / (t_pe * 1e-3) / 1e12 if t_pe > 0 else 0.0
    t_roof = max(ar["bytes"] / (pk["hbm_gbs"] * 1e9), ar["tc_flops"] / (peak_tc * 1e12))
    # the committed capture is of the batched workload's P.E launch: no figure for the others
    traffic = _profile_traffic("pe_gemm_batched") if wl.name == "batched" else None

    # ---------------------------------------------------------------- e2e: host buffers
    e2e = None
    if not args.no_e2e:
        xin = hid if fh else x
        xh = torch.empty(xin.shape, dtype=xin.dtype, pin_memory=True)
        xh.copy_(xin)
        out_canvas = torch.empty((n, L), dtype=torch.int32, pin_memory=True)
        out_conv = torch.empty((n,), dtype=torch.uint8, pin_memory=True)
        out_delta = torch.empty((n, L, d), dtype=torch.bfloat16, pin_memory=True)
        h2d = xh.numel() * xh.element_size()
        d2h = (out_canvas.numel() * 4 + out_conv.numel() + out_delta.numel() * 2)
        # Pipelined like a serving loop: step k+1's logits are copied host -> device on a
        # second stream (into the other of two device buffers) while step k computes; every
        # step's copy in and result copy out lie inside the timed region.
        copy_stream = torch.cuda.Stream(device=dev)
        xdev = [torch.empty_like(xin), torch.empty_like(xin)]
        h2d_done = [torch.cuda.Event(), torch.cuda.Event()]
        buf_free = [torch.cuda.Event(), torch.cuda.Event()]

        def e2e_h2d(k):
            b = k % 2
            copy_stream.wait_event(buf_free[b])  # the step that last read buffer b is done
            with torch.cuda.stream(copy_stream):
                xdev[b].copy_(xh, non_blocking=True)
            h2d_done[b].record(copy_stream)

        def e2e_compute(k):
            b = k % 2
            stream.wait_event(h2d_done[b])
            if fh:
                dg.dg_lm_head_denoise_step(xdev[b], E, params, seed, xs, canvas, prev, stable, acc, am, smp, ent,
                                           lse, conv, workspace=lws, stream=stream)
                dg.dg_self_cond_logits(xs, lse, params, conv, E, Wg, Wu, Wd, delta, wsp, stream=stream)
            else:
                step_calls(xdev[b])
            buf_free[b].record(stream)
            out_canvas.copy_(canvas, non_blocking=True)
            out_conv.copy_(conv, non_blocking=True)
            out_delta.copy_(delta, non_blocking=True)

        def e2e_run(nsteps, s_ev=None, e_ev=None):
            if s_ev is not None:
                s_ev.record(copy_stream)
            e2e_h2d(0)
            for k in range(nsteps):
                if k + 1 < nsteps:
                    e2e_h2d(k + 1)
                e2e_compute(k)
            if e_ev is not None:
                e_ev.record(stream)

        e2e_run(3)
        torch.cuda.synchronize()
        barrier()
        s2, e2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e2e_run(args.steps, s2, e2)
        torch.cuda.synchronize()
        barrier()
        ms2 = max_over_ranks(s2.elapsed_time(e2), dev)
        e2e = {"value": job_throughput(positions, ws, args.steps, ms2), "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": ms2 / args.steps,
               "pipelining": "next step's H2D overlaps this step's compute (two device input buffers)"}

    # ---------------------------------------------------------------- rows around the step
    # Timed alone (not part of the step): the next pass's embeddings (token rows + feedback),
    # single-pass-read choice probabilities (4 slots per position) and the commit, each
    # against the HBM roofline of its algorithmic bytes.
    around = None
    if not args.no_extras and not fh:
        rng = np.random.default_rng(5)
        emb = torch.empty((n * L, d), dtype=torch.bfloat16, device=dev)
        C = 4
        choices = torch.from_numpy(rng.integers(0, V, (n, L, C)).astype(np.int32)).to(dev)
        probs = torch.empty((n, L, C), dtype=torch.float32, device=dev)
        tokens = torch.empty((n, L), dtype=torch.int32, device=dev)
        committed = torch.empty((n,), dtype=torch.uint8, device=dev)

        def _time(fn, reps=50):
            for _ in range(5):
                fn()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(reps):
                fn()
            b.record(stream)
            torch.cuda.synchronize()
            return a.elapsed_time(b) / reps

        def _entry(ms, nbytes):
            gbs = nbytes / (ms * 1e-3) / 1e9
            return {"ms": ms, "alg_bytes": nbytes, "achieved_gbs": gbs, "frac_hbm": gbs / pk["hbm_gbs"]}

        p_all = dict(p)
        p_all["flags"] = p["flags"] | dg.DG_SAMPLE_ALL
        params_all = dg.params_tensor(p_all, dev)

        def _denoise(prm):
            return lambda: dg.dg_denoise_step(x, prm, seed, canvas, prev, stable, acc, am, smp, ent, lse, conv,
                                              workspace=dws, stream=stream)

        around = {
            "denoise_step": {"ms": _time(_denoise(params), reps=20),
                             "note": "dg_denoise_step as in the step: samples drawn at the accepted positions"},
            "denoise_step_sample_all": {"ms": _time(_denoise(params_all), reps=20),
                                        "note": "dg_denoise_step with DG_SAMPLE_ALL: every position draws its "
                                                "sample in the statistics pass"},
            "embed_canvas": _entry(_time(lambda: dg.dg_embed_canvas(canvas, E, delta.view(n * L, d), emb, 1.0,
                                                                    stream=stream)),
                                   n * L * (3 * d * 2 + 4)),
            "choice_probs": _entry(_time(lambda: dg.dg_choice_probs(x, lse, params, choices, probs, stream=stream)),
                                   n * L * (C * (4 + 4 + 2) + 4)),
            "commit": _entry(_time(lambda: dg.dg_commit(params, conv, am, tokens, prev, stable, committed,
                                                        stream=stream)),
                             n * L * 4 * 2 + n * 10),
            "note": "timed alone, not part of the step; alg_bytes: embed = E rows gathered + feedback + "
                    "output; choice_probs = 4 slots x (token + probability + logit) + lse; commit = argmax + tokens",
        }
        # Read-only canvases (single-pass reads): the step with the choice gather fused into
        # its statistics pass, against the step followed by the separate gather.
        p_ro = dict(p)
        p_ro["flags"] = p["flags"] | dg.DG_READ_ONLY
        params_ro = dg.params_tensor(p_ro, dev)
        t_ro = _time(_denoise(params_ro), reps=20)
        t_ro_fused = _time(lambda: dg.dg_denoise_step_choices(x, params_ro, seed, canvas, prev, stable, acc, am, smp,
                                                              ent, lse, conv, choices, probs, workspace=dws,
                                                              stream=stream), reps=20)
        around["read_only_step_choices"] = {
            "fused_ms": t_ro_fused, "unfused_ms": t_ro + around["choice_probs"]["ms"], "step_alone_ms": t_ro,
            "note": f"every canvas DG_READ_ONLY with {C} choices per position: dg_denoise_step_choices against "
                    "dg_denoise_step then dg_choice_probs"}
        # attention before the LM-head rows, after half a second idle: timed straight after a
        # second of GEMMs at the power cap, it would measure the clock that load left behind
        torch.cuda.synchronize()
        time.sleep(0.5)
        around["attention"] = _attention_rows(dg, synth, dev, stream, _time, peak_alone)
        # The LM head fused with the step's statistics (logits = hidden . E^T with the head tied
        # to the embedding table, stored once; entropy / lse / argmax from the GEMM's epilogue),
        # against the same work unfused: the LM head alone, then dg_denoise_step on its logits.
        hid = synth.hidden_states(n, L, d, seed=wl.seed + 7, kind="normal", device=dev)
        xl = torch.empty((n, L, V), dtype=torch.bfloat16, device=dev)
        lws = torch.empty(dg.dg_lm_head_workspace_bytes(n, L, V), dtype=torch.uint8, device=dev)
        t_lm = _time(lambda: dg.dg_lm_head_denoise_step(hid, E, params, seed, xl, canvas, prev, stable, acc, am, smp,
                                                        ent, lse, conv, workspace=lws, stream=stream), reps=10)
        t_lm_logits = _time(lambda: dg.dg_lm_head_logits(hid, E, params, xl, lws, stream=stream), reps=10)
        t_dn_xl = _time(lambda: dg.dg_denoise_step(xl, params, seed, canvas, prev, stable, acc, am, smp, ent, lse,
                                                   conv, workspace=dws, stream=stream), reps=10)
        lm_flops = 2.0 * n * L * V * d
        around["lm_head_step"] = {
            "ms": t_lm, "tflops": lm_flops / (t_lm * 1e-3) / 1e12,
            "frac_tc": lm_flops / (t_lm * 1e-3) / 1e12 / peak_alone,
            "unfused_ms": t_lm_logits + t_dn_xl, "lm_head_logits_ms": t_lm_logits,
            "denoise_on_its_logits_ms": t_dn_xl,
            "note": "dg_lm_head_denoise_step (hidden [n, L, d] x E^T -> bf16 logits + step), timed alone; "
                    "frac_tc: 2 N V d flops against the burst bf16 peak; unfused = dg_lm_head_logits "
                    "then dg_denoise_step"}
        del xl, lws, hid
        torch.cuda.synchronize()
        if dg.dg_get_device_status():
            raise RuntimeError("device status set by the rows around the step")

    # ---------------------------------------------------------------- CPU baseline (oracle)
    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline and not fh:
        import oracle
        oracle.build()
        threads = oracle.max_threads()
        xh = synth.host_logits(x)
        wh = tuple(synth.bf16_bits(t) for t in (E, Wg, Wu, Wd))
        n_sc = min(n * L, 16 * max(1, threads))  # about 10 s of feedback rows on the host cores
        per_pos, t_dn_cpu, t_sc_cpu = _oracle_sample(wl, xh, wh, p, n_sc, threads)
        del xh
        cpu = {"value": 1.0 / per_pos, "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": (f"denoise oracle on all {n} canvases ({n * L} positions x V={V}, {t_dn_cpu:.1f} s) plus "
                          f"self-conditioning on {n_sc} rows ({t_sc_cpu:.1f} s); per position = denoise time per "
                          f"position + feedback time per row")}

    if rank != 0:
        return 0
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": _config(wl, fh),
        "launch": (("CUDA graph replays of the captured step" if graph is not None
                    else "eager: every call enqueued each step")
                   + ("; acceptance and samples on a second stream beside the feedback GEMMs" if overlap else "")),
        "roofline": {"bound": "tensor", "achieved": pe_tflops, "peak": peak_tc, "unit": "TFLOP/s",
                     "frac": pe_tflops / peak_tc, "traffic": traffic,
                     "kernel": "P.E contraction (k_gemm softmax-A, N-major B) + split-K fix-up",
                     "peak_source": (f"{pk['source']} {peak_kind} bf16: timed window {window_s:.3f} s at a median "
                                     f"{clocks.get('sm_mhz')} of {clocks.get('sm_max_mhz')} MHz (burst when the "
                                     f"window is under 1 s or the clock within 3 % of its maximum)")},
        "step_roofline": {"t_roof_ms": t_roof * 1e3, "frac": (t_roof * 1e3) / ms_step,
                          "alg_bytes": ar["bytes"], "tc_flops": ar["tc_flops"],
                          "hbm_peak_gbs": pk["hbm_gbs"], "tc_peak_tflops": peak_tc},
        "kernels_ms": {("lm_head_denoise_and_prepare" if fh else "denoise_and_prepare"): t_dn, "pe": t_pe,
                       "mlp": t_mlp,
                       "denoise_hbm_frac": (None if fh else (ar["logits_bytes"] / (t_dn * 1e-3)) / (pk["hbm_gbs"] * 1e9)),
                       "lm_head_tflops": (ar["lm_flops"] / (t_dn * 1e-3) / 1e12) if fh else None,
                       "mlp_tflops": ar["mlp_flops"] / (t_mlp * 1e-3) / 1e12 if t_mlp > 0 else 0.0},
        "steps_per_s": 1e3 / ms_step, "self_cond_rows": n_sc_rows, "converged_canvases": n_conv,
        "e2e": e2e, "cpu_baseline": cpu, "gpu_launches": launches, "clocks": clocks,
        "around_step": around,
    }
    print(json.dumps(line), flush=True)
    if ws > 1:
        tdist.destroy_process_group()
    return 0


def attention_counts(seqs, W, TQ=128, TK=64):
    """(allowed (query, key) pairs, key tiles visited, key tiles in all) for sequences given as
    (q_len, kv_len, causal): a query tile visits every TK-key tile from the first key any of
    its queries may see to the last."""
    pairs = tiles = tiles_all = 0
    for ql, kl, c in seqs:
        pos = np.arange(kl - ql, kl)
        lo = np.maximum(0, pos - W) if W >= 0 else np.zeros_like(pos)
        hi = pos if c else (np.minimum(kl - 1, pos + W) if W >= 0 else np.full_like(pos, kl - 1))
        pairs += int((hi - lo + 1).sum())
        for t0 in range(0, ql, TQ):
            p0, p1 = int(pos[t0]), int(pos[min(ql, t0 + TQ) - 1])
            jl = max(0, p0 - W) if W >= 0 else 0
            jh = p1 if c else (min(kl - 1, p1 + W) if W >= 0 else kl - 1)
            tiles += jh // TK - jl // TK + 1
            tiles_all += (kl + TK - 1) // TK
    return pairs, tiles, tiles_all


def _attention_rows(dg, synth, dev, stream, time_fn, peak_tc):
    """dg_attention timed alone on a denoising batch: 8 canvases of 256 after 2048 context
    tokens (bidirectional) and 4 causal prefills of 1024, 16 query heads over 8 key/value
    heads, D = 128, without a window and with W = 512."""
    import torch
    seqs = [(256, 2304, 0)] * 8 + [(1024, 1024, 1)] * 4
    cu_q = np.cumsum([0] + [a[0] for a in seqs]).astype(np.int32)
    cu_kv = np.cumsum([0] + [a[1] for a in seqs]).astype(np.int32)
    cz = np.array([a[2] for a in seqs], np.uint8)
    Hq, Hkv, Dh, TQ, TK = 16, 8, 128, 128, 64   # 128-query tiles over 64-key tiles
    aq, ak, av = synth.attention_inputs(int(cu_q[-1]), int(cu_kv[-1]), Hq, Hkv, Dh, seed=9, device=dev)
    ao = torch.empty_like(aq)
    dq, dkv, dcz = (torch.from_numpy(t).to(dev) for t in (cu_q, cu_kv, cz))
    aws = torch.empty(dg.dg_attention_workspace_bytes(len(seqs), 1024), dtype=torch.uint8, device=dev)
    attn = {}
    for W in (-1, 512):
        pairs, tiles, tiles_all = attention_counts(seqs, W, TQ, TK)
        ms = time_fn(lambda: dg.dg_attention(aq, ak, av, ao, dq, dkv, dcz, 1024, window=W, workspace=aws,
                                             stream=stream), reps=20)
        alg = 4.0 * pairs * Dh * Hq
        exe = 4.0 * tiles * TQ * TK * Dh * Hq
        attn["window_%d" % W if W >= 0 else "no_window"] = {
            "ms": ms, "tflops_allowed": alg / (ms * 1e-3) / 1e12, "tflops_executed": exe / (ms * 1e-3) / 1e12,
            "frac_tc_executed": exe / (ms * 1e-3) / 1e12 / peak_tc, "tiles_visited": int(tiles),
            "tiles_skipped_frac": 1.0 - tiles / tiles_all}
    attn["note"] = ("dg_attention timed alone (in the step's line: after 0.5 s idle, before the LM-head rows); "
                    "allowed = 4 D flops per allowed (query, key) pair per head, executed = the visited "
                    "128 x 64 tiles; frac against the burst bf16 peak")
    del aq, ak, av, ao
    return attn


def run_attention(args):
    """--attention: dg_attention alone (the rows above), one JSON line; a small command to
    profile the attention kernel on."""
    import torch
    import entropy_bounded_denoising_gb300 as dg
    from entropy_bounded_denoising_gb300 import synth, build
    build.build()
    dg.load()
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream()

    def _time(fn, reps=20):
        for _ in range(max(3, args.warmup)):
            fn()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / reps

    pk = _peaks()
    rows = _attention_rows(dg, synth, dev, stream, _time, pk["bf16_tflops_sustained"])
    if dg.dg_get_device_status():
        raise RuntimeError("device status set by dg_attention")
    print(json.dumps({"metric": "attention TFLOP/s (executed tiles) on a denoising batch", "rows": rows,
                      "gpu_launches_per_call": 2}), flush=True)
    return 0


# --------------------------------------------------------------------------- full loop
def run_loop(args):
    """The denoising loop of a workload from the Prefill case to convergence: every step runs
    dg_denoise_step, the feedback stages and dg_advance_params on the canvases still active
    (converged canvases drop out).  Each step's logits are generated between steps, outside
    the timed region; the value is positions/s over the timed library work (active positions
    summed over the steps), with steps/s and the loop's roofline fraction beside it."""
    import torch
    import entropy_bounded_denoising_gb300 as dg
    from entropy_bounded_denoising_gb300 import synth, build

    ws, rank, local = _dist()
    if ws > 1:
        import torch.distributed as tdist
        torch.cuda.set_device(local)
        tdist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if rank == 0:
        build.build()
    if ws > 1:
        tdist.barrier()
    dg.load()
    wl = synth.WORKLOADS[args.workload]
    n, L, V, d, h = wl.n, wl.L, wl.V, wl.d, wl.h
    base = synth.canvas_params(wl, step=0)
    base["flags"] = np.where(base["flags"] & dg.DG_ACTIVE, base["flags"] | dg.DG_SELF_COND, base["flags"]).astype(np.uint32)
    E, Wg, Wu, Wd = synth.weights(V, d, h, seed=wl.seed, device=dev)
    dt = dg.DG_BF16 if wl.dtype == "bf16" else dg.DG_FP32
    z = lambda shape, t, v=0: torch.full(shape, v, dtype=t, device=dev)
    canvas, prev, stable = z((n, L), torch.int32), z((n, L), torch.int32, -1), z((n,), torch.int32)
    acc, am, smp = z((n, L), torch.uint8), z((n, L), torch.int32), z((n, L), torch.int32)
    ent, lse, conv = z((n, L), torch.float32), z((n, L), torch.float32), z((n,), torch.uint8)
    delta = torch.empty((n, L, d), dtype=torch.bfloat16, device=dev)
    wsp = torch.empty(dg.dg_self_cond_workspace_bytes(n, L, d, h), dtype=torch.uint8, device=dev)
    dws = torch.empty(dg.dg_denoise_workspace_bytes(n, L, V, dt), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    seed = 0x5EED0000 + rank
    pk = _peaks()

    def one_loop(timed):
        params = dg.params_tensor(base, dev)
        dg.dg_canvas_init(canvas, n, L, V, params, seed, stream=stream)
        prev.fill_(-1)
        stable.zero_()
        total_ms, positions, steps, t_roof = 0.0, 0, 0, 0.0
        for t in range(int(base["max_steps"].max())):
            flags = dg.unpack_params(params)["flags"]
            active = (flags & dg.DG_ACTIVE) != 0
            if not active.any():
                break
            x = synth.logits(n, L, V, seed=wl.seed + 1000 * rank, step=t, scale=wl.scale,
                             spike_frac=wl.spike_frac, dtype=wl.dtype, device=dev)
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            dg.dg_denoise_step(x, params, seed, canvas, prev, stable, acc, am, smp, ent, lse, conv,
                               workspace=dws, stream=stream)
            dg.dg_self_cond_prepare(params, conv, n, L, d, h, delta, wsp, stream=stream)
            dg.dg_self_cond_pe(x, lse, params, E, h, wsp, stream=stream)
            dg.dg_self_cond_mlp(n, L, Wg, Wu, Wd, delta, wsp, stream=stream)
            dg.dg_advance_params(params, conv, n, stream=stream)
            b.record(stream)
            torch.cuda.synchronize()
            del x
            if timed:
                conv_h = conv.cpu().numpy().astype(bool)
                rows = int(active.sum()) * L
                sc_rows = int((active & ~conv_h).sum()) * L
                ar = _workload_arith(wl, sc_rows, rows)
                t_roof += max(ar["bytes"] / (pk["hbm_gbs"] * 1e9), ar["tc_flops"] / (pk["bf16_tflops_sustained"] * 1e12))
                total_ms += a.elapsed_time(b)
                positions += rows
                steps += 1
        return total_ms, positions, steps, t_roof

    for _ in range(max(0, args.warmup)):
        one_loop(False)   # whole warm-up loops (the first builds kernels' tensor maps and caches)
    if dg.dg_get_device_status():
        raise RuntimeError("device status set during the warm-up loop")
    with ClockSampler(local) as clk:
        time.sleep(0.3)
        clk.mark("t_start")
        launches0 = dg.dg_launch_count()
        total_ms, positions, steps, t_roof = one_loop(True)
        launches = dg.dg_launch_count() - launches0
        clk.mark("t_end")
    if dg.dg_get_device_status():
        raise RuntimeError("device status set during the timed loop")
    total_ms = max_over_ranks(total_ms, dev)
    if rank != 0:
        return 0
    line = {
        "metric": METRIC, "value": job_throughput(positions, ws, 1, total_ms), "unit": UNIT, "n_gpus": ws,
        "steps": steps, "warmup": args.warmup, "ms_per_step": total_ms / max(1, steps), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": dict(_config(wl), mode="full loop from the Prefill case until every canvas converges or "
                       "reaches its step cap; converged canvases drop out; logits generated between steps, "
                       "outside the timed region"),
        "steps_per_s": 1e3 * steps / total_ms, "positions": positions,
        "loop_roofline": {"t_roof_ms": t_roof * 1e3, "frac": t_roof * 1e3 / total_ms},
        "gpu_launches": launches, "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)
    if ws > 1:
        tdist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="batched", choices=["batched", "sweep", "ragged", "single", "tiny", "profile"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-extras", action="store_true", help="skip timing the rows around the step")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--from-hidden", action="store_true",
                    help="start each step from hidden states: the LM head fused with the step's statistics")
    ap.add_argument("--graph", action="store_true", help="time replays of the step captured as a CUDA graph")
    ap.add_argument("--attention", action="store_true",
                    help="time only the attention kernel on a denoising batch (one JSON line)")
    ap.add_argument("--loop", action="store_true",
                    help="time the workload's whole denoising loop (e.g. --workload sweep) instead of repeated steps")
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)
    if args.loop:
        return run_loop(args)
    if args.attention:
        return run_attention(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
