#!/usr/bin/env python
"""Benchmark of the Vertical-Slash sparse attention hot path on GB300.

One step = the whole path over one batch of synthetic input: online
estimation (vertical / slash selection), sparse index build, sparse forward
and sparse backward.  The headline workload is one Qwen2.5-3B-shaped
attention layer at 128K tokens (B=1, N=131072, Hq=16, Hkv=2, d=128,
kv=1024, ks=2048, last_q=64).

Prints ONE JSON line (rank 0).  ``value`` is the executed sparse FLOPs of the
forward + backward (the query-major cover credited at 4 d and 10 d per
covered entry) divided by the device time of a whole step, summed over
ranks.  Usage:

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME]

``--workload qwen3b-512k-striped8`` runs worker 0 of the 8-worker striped
ring instead (524288 global tokens, 64-token stripes) and adds each ring
step's executed FLOPs and time and their imbalance to the line.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "VS-sparse attn fwd+bwd effective TFLOP/s at 128K; % BF16 tensor peak; x vs dense"
UNIT = "TFLOP/s"
L2_FLUSH_BYTES = 256 << 20


def max_over_ranks(value: float, device, world: int) -> float:
    """The largest ``value`` over all ranks of the process group (a job's step
    time is its slowest rank's); ``value`` itself for one process."""
    if world <= 1:
        return float(value)
    import torch

    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_tflops(world: int, flops_per_rank: float, ms_max: float) -> float:
    """Whole-job throughput: every rank runs the same step (replicas), the job
    takes the slowest rank's time."""
    return world * flops_per_rank / (ms_max * 1e-3) / 1e12


def _traffic(workload: str, kernel: str):
    """DRAM bytes per launch of `kernel` at `workload` from the committed ncu
    summary (profiles/dram_traffic_<workload>.json), or None when there is
    none or the kernel's sources have changed since it was taken (the summary
    records each kernel's source digest: contents only, no paths)."""
    path = os.path.join(ROOT, "profiles", "dram_traffic_%s.json" % workload)
    try:
        with open(path) as fh:
            d = json.load(fh)
        from dynamic_vertical_slash_gb300 import _build

        rec = d["kernels"][kernel]
        if rec.get("source_digest") != _build.source_digest(kernel):
            return None
        return float(rec["bytes_per_launch"])
    except Exception:
        return None


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            d = json.load(fh)
        return {"bf16_burst": float(d["bf16_tflops"]), "bf16_sustained": float(d["bf16_tflops_sustained"]),
                "hbm_gbs": float(d["hbm_gbs"]), "source": "measured"}
    except Exception:
        return {"bf16_burst": 1900.0, "bf16_sustained": 1700.0, "hbm_gbs": 6800.0, "source": "fallback"}


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", self.gpu_id, "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self) -> dict:
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in getattr(self, "lines", []):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = max(mx, float(parts[2]))
            except ValueError:
                continue
            for name, flag in zip(names, parts[5:9]):
                if flag.lower() in ("active", "1", "yes"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx or None,
                "reasons": sorted(reasons), "samples": len(sm)}


def _gpu_id(dev_index: int) -> str:
    import torch

    try:
        return "GPU-" + str(torch.cuda.get_device_properties(dev_index).uuid)
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        return vis.split(",")[dev_index] if vis else str(dev_index)


# ------------------------------------------------------------------ accounting
def query_cover_units(iv: np.ndarray, is_: np.ndarray, N: int) -> np.ndarray:
    """Query-major work units (128 x 64 entries) of the kernels' cover of an
    unstriped selection, from the cover's definition: per head the selected
    offsets dilated to E = {u : some selected o in [u - 127, u]}, covered
    greedily by 64-wide intervals starting at u_s; the 128-row tile t takes one
    slash unit per u_s <= 128 t + 127 and one bar chunk per 64 selected
    columns whose first column is <= 128 t + 127.  Lists may end in -1.
    Returns int64 [B, H, 2] (slash tiles, bar chunks)."""
    B, H = iv.shape[:2]
    T = (N + 127) // 128
    last = 128 * np.arange(T, dtype=np.int64) + 127
    out = np.zeros((B, H, 2), np.int64)
    for b in range(B):
        for h in range(H):
            offs = np.unique(is_[b, h][is_[b, h] >= 0].astype(np.int64))
            starts, nxt, i = [], 0, 0
            while i < offs.size:  # maximal runs of E, then greedy 64-wide starts
                a, e = offs[i], offs[i] + 127
                i += 1
                while i < offs.size and offs[i] <= e + 1:
                    e = offs[i] + 127
                    i += 1
                u = max(a, nxt)
                while u <= e:
                    starts.append(u)
                    u += 64
                nxt = max(nxt, u)
            starts = np.asarray(starts, np.int64)
            cols = np.sort(iv[b, h][iv[b, h] >= 0].astype(np.int64))
            first = cols[::64]
            out[b, h, 0] = np.searchsorted(starts, last, side="right").sum()
            out[b, h, 1] = np.searchsorted(first, last, side="right").sum()
    return out


def mask_entries(iv: np.ndarray, is_: np.ndarray, N: int) -> np.ndarray:
    """|M| per head of the exact mask M[n, m] = (m <= n) and (m in iv or
    n - m in is) on an unstriped sequence of N tokens, in closed form: the
    column entries sum(N - m), the diagonal entries sum(N - o), minus the
    entries on both (for each selected column m, the selected offsets
    o <= N - 1 - m).  int64 [B, H]."""
    B, H = iv.shape[:2]
    out = np.zeros((B, H), np.int64)
    for b in range(B):
        for h in range(H):
            cols = np.unique(iv[b, h][iv[b, h] >= 0].astype(np.int64))
            offs = np.unique(is_[b, h][is_[b, h] >= 0].astype(np.int64))
            both = np.searchsorted(offs, N - 1 - cols, side="right").sum()
            out[b, h] = (N - cols).sum() + (N - offs).sum() - both
    return out


def block_mask_entries(iv: np.ndarray, is_: np.ndarray, N: int) -> np.ndarray:
    """|M| per head of the block-cover mask M[n, m] = (m <= n) and (m in iv or
    block diagonal D = floor(n/64) - floor(m/64) is active), D active iff a
    selected offset o has |o - 64 D| <= 63, for N a multiple of 64, in closed
    form: 2080 causal entries per diagonal block and 4096 per block of an
    active diagonal D >= 1 (N/64 - D of them), plus, per selected column m in
    block J, its causal rows on inactive diagonals (64 - m mod 64 in block J,
    64 in every later block).  int64 [B, H]."""
    assert N % 64 == 0
    nb = N // 64
    B, H = iv.shape[:2]
    out = np.zeros((B, H), np.int64)
    D = np.arange(nb, dtype=np.int64)
    for b in range(B):
        for h in range(H):
            offs = np.unique(is_[b, h][is_[b, h] >= 0].astype(np.int64))
            act = np.zeros(nb, bool)
            for dd in (0, 1):  # |o - 64 D| <= 63 holds for D = floor(o/64) and, if 64 does not divide o, the next
                c = offs // 64 + dd
                ok = (c < nb) & (np.abs(offs - 64 * c) <= 63)
                act[c[ok]] = True
            area = (2080 * nb if act[0] else 0) + int((4096 * (nb - D[1:]))[act[1:]].sum())
            inact = (~act).astype(np.int64)
            cum = np.cumsum(inact)  # cum[t] = inactive diagonals among 0..t
            cols = np.unique(iv[b, h][iv[b, h] >= 0].astype(np.int64))
            J = cols // 64
            area += int((inact[0] * (64 - cols % 64) + 64 * (cum[nb - 1 - J] - cum[0])).sum())
            out[b, h] = area
    return out


def step_flops(units_q: np.ndarray, entries: np.ndarray, B: int, N: int, Hq: int, d: int) -> dict:
    """Executed (query-major cover, 4 d + 10 d per covered entry), algorithmic
    (the same per entry of the exact mask, MagiAttention's cost = mask area)
    and dense causal FLOPs of one forward + backward."""
    area_q = float(units_q.sum()) * 128 * 64
    m = float(entries.sum())
    causal = B * Hq * N * (N + 1) / 2.0
    return {"executed": 14.0 * area_q * d, "algorithmic": 14.0 * m * d, "dense": 14.0 * causal * d,
            "mask_entries": m, "mask_density": m / causal, "executed_density": area_q / causal}


# ------------------------------------------------------------------ CPU oracle
def _oracle_inputs(x, h: int, hk: int):
    import synth

    f64 = lambda a: synth.bf16_to_f32(a).astype(np.float64)
    return (f64(x["q"][:, :, h:h + 1]), f64(x["k"][:, :, hk:hk + 1]), f64(x["v"][:, :, hk:hk + 1]),
            f64(x["dout"][:, :, h:h + 1]))


def oracle_step_sample(x, w, h: int, R: int):
    """One bounded sample of the whole step, run by the oracle as it stands:
    query head h's estimate and selection (Algorithm 1) and a complete
    forward + backward on its exact mask restricted to R query rows spread
    evenly over the sequence (O, LSE, dQ of those rows and the dK, dV they
    contribute to every key).  Returns (seconds, mask entries of the sample,
    seconds of the estimate + selection)."""
    import oracle

    q, k, v, do = _oracle_inputs(x, h, h // (w.Hq // w.Hkv))
    t0 = time.perf_counter()
    vs_, ss_ = oracle.estimate(q, k, w.last_q, w.scale)
    iv, is_ = oracle.select(vs_, ss_, w.kv, w.ks)
    t_est = time.perf_counter() - t0
    rows = np.sort(w.N - 1 - (w.N // R) * np.arange(R)).astype(np.int64)
    p = oracle.Problem(q[:, rows], k, v, iv, is_, w.scale, dout=do[:, rows], qpos=rows, n_global=w.N)
    t1 = time.perf_counter()
    oracle.attention(p)
    t_attn = time.perf_counter() - t1
    return t_attn + t_est, oracle.mask_count(p), t_est, t_attn


def oracle_baseline(x, w, target_s: float, heads, executed: float, algorithmic: float):
    """The oracle's time for a whole step, extrapolated from bounded samples
    (oracle_step_sample on the given query heads): per head the estimate plus
    N / R times the R-row forward + backward, summed over B * Hq heads.  Also
    its rates on the GPU line's two accountings (executed cover FLOPs and
    algorithmic mask FLOPs per step)."""
    import oracle

    R = 256
    _, _, _, ta = oracle_step_sample(x, w, heads[0], R)  # calibration
    R = int(max(64, min(w.N, R * target_s / max(1, len(heads)) / max(ta, 1e-3))))
    R = max(64, min(w.N, R))
    per_head, ent, secs = [], 0, 0.0
    for h in heads:
        t, e, te, ta = oracle_step_sample(x, w, h, R)
        per_head.append(te + ta * w.N / R)
        ent += e
        secs += t
    full = w.B * w.Hq * float(np.mean(per_head))
    return {"value": executed / full / 1e12, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
            "value_algorithmic": algorithmic / full / 1e12,
            "value_sample_mask_entries": 14.0 * w.d * ent / secs / 1e12,
            "extrapolated_full_step_s": full, "extrapolated": True,
            "sample": ("query heads %s of %s, each: the estimate + selection and a full forward + backward (O, LSE, "
                       "dQ, dK, dV) on the exact mask of %d query rows spread evenly over the sequence, fp64; "
                       "%.1f s of oracle time, %d mask entries. Whole step extrapolated as B*Hq * (estimate + N/R * "
                       "sample); value = the GPU line's executed FLOPs per step / that time, value_algorithmic = "
                       "14 d FLOPs per mask entry of the step / that time" % (list(heads), w.name, R, secs, ent))}


def _selection_all_heads(x, w):
    """The oracle's selection for every query head (outside any timing)."""
    import oracle

    iv = np.zeros((w.B, w.Hq, w.kv), np.int32)
    is_ = np.zeros((w.B, w.Hq, w.ks), np.int32)
    for h in range(w.Hq):
        q, k, _, _ = _oracle_inputs(x, h, h // (w.Hq // w.Hkv))
        a, c = oracle.estimate(q, k, w.last_q, w.scale)
        iv[:, h:h + 1], is_[:, h:h + 1] = oracle.select(a, c, w.kv, w.ks)
    return iv, is_


def reference_arm(args, w, x):
    """--impl reference: the oracle as it stands, on the host cores.  Each
    step is one bounded sample of the workload (oracle_step_sample, query
    head rotating with the step); the line's value puts it on the GPU line's
    accounting: executed cover FLOPs of a whole step over the extrapolated
    whole-step time."""
    import oracle

    iv, is_ = _selection_all_heads(x, w)
    fl = step_flops(query_cover_units(iv, is_, w.N), mask_entries(iv, is_, w.N), w.B, w.N, w.Hq, w.d)
    budget = max(1.0, 150.0 / max(1, args.steps + args.warmup))
    _, _, _, ta = oracle_step_sample(x, w, 0, 256)
    R = int(max(64, min(w.N, 256 * budget / max(ta, 1e-3))))
    for i in range(args.warmup):
        oracle_step_sample(x, w, i % w.Hq, R)
    times, full = [], []
    for i in range(args.steps):
        t, _, te, ta = oracle_step_sample(x, w, i % w.Hq, R)
        times.append(t)
        full.append(w.B * w.Hq * (te + ta * w.N / R))
    ms = 1e3 * statistics.mean(times)
    full_s = statistics.mean(full)
    value = fl["executed"] / full_s / 1e12
    sample = ("per step one query head (rotating) of the %s workload: estimate + selection and a full forward + "
              "backward on the exact mask of %d query rows spread evenly over the sequence, fp64; whole step "
              "extrapolated as B*Hq * (estimate + N/R * sample) = %.1f s; value = executed cover FLOPs of a whole "
              "step (%.4g, the GPU line's accounting) / that time" % (w.name, R, full_s, fl["executed"]))
    cpu = {"value": value, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle", "sample": sample,
           "value_algorithmic": fl["algorithmic"] / full_s / 1e12, "extrapolated_full_step_s": full_s,
           "extrapolated": True}
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": _config(w), "cpu_baseline": cpu,
            "flops": {"executed_per_step": fl["executed"], "algorithmic_per_step": fl["algorithmic"],
                      "mask_density": fl["mask_density"], "executed_density": fl["executed_density"]},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    return line


def _variant_kwargs(args, w):
    """VSAttention options of the selected variant of the path: the exact
    token mask with fixed budgets (the headline), the block-cover reading,
    top-p budgets (capped at --kv-cap / --ks-cap), or one selection per KV
    group."""
    if args.variant == "block":
        return {"block_cover": True}
    if args.variant == "shared":
        return {"shared": True}
    if args.variant == "shared-packed":
        return {"shared": True, "packed": True}
    if args.variant == "topp":
        return {"pv": args.pv, "ps": args.ps, "kv_cap": args.kv_cap, "ks_cap": args.ks_cap}
    return {}


def _variant_note(args, attn):
    if args.variant == "topp":
        kv, ks = (b.float().cpu().numpy() for b in attn.budgets)
        return {"name": "topp", "pv": args.pv, "ps": args.ps, "kv_cap": args.kv_cap, "ks_cap": args.ks_cap,
                "kv_mean": float(kv.mean()), "kv_min": int(kv.min()), "kv_max": int(kv.max()),
                "ks_mean": float(ks.mean()), "ks_min": int(ks.min()), "ks_max": int(ks.max())}
    return {"name": args.variant}


def _config(w):
    return {"workload": w.name, "B": w.B, "N": w.N, "Hq": w.Hq, "Hkv": w.Hkv, "d": w.d, "kv": w.kv, "ks": w.ks,
            "last_q": w.last_q, "parallelism": "replicas",
            "l2": "256 MiB buffer written between timed steps; Q/dO/O/dQ also exceed L2"}


# ------------------------------------------------------------------ GPU arm
def ours(args, w, x, rank, world):
    import torch

    import dynamic_vertical_slash_gb300 as vs
    from dynamic_vertical_slash_gb300.pipeline import dense_causal_flops, flop_counts

    dev = torch.device("cuda", torch.cuda.current_device())
    to_dev = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
    q, k, v, do = to_dev(x["q"]), to_dev(x["k"]), to_dev(x["v"]), to_dev(x["dout"])
    vkw = _variant_kwargs(args, w)
    attn = vs.VSAttention(w.B, w.N, w.Hq, w.Hkv, w.d, vkw.pop("kv_cap", w.kv), vkw.pop("ks_cap", w.ks), device=dev,
                          last_q=w.last_q, scale=w.scale, **vkw)
    args._attn_kwargs = (attn.kv, attn.ks, vkw)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def step():
        attn.forward(q, k, v)
        attn.backward(do)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    attn.check()
    counts = attn.counts()
    fl = flop_counts(counts, w.d)
    executed = fl["fwd_executed"] + fl["bwd_executed"]
    acct = _accounting(attn, counts, w)

    # ---------------- timed region: K steps, L2 flushed between them
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    vs.trace_reset()
    launches0 = vs.launch_count()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(_gpu_id(dev.index)) as clk:
        vs.trace_enable(True)
        for i in range(args.steps):
            flush.zero_()
            ev[i][0].record()
            step()
            ev[i][1].record()
        vs.trace_enable(False)
        torch.cuda.synchronize()
    launches = vs.launch_count() - launches0
    step_ms = [a.elapsed_time(b) for a, b in ev]
    trace = vs.trace_report()
    vs.trace_reset()
    attn.check()
    ms = statistics.mean(step_ms)
    ms_max = max_over_ranks(ms, dev, world)
    if world > 1:
        torch.distributed.barrier()
    value = job_tflops(world, executed, ms_max)

    # per-kernel breakdown and the roofline of the dominant attention kernel
    per_kernel = {name: {"launches": c, "ms_total": t, "ms_avg": t / max(c, 1)} for name, (c, t) in trace.items()}
    units = fl["units"]
    tile = 128 * 64 * w.d
    issued_per_step = {"fwd": 4.0 * tile * (units[0] + units[1]), "bwd_dq": 6.0 * tile * (units[0] + units[1]),
                       "bwd_dkv_slash": 8.0 * tile * units[2], "bwd_dkv_bar": 8.0 * tile * units[3]}
    peaks = _peaks()
    att = {kname: per_kernel[kname] for kname in issued_per_step if kname in per_kernel}
    dom = max(att, key=lambda kname: att[kname]["ms_total"]) if att else None
    roofline = None
    if dom:
        achieved = issued_per_step[dom] / (att[dom]["ms_avg"] * 1e-3) / 1e12
        roofline = {"kernel": dom, "bound": "tensor", "achieved": achieved, "peak": peaks["bf16_sustained"],
                    "unit": "TFLOP/s", "frac": achieved / peaks["bf16_sustained"],
                    "traffic": _traffic(w.name, dom), "traffic_unit": "bytes per launch (ncu dram read + write)",
                    "peak_kind": "sustained bf16 (%s): the kernel is timed inside a long step" % peaks["source"]}
        for kname in att:
            att[kname]["issued_tflops"] = issued_per_step[kname] / (att[kname]["ms_avg"] * 1e-3) / 1e12
    attn_ms = sum(per_kernel[kname]["ms_avg"] for kname in att)

    # ---------------- end to end through the public API, host buffers (run
    # right after the timed region, before the optional dense comparison)
    e2e = None
    if not args.no_e2e:
        e2e = _e2e(args, w, attn, q, k, v, do, dev, world, executed)

    extra = {}
    # ---------------- same kernels on the dense causal mask (every offset selected)
    if rank == 0 and not args.no_dense:
        ks_all = torch.arange(w.N, dtype=torch.int32, device=dev).repeat(w.B, w.Hq, 1).contiguous()
        arena_d = vs.vs_build_block_index(q, k, attn.v_idx, ks_all)
        o_d, lse_d = torch.empty_like(q), torch.empty(w.B, w.Hq, w.N, device=dev)
        dq_d, dk_d, dv_d = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        import ctypes
        ws_b = torch.zeros(vs.lib().vs_attn_bwd_workspace(ctypes.byref(vs.make_shape(q, k)), w.kv), dtype=torch.uint8,
                           device=dev)
        ws_f = torch.zeros(256, dtype=torch.uint8, device=dev)

        def dense_step():
            vs.vs_attn_fwd(q, k, v, arena_d, w.scale, o_d, lse_d, None, ws_f)
            vs.vs_attn_bwd(q, k, v, o_d, lse_d, do, arena_d, w.kv, w.scale, dq_d, dk_d, dv_d, None, ws_b)

        dense_step()
        torch.cuda.synchronize()
        dts = []
        for _ in range(args.dense_steps):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            dense_step()
            b.record()
            torch.cuda.synchronize()
            dts.append(a.elapsed_time(b))
        if vs.vs_check_status(ws_f) or vs.vs_check_status(ws_b) or vs.vs_check_status(arena_d):
            raise RuntimeError("dense comparison recorded a device error")
        dense_ms = statistics.mean(dts)
        dfl = dense_causal_flops(w.B, w.N, w.Hq, w.d)
        extra["dense"] = {"ms_fwd_bwd": dense_ms, "tflops": (dfl["fwd"] + dfl["bwd"]) / (dense_ms * 1e-3) / 1e12}
        extra["x_vs_dense"] = dense_ms / ms
        extra["x_vs_dense_attention_only"] = dense_ms / attn_ms if attn_ms else None
        del arena_d, o_d, dq_d, dk_d, dv_d, ws_b

    dense_f = dense_causal_flops(w.B, w.N, w.Hq, w.d)
    cfg = _config(w)
    if args.variant != "exact":
        cfg["variant"] = _variant_note(args, attn)
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": cfg,
            "roofline": roofline, "e2e": e2e, "gpu_launches": launches,
            "pct_bf16_peak": 100.0 * value / world / peaks["bf16_burst"],
            "value_algorithmic": job_tflops(world, acct["algorithmic_per_step"], ms_max) if acct else None,
            "flops": {"executed_per_step": executed, "issued_per_step": fl["fwd_issued"] + fl["bwd_issued"],
                      "dense_causal_per_step": dense_f["fwd"] + dense_f["bwd"],
                      "executed_density": executed / (dense_f["fwd"] + dense_f["bwd"]), "units": units,
                      **(acct or {})},
            "kernels": per_kernel, "attention_ms_per_step": attn_ms, "step_ms_all": step_ms}
    line.update(extra)
    return line, clk.summary()


def _accounting(attn, counts, w):
    """Algorithmic FLOPs and mask density of the step on the GPU: |M| per head
    counted by vs_ring_work with one worker (every mask entry), checked against
    the closed form on the host; the host model of the query-major cover is
    checked against the arena's unit counts.  None for the block-cover variant
    (its mask is not the exact VS mask)."""
    import torch

    import dynamic_vertical_slash_gb300 as vs

    if attn.block_cover:
        # the block-cover mask: its area from the host's closed form
        iv, is_ = attn.v_idx.cpu().numpy(), attn.s_idx.cpu().numpy()
        per_head = block_mask_entries(iv, is_, w.N)
        gpu_u = np.asarray(counts).reshape(w.B, w.Hq, 4)[..., :2]
        fl = step_flops(gpu_u, per_head, w.B, w.N, w.Hq, w.d)
        return {"algorithmic_per_step": fl["algorithmic"], "mask_entries": int(per_head.sum()),
                "mask_density": fl["mask_density"], "mask_entries_source": "host closed form of the block-cover mask",
                "executed_over_algorithmic": fl["executed"] / fl["algorithmic"] if fl["algorithmic"] else None}
    per_head = np.zeros((w.B, w.Hq), np.int64)
    for b in range(w.B):
        for h in range(w.Hq):
            cnt = vs.vs_ring_work(attn.v_idx[b:b + 1, h:h + 1].contiguous(),
                                  attn.s_idx[b:b + 1, h:h + 1].contiguous(), w.N, 1)
            per_head[b, h] = int(cnt.sum().item())
    torch.cuda.synchronize()
    iv, is_ = attn.v_idx.cpu().numpy(), attn.s_idx.cpu().numpy()
    host_m = mask_entries(iv, is_, w.N)
    gpu_u = np.asarray(counts).reshape(w.B, w.Hq, 4)[..., :2]
    # the host model is of the one-head-per-tile cover
    host_u = None if attn.packed else query_cover_units(iv, is_, w.N)
    fl = step_flops(gpu_u, per_head, w.B, w.N, w.Hq, w.d)
    dens = per_head / (w.N * (w.N + 1) / 2.0)
    return {"algorithmic_per_step": fl["algorithmic"], "mask_entries": int(per_head.sum()),
            "mask_density": fl["mask_density"], "mask_density_per_head": [round(float(x), 5) for x in dens.ravel()],
            "executed_over_algorithmic": fl["executed"] / fl["algorithmic"] if fl["algorithmic"] else None,
            "host_checks": {"mask_entries_closed_form_equal": bool(np.array_equal(host_m, per_head)),
                            "cover_units_equal": None if host_u is None else bool(np.array_equal(host_u, gpu_u))}}


def _e2e(args, w, attn, q, k, v, do, dev, world, executed):
    """The same metric through the public API (VSAttention), with every
    step's inputs copied in from pinned host memory and its results (O, dQ,
    dK, dV) copied back, all inside the timed region.

    Two schedules: `serial` (copy in, compute, copy out, one after the other
    on one stream) and `pipelined` (the line's value): two VSAttention
    instances and two input buffer sets alternate between steps, step i's
    host->device copy runs on its own stream while step i-1 computes (dO may
    still be arriving while step i's forward runs), and its results go back
    on a third stream (O while step i's backward runs, the gradients while
    step i+1 computes) -- the usual prefetching of the next batch.  Device time from CUDA events spanning
    the first copy to the last one; SM clocks are sampled during both timed
    loops and reported beside each (a long run under load can be power
    capped below the clocks of the short kernel-timed region)."""
    import torch

    import dynamic_vertical_slash_gb300 as vs

    pin = lambda t: torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
    hin = [pin(t) for t in (q, k, v, do)]
    for hbuf, t in zip(hin, (q, k, v, do)):
        hbuf.copy_(t)
    hout = [pin(t) for t in (q, q, k, v)]
    h2d = sum(t.numel() * t.element_size() for t in hin)
    d2h = sum(t.numel() * t.element_size() for t in hout)

    def reduce_max(ms):
        return max_over_ranks(ms, dev, world)

    # ---- serial
    din0 = [torch.empty_like(t) for t in (q, k, v, do)]

    def serial_step():
        for dst, src in zip(din0, hin):
            dst.copy_(src, non_blocking=True)
        o, _ = attn.forward(din0[0], din0[1], din0[2])
        gq, gk, gv = attn.backward(din0[3])
        for dst, src in zip(hout, (o, gq, gk, gv)):
            dst.copy_(src, non_blocking=True)

    serial_step()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(_gpu_id(dev.index)) as clk_s:
        a.record()
        for _ in range(args.steps):
            serial_step()
        b.record()
        torch.cuda.synchronize()
    serial_ms = reduce_max(a.elapsed_time(b) / args.steps)
    attn.check()

    # ---- pipelined
    kv_cap, ks_cap, vkw = args._attn_kwargs
    att = [attn, vs.VSAttention(w.B, w.N, w.Hq, w.Hkv, w.d, kv_cap, ks_cap, device=dev, last_q=w.last_q, scale=w.scale,
                                **vkw)]
    din = [din0, [torch.empty_like(t) for t in (q, k, v, do)]]
    s_in, s_comp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()

    def run(n):
        start = torch.cuda.Event(enable_timing=True)
        start.record(s_in)
        comp_done, out_done = [None, None], [None, None]
        for i in range(n):
            sl = i % 2
            with torch.cuda.stream(s_in):
                if comp_done[sl] is not None:  # step i - 2 has finished reading this input set
                    s_in.wait_event(comp_done[sl])
                for dst, src in zip(din[sl][:3], hin[:3]):
                    dst.copy_(src, non_blocking=True)
                qkv_in = torch.cuda.Event()
                qkv_in.record(s_in)
                din[sl][3].copy_(hin[3], non_blocking=True)  # dO: needed by the backward only
                do_in = torch.cuda.Event()
                do_in.record(s_in)
            s_comp.wait_event(qkv_in)
            if out_done[sl] is not None:  # step i - 2's results have left this instance's buffers
                s_comp.wait_event(out_done[sl])
            o, _ = att[sl].forward(din[sl][0], din[sl][1], din[sl][2], stream=s_comp)
            fwd_done = torch.cuda.Event()
            fwd_done.record(s_comp)
            s_comp.wait_event(do_in)
            gq, gk, gv = att[sl].backward(din[sl][3], stream=s_comp)
            cd = torch.cuda.Event()
            cd.record(s_comp)
            comp_done[sl] = cd
            with torch.cuda.stream(s_out):
                s_out.wait_event(fwd_done)  # O leaves while the backward runs
                hout[0].copy_(o, non_blocking=True)
                s_out.wait_event(cd)
                for dst, src in zip(hout[1:], (gq, gk, gv)):
                    dst.copy_(src, non_blocking=True)
                od = torch.cuda.Event()
                od.record(s_out)
                out_done[sl] = od
        end = torch.cuda.Event(enable_timing=True)
        end.record(s_out)
        return start, end

    run(2)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    with ClockSampler(_gpu_id(dev.index)) as clk_p:
        start, end = run(args.steps)
        torch.cuda.synchronize()
    pipe_ms = reduce_max(start.elapsed_time(end) / args.steps)
    for a_ in att:
        a_.check()
    return {"value": job_tflops(world, executed, pipe_ms), "unit": UNIT, "ms_per_step": pipe_ms,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "clocks": clk_p.summary(),
            "serial": {"value": job_tflops(world, executed, serial_ms), "ms_per_step": serial_ms,
                       "clocks": clk_s.summary()},
            "path": "VSAttention.forward/backward (C ABI) with pinned host inputs and outputs; pipelined: next "
                    "step's inputs copied in and previous step's results copied out on separate streams while a "
                    "step computes (two instances, two input sets; dO copied in during the forward, O copied out "
                    "during the backward)"}


def striped(args, w, x, rank, world):
    """Striped-shard workload: worker 0 of ``w.world`` runs the whole ring on
    one GPU (global selection, one index per ring step, forward merging each
    step's partial, backward accumulating dQ and emitting each source shard's
    dK / dV).  Reports per ring step the executed FLOPs and device time and
    their imbalance (max / mean)."""
    import torch

    import dynamic_vertical_slash_gb300 as vs
    from dynamic_vertical_slash_gb300.pipeline import dense_causal_flops, flop_counts

    dev = torch.device("cuda", torch.cuda.current_device())
    to_dev = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
    W = w.world
    q, k, v, do = to_dev(x["q"]), to_dev(x["k"]), to_dev(x["v"]), to_dev(x["dout"])
    q0 = vs.striped_permute(q, W, w.stripe, only_rank=0)
    do0 = vs.striped_permute(do, W, w.stripe, only_rank=0)
    ksh, vsh = vs.striped_permute(k, W, w.stripe), vs.striped_permute(v, W, w.stripe)
    wk = vs.StripedWorker(w.B, w.N, w.Hq, w.Hkv, w.d, w.kv, w.ks, W, rank=0, stripe=w.stripe, device=dev,
                          last_q=w.last_q, scale=w.scale, inner=args.inner)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    # block-level striping inside the step: worker 0's Q and dO shards, every KV shard
    permuted = [(q, q0, 0), (do, do0, 0), (k, ksh, -1), (v, vsh, -1)]
    permute_bytes = 2.0 * sum(y.numel() * y.element_size() for _, y, _ in permuted)  # read + write

    def step():
        for src, dst, r in permuted:
            vs.striped_permute(src, W, w.stripe, only_rank=r, y=dst)
        wk.select(q, k)
        wk.build_index(q0, ksh)
        wk.forward(q0, ksh, vsh)
        wk.backward(do0)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    wk.check()
    counts = wk.counts()
    per = [flop_counts(c, w.d) for c in counts]
    executed = sum(f["fwd_executed"] + f["bwd_executed"] for f in per)

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    vs.trace_reset()
    launches0 = vs.launch_count()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(_gpu_id(dev.index)) as clk:
        vs.trace_enable(True)
        for i in range(args.steps):
            flush.zero_()
            ev[i][0].record()
            step()
            ev[i][1].record()
        vs.trace_enable(False)
        torch.cuda.synchronize()
    launches = vs.launch_count() - launches0
    step_ms = [a.elapsed_time(b) for a, b in ev]
    ring_ms = wk.step_times()  # the last timed step's ring steps
    trace = vs.trace_report()
    vs.trace_reset()
    wk.check()
    ms = max_over_ranks(statistics.mean(step_ms), dev, world)
    value = job_tflops(world, executed, ms)
    per_kernel = {name: {"launches": c, "ms_total": t, "ms_avg": t / max(c, 1)} for name, (c, t) in trace.items()}
    peaks = _peaks()
    tile = 128 * 64 * w.d
    units = np.sum([f["units"] for f in per], axis=0)
    issued = {"fwd": 4.0 * tile * (units[0] + units[1]), "bwd_dq": 6.0 * tile * (units[0] + units[1]),
              "bwd_dkv_slash": 8.0 * tile * units[2], "bwd_dkv_bar": 8.0 * tile * units[3]}
    att = {kn: per_kernel[kn] for kn in issued if kn in per_kernel}
    dom = max(att, key=lambda kn: att[kn]["ms_total"])
    achieved = issued[dom] / (att[dom]["ms_total"] / args.steps * 1e-3) / 1e12
    roofline = {"kernel": dom, "bound": "tensor", "achieved": achieved, "peak": peaks["bf16_sustained"],
                "unit": "TFLOP/s", "frac": achieved / peaks["bf16_sustained"], "traffic": _traffic(w.name, dom),
                "peak_kind": "sustained bf16 (%s): all ring steps of the kernel per timed step" % peaks["source"]}
    ring = []
    for s in range(W):
        f = per[s]
        ring.append({"step": s, "src": wk.source(s), "executed_flops": f["fwd_executed"] + f["bwd_executed"],
                     "units": f["units"], "ms_fwd": ring_ms[s][0], "ms_bwd": ring_ms[s][1]})
    fl = np.array([r["executed_flops"] for r in ring])
    tm = np.array([r["ms_fwd"] + r["ms_bwd"] for r in ring])
    dense_f = dense_causal_flops(w.B, w.N, w.Hq, w.d)
    cfg = _config(w)
    cfg.update({"world": W, "stripe": w.stripe, "worker": 0,
                "ring": ("hierarchical: nodes of %d cards, inner rings inside an outer ring" % args.inner
                         if args.inner else "flat: src = -s mod world") + "; KV shards local"})
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": cfg, "roofline": roofline,
            "e2e": None, "gpu_launches": launches,
            "pct_bf16_peak": 100.0 * value / world / peaks["bf16_burst"],
            "flops": {"executed_per_step": executed,
                      "dense_causal_worker_per_step": (dense_f["fwd"] + dense_f["bwd"]) / W,
                      "executed_density": executed / ((dense_f["fwd"] + dense_f["bwd"]) / W)},
            "ring_steps": ring,
            "imbalance": {"flops_max_over_mean": float(fl.max() / fl.mean()),
                          "ms_max_over_mean": float(tm.max() / tm.mean())},
            "kernels": per_kernel, "step_ms_all": step_ms}
    line["layouts"] = _layout_work(wk.v_idx, wk.s_idx, w.N, W)
    if args.layouts:
        line["layouts_measured"] = _layouts_measured(args, w, q, k, v, do, dev, wk.v_idx, wk.s_idx)
    ent = np.array(line["layouts"]["striped"]["entries_per_step_worker"], np.float64)[:, 0]  # worker 0, per step
    for r in ring:
        r["mask_entries"] = int(ent[r["step"]])
        r["algorithmic_flops"] = 14.0 * w.d * ent[r["step"]]
    alg = 14.0 * w.d * float(ent.sum())
    line["value_algorithmic"] = job_tflops(world, alg, ms)
    line["flops"].update({"algorithmic_per_step": alg, "executed_over_algorithmic": executed / alg,
                          "mask_density_worker": float(ent.sum()) / (w.B * w.Hq * w.N * (w.N + 1) / 2.0 / W)})
    line["imbalance"]["algorithmic_max_over_mean"] = float(ent.max() / ent.mean())
    if "striped_permute" in per_kernel:
        pms = per_kernel["striped_permute"]["ms_total"] / args.steps
        line["permute"] = {"ms_per_step": pms, "bytes_per_step": permute_bytes,
                           "gbs": permute_bytes / (pms * 1e-3) / 1e9, "peak_gbs": peaks["hbm_gbs"],
                           "frac": permute_bytes / (pms * 1e-3) / 1e9 / peaks["hbm_gbs"],
                           "what": "worker 0's Q and dO shards and all KV shards, 64-token stripes; bytes = "
                                   "read + write of the permuted elements"}
    if args.all_workers:
        line["workers"] = _all_workers(args, w, q, k, v, to_dev(x["dout"]), dev)
    return line, clk.summary()


def _layout_work(iv, is_, N, W):
    """Effective work (mask entries) of every worker and ring step under the
    striped and the ZigZag layout of the same global selection (computed on
    the GPU, outside the timed region), and its imbalance: worker-level =
    max / mean over the workers at one ring step, step-level = max / mean over
    the ring steps of one worker, each reported as mean and max; plus the
    imbalance of the workers' totals."""
    import dynamic_vertical_slash_gb300 as vs

    out = {}
    for layout in ("striped", "zigzag"):
        M = vs.vs_ring_work(iv, is_, N, W, layout).cpu().numpy().astype(np.float64)
        st = np.array([[M[r, (r - s) % W] for r in range(W)] for s in range(W)])  # [step][worker]
        wl = st.max(1) / st.mean(1)
        sl = st.max(0) / st.mean(0)
        tot = M.sum(1)
        out[layout] = {"entries_per_step_worker": st.astype(np.int64).tolist(),
                       "worker_level_mean": float(wl.mean()), "worker_level_max": float(wl.max()),
                       "step_level_mean": float(sl.mean()), "step_level_max": float(sl.max()),
                       "worker_totals_max_over_mean": float(tot.max() / tot.mean())}
    return out


def _ring_times(wk, q_r, ksh, vsh, do_r, reps: int):
    """Per ring step of one worker: device time (forward + backward, mean over
    `reps` timed repetitions after one warm-up) and executed FLOPs."""
    import torch

    from dynamic_vertical_slash_gb300.pipeline import flop_counts

    wk.build_index(q_r, ksh)
    wk.forward(q_r, ksh, vsh)
    wk.backward(do_r)
    torch.cuda.synchronize()
    wk.check()
    W = len(wk.events)
    ms = np.zeros(W)
    for _ in range(reps):
        wk.forward(q_r, ksh, vsh)
        wk.backward(do_r)
        torch.cuda.synchronize()
        ms += np.array([a + b for a, b in wk.step_times()])
    wk.check()
    fl = [flop_counts(c, wk.d) for c in wk.counts()]
    return ms / reps, np.array([f["fwd_executed"] + f["bwd_executed"] for f in fl])


def _layouts_measured(args, w, q, k, v, do, dev, iv, is_):
    """The ring run on the GPU under both layouts of the same global
    selection: striped (64-token stripes) and ZigZag (2W chunks, worker r
    holds chunks r and 2W - 1 - r; each step is its causal chunk pairs).  For
    worker 0 (every worker with --all-workers): per ring step the device time
    and executed FLOPs; step-level imbalance = max / mean over a worker's
    steps; worker-level imbalance = max / mean over the workers at one step
    (mean and max over the steps); the imbalance of the workers' total times."""
    import torch

    import dynamic_vertical_slash_gb300 as vs

    W = w.world
    workers = range(W) if args.all_workers else [0]
    out = {}
    for layout in ("striped", "zigzag"):
        ksh, vsh = vs.ring_permute(k, W, layout), vs.ring_permute(v, W, layout)
        per = []
        for r in workers:
            q_r = vs.ring_permute(q, W, layout, only_rank=r)
            do_r = vs.ring_permute(do, W, layout, only_rank=r)
            cls = vs.StripedWorker if layout == "striped" else vs.ZigZagWorker
            wk = cls(w.B, w.N, w.Hq, w.Hkv, w.d, w.kv, w.ks, W, rank=r, device=dev, last_q=w.last_q, scale=w.scale)
            wk.v_idx.copy_(iv)
            wk.s_idx.copy_(is_)
            ms, fl = _ring_times(wk, q_r, ksh, vsh, do_r, args.layout_reps)
            per.append({"worker": r, "src": [wk.source(s) for s in range(W)], "ms": ms.tolist(),
                        "executed_flops": fl.tolist(), "step_imbalance_ms": float(ms.max() / ms.mean()),
                        "step_imbalance_flops": float(fl.max() / fl.mean())})
            del wk, q_r, do_r
            torch.cuda.synchronize()
        rec = {"per_worker": per}
        if len(per) > 1:
            st = np.array([[p["ms"][s] for p in per] for s in range(W)])  # [step][worker]
            wl = st.max(1) / st.mean(1)
            tot = st.sum(0)
            rec.update({"worker_level_ms_mean": float(wl.mean()), "worker_level_ms_max": float(wl.max()),
                        "worker_totals_ms_max_over_mean": float(tot.max() / tot.mean())})
        out[layout] = rec
        del ksh, vsh
        torch.cuda.synchronize()
    out["how"] = ("flat ring src = rank - s mod W; one warm-up, then the mean of %d timed repetitions per step "
                  "(CUDA events around each step's forward and backward)" % args.layout_reps)
    return out


def _all_workers(args, w, q, k, v, do, dev):
    """Every worker's ring on this GPU, one after the other: per worker and
    ring step the executed FLOPs (from its index) and device time (one timed
    step after one warm-up), and the imbalance across workers of their total
    time and FLOPs."""
    import torch

    import dynamic_vertical_slash_gb300 as vs
    from dynamic_vertical_slash_gb300.pipeline import flop_counts

    W = w.world
    ksh, vsh = vs.striped_permute(k, W, w.stripe), vs.striped_permute(v, W, w.stripe)
    out = []
    for r in range(W):
        q_r = vs.striped_permute(q, W, w.stripe, only_rank=r)
        do_r = vs.striped_permute(do, W, w.stripe, only_rank=r)
        wk = vs.StripedWorker(w.B, w.N, w.Hq, w.Hkv, w.d, w.kv, w.ks, W, rank=r, stripe=w.stripe, device=dev,
                              last_q=w.last_q, scale=w.scale, inner=args.inner)
        wk.select(q, k)
        wk.build_index(q_r, ksh)
        for _ in range(2):
            wk.forward(q_r, ksh, vsh)
            wk.backward(do_r)
        torch.cuda.synchronize()
        wk.check()
        fl = [flop_counts(c, w.d) for c in wk.counts()]
        ms = wk.step_times()
        out.append({"worker": r, "src": [wk.source(s) for s in range(W)],
                    "executed_flops": [f["fwd_executed"] + f["bwd_executed"] for f in fl],
                    "ms": [a + b for a, b in ms]})
        del wk, q_r, do_r
    tot_ms = np.array([sum(o["ms"]) for o in out])
    tot_fl = np.array([sum(o["executed_flops"]) for o in out])
    step_ms = np.array([o["ms"] for o in out])
    return {"per_worker": out,
            "imbalance_ms_max_over_mean": float(tot_ms.max() / tot_ms.mean()),
            "imbalance_flops_max_over_mean": float(tot_fl.max() / tot_fl.mean()),
            "step_imbalance_ms_max_over_mean": float(step_ms.max() / step_ms.mean())}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="qwen3b-128k")
    ap.add_argument("--dense-steps", type=int, default=2)
    ap.add_argument("--no-dense", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--inner", type=int, default=0,
                    help="striped workloads: cards per node for the hierarchical ring order (0 = flat ring)")
    ap.add_argument("--variant", choices=["exact", "block", "topp", "shared", "shared-packed"], default="exact",
                    help="path variant: exact token mask with fixed budgets (headline), block-cover slashes, "
                         "top-p budgets, one selection per KV group, or that with the group's query heads "
                         "packed into the query-major tiles")
    ap.add_argument("--pv", type=float, default=0.9, help="top-p variant: vertical mass fraction")
    ap.add_argument("--ps", type=float, default=0.9, help="top-p variant: slash mass fraction")
    ap.add_argument("--kv-cap", type=int, default=4096, help="top-p variant: vertical list capacity")
    ap.add_argument("--ks-cap", type=int, default=8192, help="top-p variant: slash list capacity")
    ap.add_argument("--layouts", action="store_true",
                    help="striped workloads: also time the ring under both layouts (striped and ZigZag)")
    ap.add_argument("--layout-reps", type=int, default=2, help="timed repetitions per layout and worker")
    ap.add_argument("--all-workers", action="store_true",
                    help="striped workloads: also run every worker's ring and report the imbalance across workers")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    import synth

    w = synth.workloads()[args.workload]

    if args.impl == "reference":
        if rank != 0:
            return
        x = synth.make_batch(w)
        print(json.dumps(reference_arm(args, w, x)), flush=True)
        return

    import torch

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        import datetime

        torch.distributed.init_process_group("nccl", timeout=datetime.timedelta(minutes=10))
    x = synth.make_batch(w)
    line, clocks = (striped if w.world > 1 else ours)(args, w, x, rank, world)
    line["clocks"] = clocks
    if rank == 0 and world == 1 and w.world == 1 and not args.no_cpu_baseline and line["flops"].get("mask_entries"):
        line["cpu_baseline"] = oracle_baseline(x, w, 20.0, [0, w.Hq - 1], line["flops"]["executed_per_step"],
                                               line["flops"]["algorithmic_per_step"])
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
