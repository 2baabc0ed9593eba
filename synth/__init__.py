"""Seeded synthetic inputs for Vertical-Slash sparse attention.

This module is shared by the tests, the benchmark, the CPU oracle side and
the CUDA side.  It holds none of the method's arithmetic: it only draws
Gaussian tensors, applies rotary position embeddings and plants vertical and
slash structure, then rounds to bf16.

Recipe for one sequence (seeded numpy PCG64 streams spawned from the seed,
float32 until the final round-to-nearest-even bf16):

1. Q, K, V, dO ~ i.i.d. N(0, 1) with shape [N, H, d].
2. Rotate-half RoPE on Q and K, theta_i = 10000^(-2i/d) for i < d/2, pairing
   channel i with i + d/2, positions 0..N-1 (the convention whose dot product
   is the expansion in the proof of Theorem 3.1 of the MTraining paper).
3. Vertical plant: per KV head, ``n_out`` key rows chosen without
   replacement are multiplied by 4 (outlier tokens with large key norm,
   section 3.2).
4. Slash plant: for each planted offset o and every n >= o, in post-RoPE
   space q[n, h] += c * k[n - o, h // g] with c = gamma / sqrt(#planted
   offsets).  Each planted diagonal gains about gamma * sqrt(d / #planted)
   logits; the other logits gain noise of standard deviation about gamma.
   Planted offsets are either ``n_slash`` random offsets in [1, N/8) or the
   contiguous band [1, w].
"""
from __future__ import annotations

import dataclasses
import math
import os
from typing import List, Optional, Sequence

import numpy as np

ROPE_THETA = 10000.0
OUTLIER_SCALE = 4.0
SLASH_GAMMA = 1.0


def bf16_round(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round to nearest, ties to even."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    rounding = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    out = ((u + rounding) >> np.uint32(16)).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        out[nan] = np.uint16(0x7FC0)
    return out


def bf16_to_f32(u: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> exact float32 values."""
    return (np.ascontiguousarray(u, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def rope_tables(N: int, d: int, theta: float = ROPE_THETA, positions: Optional[np.ndarray] = None):
    half = d // 2
    inv = theta ** (-2.0 * np.arange(half, dtype=np.float64) / d)
    pos = np.arange(N, dtype=np.float64) if positions is None else np.asarray(positions, np.float64)
    ang = pos[:, None] * inv[None, :]
    return np.cos(ang).astype(np.float32), np.sin(ang).astype(np.float32)


def apply_rope(x: np.ndarray, cos: np.ndarray, sin: np.ndarray) -> np.ndarray:
    """Rotate-half RoPE on x [N, H, d] (float32), in place and returned."""
    half = x.shape[-1] // 2
    c = cos[:, None, :]
    s = sin[:, None, :]
    lo = x[..., :half].copy()
    hi = x[..., half:].copy()
    x[..., :half] = lo * c - hi * s
    x[..., half:] = hi * c + lo * s
    return x


@dataclasses.dataclass
class SeqSpec:
    """Planting recipe of one sequence."""
    seed: int
    n_out: int = 0                 # outlier key columns per KV head
    n_slash: int = 0               # random planted diagonals in [1, N/8)
    band: int = 0                  # or a contiguous planted band [1, band]
    gamma: float = SLASH_GAMMA


@dataclasses.dataclass
class Workload:
    """A VS attention workload: shapes, budgets and per-sequence recipes."""
    name: str
    N: int
    Hq: int
    Hkv: int
    d: int
    kv: int
    ks: int
    seqs: List[SeqSpec]
    last_q: int = 64
    world: int = 1                 # striped-shard mode: number of workers
    stripe: int = 64

    @property
    def B(self) -> int:
        return len(self.seqs)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)


def workloads() -> dict:
    """The named workloads (Qwen2.5-3B attention shapes: 16 query heads,
    2 KV heads, head_dim 128, except the tiny case)."""
    W = {}
    W["tiny-1k"] = Workload("tiny-1k", N=1024, Hq=2, Hkv=1, d=64, kv=32, ks=32,
                            seqs=[SeqSpec(seed=1, n_out=8)])
    W["qwen3b-32k"] = Workload("qwen3b-32k", N=32768, Hq=16, Hkv=2, d=128, kv=1024, ks=2048,
                               seqs=[SeqSpec(seed=2, n_out=64, n_slash=16)])
    W["qwen3b-128k"] = Workload("qwen3b-128k", N=131072, Hq=16, Hkv=2, d=128, kv=1024, ks=2048,
                                seqs=[SeqSpec(seed=3, n_out=256, n_slash=32)])
    W["qwen3b-512k-striped8"] = Workload("qwen3b-512k-striped8", N=524288, Hq=16, Hkv=2, d=128, kv=1024,
                                         ks=2048, seqs=[SeqSpec(seed=4, n_out=256, n_slash=32)], world=8)
    W["batch4-64k"] = Workload("batch4-64k", N=65536, Hq=16, Hkv=2, d=128, kv=1024, ks=2048,
                               seqs=[SeqSpec(seed=10, n_out=0, band=16), SeqSpec(seed=11, n_out=16, band=64),
                                     SeqSpec(seed=12, n_out=128, band=256), SeqSpec(seed=13, n_out=512, band=1024)])
    W["dense-64k"] = Workload("dense-64k", N=65536, Hq=16, Hkv=2, d=128, kv=1024, ks=65536,
                              seqs=[SeqSpec(seed=14, n_out=0)])
    return W


def _chunks(N: int):
    """Fixed token chunking (depends on N only, so results do not depend on
    the number of worker threads)."""
    n = max(1, min(64, N // 1024))
    b = np.linspace(0, N, n + 1).astype(np.int64)
    return [(int(b[i]), int(b[i + 1])) for i in range(n)]


def _pool():
    import concurrent.futures as cf

    return cf.ThreadPoolExecutor(max_workers=max(1, min(32, os.cpu_count() or 1)))


def make_sequence(N: int, Hq: int, Hkv: int, d: int, spec: SeqSpec, with_dout: bool = True):
    """One sequence: dict of bf16 bit arrays q, k, v, dout ([N, H, d] uint16)
    plus the planted columns / offsets for reference.

    Random streams: the seed's SeedSequence spawns one stream for the plant
    choices and one per fixed token chunk (its K, V, Q, dO draws, in that
    order)."""
    ss = np.random.SeedSequence(spec.seed)
    main_ss, chunk_ss = ss.spawn(2)
    chunks = _chunks(N)
    gens = [np.random.Generator(np.random.PCG64(c)) for c in chunk_ss.spawn(len(chunks))]
    rng = np.random.Generator(np.random.PCG64(main_ss))
    cos, sin = rope_tables(N, d)
    k = np.empty((N, Hkv, d), np.float32)
    v16 = np.empty((N, Hkv, d), np.uint16)
    q16 = np.empty((N, Hq, d), np.uint16)
    do16 = np.empty((N, Hq, d), np.uint16) if with_dout else None

    def kv_part(i):
        a, b = chunks[i]
        g = gens[i]
        kk = g.standard_normal((b - a, Hkv, d), dtype=np.float32)
        k[a:b] = apply_rope(kk, cos[a:b], sin[a:b])
        v16[a:b] = bf16_round(g.standard_normal((b - a, Hkv, d), dtype=np.float32))

    with _pool() as ex:
        list(ex.map(kv_part, range(len(chunks))))
    cols = np.zeros((Hkv, spec.n_out), np.int64)
    for hk in range(Hkv):
        if spec.n_out:
            cols[hk] = np.sort(rng.choice(N, size=spec.n_out, replace=False))
            k[cols[hk], hk, :] *= OUTLIER_SCALE
    if spec.band:
        offs = np.arange(1, min(spec.band, N - 1) + 1, dtype=np.int64)
    elif spec.n_slash:
        hi = max(2, N // 8)
        offs = np.sort(rng.choice(np.arange(1, hi), size=min(spec.n_slash, hi - 1), replace=False))
    else:
        offs = np.zeros(0, np.int64)
    g_rep = Hq // Hkv
    c = np.float32(spec.gamma / math.sqrt(offs.size)) if offs.size else np.float32(0)

    def plant(a, b):
        """c * sum over planted o of k[n - o] for n in [a, b), [b - a, Hkv, d]."""
        if spec.band:
            w = offs.size
            lo = max(0, a - w)
            pre = np.zeros((b - lo + 1, Hkv, d), np.float64)
            np.cumsum(k[lo:b], axis=0, dtype=np.float64, out=pre[1:])
            n = np.arange(a, b)
            add = (pre[n - lo] - pre[np.maximum(n - w, 0) - lo]).astype(np.float32)
        else:
            add = np.zeros((b - a, Hkv, d), np.float32)
            for o in offs:
                s0 = max(a, int(o))
                if s0 < b:
                    add[s0 - a:] += k[s0 - o:b - o]
        add *= c
        return add

    def q_part(i):
        a, b = chunks[i]
        g = gens[i]
        qq = g.standard_normal((b - a, Hq, d), dtype=np.float32)
        apply_rope(qq, cos[a:b], sin[a:b])
        if offs.size:
            qq += np.repeat(plant(a, b), g_rep, axis=1)
        q16[a:b] = bf16_round(qq)
        if with_dout:
            do16[a:b] = bf16_round(g.standard_normal((b - a, Hq, d), dtype=np.float32))

    with _pool() as ex:
        list(ex.map(q_part, range(len(chunks))))
    out = {"q": q16, "k": bf16_round(k), "v": v16, "planted_cols": cols, "planted_offsets": offs}
    if with_dout:
        out["dout"] = do16
    return out


def make_batch(w: Workload, with_dout: bool = True, seqs: Optional[Sequence[int]] = None):
    """All sequences of a workload stacked to [B, N, H, d] bf16 bit arrays."""
    idx = list(range(w.B)) if seqs is None else list(seqs)
    parts = [make_sequence(w.N, w.Hq, w.Hkv, w.d, w.seqs[i], with_dout) for i in idx]
    out = {key: np.stack([p[key] for p in parts]) for key in ("q", "k", "v") + (("dout",) if with_dout else ())}
    out["planted_cols"] = [p["planted_cols"] for p in parts]
    out["planted_offsets"] = [p["planted_offsets"] for p in parts]
    return out


def small_workload(N: int, Hq: int, Hkv: int, d: int, kv: int, ks: int, seed: int, n_out: int = 0,
                   n_slash: int = 0, band: int = 0, B: int = 1, last_q: int = 64, world: int = 1) -> Workload:
    """An ad-hoc workload for tests."""
    return Workload(f"N{N}-H{Hq}x{Hkv}-d{d}", N=N, Hq=Hq, Hkv=Hkv, d=d, kv=kv, ks=ks,
                    seqs=[SeqSpec(seed=seed + i, n_out=n_out, n_slash=n_slash, band=band) for i in range(B)],
                    last_q=last_q, world=world)


def score_lists(B: int, H: int, N: int, seed: int, total: float = 64.0):
    """Seeded synthetic vertical / slash score lists, float32 [B, H, N] each,
    shaped like an observation window's column and diagonal sums (each list
    sums to about ``total``, the window length): vertical scores are a
    heavy (Pareto) tail with a sink at column 0 and a few outlier columns;
    slash scores decay with the offset (a local band) plus a few planted
    diagonals and a tail.  A draw of inputs for the selection step, no part
    of the method."""
    rng = np.random.default_rng(seed)
    v = rng.pareto(1.2, (B, H, N)) + 1e-3
    v[:, :, 0] += 0.2 * N
    for b in range(B):
        for h in range(H):
            v[b, h, rng.choice(N, 8, replace=False)] += rng.uniform(0.01, 0.05) * N
    o = np.arange(N, dtype=np.float64)
    s = rng.pareto(1.5, (B, H, N)) * 0.05 + 50.0 / (1.0 + o / 16.0) ** 2
    for b in range(B):
        for h in range(H):
            s[b, h, rng.choice(N, 6, replace=False)] += rng.uniform(0.5, 3.0) * s[b, h].mean() * 20
    v *= total / v.sum(-1, keepdims=True)
    s *= total / s.sum(-1, keepdims=True)
    return v.astype(np.float32), s.astype(np.float32)
