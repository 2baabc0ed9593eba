"""The whole hot path on preallocated device buffers, and FLOP accounting.

``VSAttention`` runs Algorithm 1 end to end for one layer's attention:
estimate (vertical / slash selection) -> sparse index -> sparse forward ->
sparse backward, each a call into libvs.so.  Buffers are allocated once with
torch so that repeated steps launch kernels only.
"""
from __future__ import annotations

import math
from typing import Optional

import numpy as np
import torch

from . import _binding as B_


def flop_counts(counts: np.ndarray, d: int) -> dict:
    """FLOPs of one forward + backward from the arena's work counts
    ([B, Hq, 4]: query-major slash tiles, query-major bar chunks, key-major
    slash units, key-major bar units; every unit is 128 x 64 entries).

    executed: the query-major cover credited at 4 * area * d (forward) and
      10 * area * d (backward, five GEMMs), the fixed formula of the
      throughput metric;
    issued: the tensor-core work the kernels actually run (forward 2 GEMMs
      and backward dQ 3 GEMMs on the query-major cover, dK / dV 4 GEMMs on the
      key-major cover).
    """
    c = counts.reshape(-1, 4).sum(0).astype(np.float64)
    area_q = (c[0] + c[1]) * 128 * 64
    area_k = (c[2] + c[3]) * 128 * 64
    return {
        "units": c.tolist(),
        "fwd_executed": 4.0 * area_q * d,
        "bwd_executed": 10.0 * area_q * d,
        "fwd_issued": 4.0 * area_q * d,
        "bwd_issued": 6.0 * area_q * d + 8.0 * area_k * d,
    }


def dense_causal_flops(B: int, N: int, Hq: int, d: int) -> dict:
    """Dense causal attention at the same shape: 4 d per mask entry forward,
    10 d backward, over N (N + 1) / 2 entries per head."""
    area = B * Hq * N * (N + 1) / 2.0
    return {"fwd": 4.0 * area * d, "bwd": 10.0 * area * d}


class VSAttention:
    """Vertical-Slash sparse attention for one layer (one process, one GPU).

    forward(q, k, v) -> (o, lse) and backward(dO) -> (dq, dk, dv) run the
    estimator, the index build and the sparse kernels with fixed budgets
    kv / ks, or, when ``pv`` and ``ps`` are given, with per-head top-p
    budgets (Algorithm 1) of at most kv / ks entries (``budgets`` then holds
    the [B, Hq] budgets of the last forward).  ``block_cover`` selects the
    block-cover reading of the slashes (whole 64 x 64 blocks, see
    vs_build_block_index_ex); ``shared`` one selection per KV group
    (vs_estimate_group); ``packed`` (with ``shared``) packs the group's query
    heads into the query-major tiles (VS_INDEX_PACK_GQA: 128 / g tokens of the
    g heads per tile).  All tensors are BSHD bf16 on the device.
    """

    def __init__(self, B: int, N: int, Hq: int, Hkv: int, d: int, kv: int, ks: int,
                 device="cuda", last_q: int = 64, scale: Optional[float] = None,
                 pv: Optional[float] = None, ps: Optional[float] = None, block_cover: bool = False,
                 shared: bool = False, packed: bool = False):
        self.B, self.N, self.Hq, self.Hkv, self.d, self.kv, self.ks = B, N, Hq, Hkv, d, kv, ks
        if (pv is None) != (ps is None):
            raise ValueError("top-p mode needs both pv and ps")
        self.pv, self.ps = pv, ps
        self.block_cover = block_cover
        self.shared = shared
        if packed and not shared:
            raise ValueError("head packing needs one selection per KV group (shared=True)")
        self.packed = packed
        self.last_q = last_q
        self.scale = 1.0 / math.sqrt(d) if scale is None else scale
        dev = torch.device(device)
        q0 = torch.empty(B, N, Hq, d, dtype=torch.bfloat16, device=dev)
        k0 = torch.empty(B, N, Hkv, d, dtype=torch.bfloat16, device=dev)
        sh = B_.make_shape(q0, k0)
        L = B_.lib()
        import ctypes
        self.v_idx = torch.empty(B, Hq, kv, dtype=torch.int32, device=dev)
        self.s_idx = torch.empty(B, Hq, ks, dtype=torch.int32, device=dev)
        self.v_score = torch.empty(B, Hq, N, dtype=torch.float32, device=dev)
        self.s_score = torch.empty(B, Hq, N, dtype=torch.float32, device=dev)
        self.ws_est = torch.zeros(max(256, L.vs_estimate_workspace(ctypes.byref(sh), last_q)), dtype=torch.uint8,
                                  device=dev)
        self.arena = torch.empty(L.vs_block_index_bytes(ctypes.byref(sh), kv, ks, None), dtype=torch.uint8,
                                 device=dev)
        self.o = torch.empty_like(q0)
        self.lse = torch.empty(B, Hq, N, dtype=torch.float32, device=dev)
        self.ws_fwd = torch.zeros(256, dtype=torch.uint8, device=dev)
        self.dq = torch.empty_like(q0)
        self.dk = torch.empty_like(k0)
        self.dv = torch.empty_like(k0)
        self.ws_bwd = torch.zeros(L.vs_attn_bwd_workspace(ctypes.byref(sh), kv), dtype=torch.uint8, device=dev)
        self.budgets = (torch.zeros(B, Hq, dtype=torch.int32, device=dev),
                        torch.zeros(B, Hq, dtype=torch.int32, device=dev)) if pv is not None else None
        self._qkv = None

    def forward(self, q, k, v, stream=None, selection=None):
        """Estimate, index, sparse forward.  ``selection`` = (v_idx, s_idx)
        int32 device tensors [B, Hq, kv] / [B, Hq, ks] (sorted ascending,
        optionally ending in -1) replaces the estimator, e.g. to reuse one
        layer's selection."""
        if selection is None and self.pv is not None:
            B_.vs_estimate_topp(q, k, self.pv, self.ps, self.kv, self.ks, self.scale, self.last_q, self.v_idx,
                                self.s_idx, self.budgets[0], self.budgets[1], self.v_score, self.s_score, self.ws_est,
                                stream)
        elif selection is None:
            B_.vs_estimate(q, k, self.kv, self.ks, self.scale, self.last_q, self.v_idx, self.s_idx, self.v_score,
                           self.s_score, self.ws_est, stream, self.shared)
        else:
            self.v_idx.copy_(selection[0])
            self.s_idx.copy_(selection[1])
        B_.vs_build_block_index(q, k, self.v_idx, self.s_idx, None, self.arena, stream, self.block_cover,
                                self.packed)
        B_.vs_attn_fwd(q, k, v, self.arena, self.scale, self.o, self.lse, None, self.ws_fwd, stream)
        self._qkv = (q, k, v)
        return self.o, self.lse

    def backward(self, dO, stream=None):
        q, k, v = self._qkv
        B_.vs_attn_bwd(q, k, v, self.o, self.lse, dO, self.arena, self.kv, self.scale, self.dq, self.dk, self.dv,
                       None, self.ws_bwd, stream)
        return self.dq, self.dk, self.dv

    def check(self):
        """Raises if any kernel recorded a device error."""
        for buf in (self.ws_est, self.arena, self.ws_fwd, self.ws_bwd):
            code = B_.vs_check_status(buf)
            if code:
                raise B_.VSError(code, "device status")

    def counts(self) -> np.ndarray:
        return B_.vs_index_counts(self.arena)


def ring_source(rank: int, s: int, world: int, inner: int = 0) -> int:
    """The KV shard that worker ``rank`` attends to at ring step ``s`` of a
    ``world``-worker ring: the flat ring receives from the previous worker,
    (rank - s) mod world; with ``inner`` cards per node (Hierarchical
    Balanced Sparse Ring Attention, Algorithm 2) step s = i * inner + j is
    inner step j of outer step i, and reads the shard of worker
    ((n - i) mod nodes) * inner + (c - j) mod inner for rank = n * inner + c."""
    if not inner:
        return (rank - s) % world
    nodes = world // inner
    n, c = divmod(rank, inner)
    i, j = divmod(s, inner)
    return ((n - i) % nodes) * inner + (c - j) % inner


class StripedWorker:
    """One worker's side of the striped ring on one GPU (MTraining, section
    4.2 (ii) and Algorithm 2): the sequence of N_global tokens is cut into
    ``stripe``-token blocks dealt round-robin to ``world`` workers; worker
    ``rank`` keeps its query shard and, at ring step s, attends to the KV
    shard of source ``(rank - s) mod world`` with the index built on global
    positions, merging each step's (O, LSE) into the running result.

    The KV shards of every source sit in this GPU's memory (the ring's
    point-to-point rotation is not run); each step's forward and backward are
    timed with CUDA events so per-step load and its imbalance can be read
    off.  Buffers are preallocated; the selection is made once, on the
    global sequence, by ``select``.

    ``inner`` > 0 selects the hierarchical order of Hierarchical Balanced
    Sparse Ring Attention (section 4.2 (i)-(ii), Algorithm 2): workers are
    grouped in nodes of ``inner`` cards (worker r = node n * inner + card c);
    at outer step i the node holds the KV buffer of node n - i, and its inner
    ring passes slices among the node's cards, so inner step j of outer step
    i attends to the shard of worker ((n - i) mod nodes) * inner +
    ((c - j) mod inner).  Only the order of the steps changes; the merged
    result is the same up to the summation order.
    """

    def __init__(self, B: int, N_global: int, Hq: int, Hkv: int, d: int, kv: int, ks: int, world: int,
                 rank: int = 0, stripe: int = 64, device="cuda", last_q: int = 64, scale: Optional[float] = None,
                 inner: int = 0, block_cover: bool = False):
        if N_global % (world * stripe):
            raise ValueError("N_global must be a multiple of world * stripe")
        self.block_cover = block_cover
        if inner and world % inner:
            raise ValueError("world must be a multiple of the node size")
        self.inner = inner
        self.B, self.N, self.Hq, self.Hkv, self.d, self.kv, self.ks = B, N_global, Hq, Hkv, d, kv, ks
        self.world, self.rank, self.stripe, self.last_q = world, rank, stripe, last_q
        self.scale = 1.0 / math.sqrt(d) if scale is None else scale
        dev = torch.device(device)
        Nl = N_global // world
        self.Nl = Nl
        L = B_.lib()
        import ctypes
        qg = torch.empty(B, N_global, Hq, d, dtype=torch.bfloat16, device="meta")
        kg = torch.empty(B, N_global, Hkv, d, dtype=torch.bfloat16, device="meta")
        shg = B_.make_shape(qg, kg)
        self.v_idx = torch.empty(B, Hq, kv, dtype=torch.int32, device=dev)
        self.s_idx = torch.empty(B, Hq, ks, dtype=torch.int32, device=dev)
        self.v_score = torch.empty(B, Hq, N_global, dtype=torch.float32, device=dev)
        self.s_score = torch.empty(B, Hq, N_global, dtype=torch.float32, device=dev)
        self.ws_est = torch.zeros(max(256, L.vs_estimate_workspace(ctypes.byref(shg), last_q)), dtype=torch.uint8,
                                  device=dev)
        ql = torch.empty(B, Nl, Hq, d, dtype=torch.bfloat16, device=dev)
        kl = torch.empty(B, Nl, Hkv, d, dtype=torch.bfloat16, device=dev)
        shl = B_.make_shape(ql, kl)
        self.stripes = [B_.make_stripe(world, rank, self.source(s), N_global, stripe) for s in range(world)]
        self.arenas = [torch.empty(L.vs_block_index_bytes(ctypes.byref(shl), kv, ks, ctypes.byref(st)),
                                   dtype=torch.uint8, device=dev) for st in self.stripes]
        self.o = torch.empty_like(ql)
        self.lse = torch.empty(B, Hq, Nl, dtype=torch.float32, device=dev)
        self.o_acc = torch.empty(B, Nl, Hq, d, dtype=torch.float32, device=dev)
        self.ws_fwd = torch.zeros(256, dtype=torch.uint8, device=dev)
        self.dq = torch.empty_like(ql)
        self.dq_acc = torch.empty(B, Nl, Hq, d, dtype=torch.float32, device=dev)
        self.dk = torch.empty(world, B, Nl, Hkv, d, dtype=torch.bfloat16, device=dev)
        self.dv = torch.empty_like(self.dk)
        self.ws_bwd = torch.zeros(L.vs_attn_bwd_workspace(ctypes.byref(shl), kv), dtype=torch.uint8, device=dev)
        # per ring step: forward start / end, backward start / end
        self.events = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(world)]
        self._qkv = None

    def source(self, s: int) -> int:
        """The KV shard worker ``rank`` attends to at ring step s."""
        return ring_source(self.rank, s, self.world, self.inner)

    def select(self, q_global, k_global, stream=None):
        """Vertical / slash selection on the global sequence (Algorithm 1's
        estimate over the last ``last_q`` global queries)."""
        B_.vs_estimate(q_global, k_global, self.kv, self.ks, self.scale, self.last_q, self.v_idx, self.s_idx,
                       self.v_score, self.s_score, self.ws_est, stream)
        return self.v_idx, self.s_idx

    def build_index(self, q_shard, k_shards, stream=None):
        """One index per ring step, on global positions through the stripe map."""
        for s in range(self.world):
            B_.vs_build_block_index(q_shard, k_shards[self.source(s)], self.v_idx, self.s_idx, self.stripes[s],
                                    self.arenas[s], stream, self.block_cover)

    def forward(self, q_shard, k_shards, v_shards, stream=None):
        """World ring steps; each merges its partial (O, LSE) into the running
        result (merge_out_and_lse).  Returns (o bf16, lse fp32)."""
        self.lse.fill_(-math.inf)
        self.o_acc.zero_()
        for s in range(self.world):
            src = self.source(s)
            self.events[s][0].record(stream)
            B_.vs_attn_fwd(q_shard, k_shards[src], v_shards[src], self.arenas[s], self.scale, self.o, self.lse,
                           self.o_acc, self.ws_fwd, stream)
            self.events[s][1].record(stream)
        self._qkv = (q_shard, k_shards, v_shards)
        return self.o, self.lse

    def backward(self, dO_shard, stream=None):
        """dQ accumulated over the ring steps; dK / dV of each source shard
        from this worker's queries (what goes back to the shard's owner)."""
        q, ks_, vs_ = self._qkv
        self.dq_acc.zero_()
        for s in range(self.world):
            src = self.source(s)
            self.events[s][2].record(stream)
            B_.vs_attn_bwd(q, ks_[src], vs_[src], self.o, self.lse, dO_shard, self.arenas[s], self.kv, self.scale,
                           self.dq, self.dk[src], self.dv[src], self.dq_acc, self.ws_bwd, stream)
            self.events[s][3].record(stream)
        return self.dq, self.dk, self.dv

    def step_times(self):
        """Per ring step (forward ms, backward ms) of the last forward /
        backward pair (after a synchronize)."""
        return [(e[0].elapsed_time(e[1]), e[2].elapsed_time(e[3])) for e in self.events]

    def check(self):
        """Raises if any kernel recorded a device error."""
        for buf in [self.ws_est, self.ws_fwd, self.ws_bwd] + self.arenas:
            code = B_.vs_check_status(buf)
            if code:
                raise B_.VSError(code, "device status")

    def counts(self) -> np.ndarray:
        """Work units per ring step: [world, B, Hq, 4]."""
        return np.stack([B_.vs_index_counts(a) for a in self.arenas])


class ZigZagWorker:
    """One worker's side of a ZigZag ring on one GPU (the layout MTraining
    contrasts with striping, section 2 and Figure 1): the sequence of N_global
    tokens is cut into 2 * world chunks of C = N_global / (2 world) tokens and
    worker ``rank`` holds chunks rank and 2 world - 1 - rank (its shard is the
    two chunks in that order, see ring_permute).  At ring step s it attends to
    the KV shard of source (rank - s) mod world.

    A step is made of chunk pairs (a query chunk of this worker, a key chunk
    of the source) with the query chunk not before the key chunk on the
    sequence (a pair in the other order has no causal entry).  Each pair is a
    windowed problem (make_window) with its own index built on global
    positions: the forward merges the pair's (O, LSE) into its query chunk's
    running result, the backward accumulates dQ per query chunk and dK / dV
    per key chunk of the source (vs_attn_bwd_ex), with the merged LSE.  Each
    step's forward and backward are timed with CUDA events.  The KV shards of
    every source sit in this GPU's memory; the selection is made once, on the
    global sequence, by ``select``.
    """

    def __init__(self, B: int, N_global: int, Hq: int, Hkv: int, d: int, kv: int, ks: int, world: int,
                 rank: int = 0, device="cuda", last_q: int = 64, scale: Optional[float] = None):
        if N_global % (2 * world * 64):
            raise ValueError("N_global must be a multiple of 128 * world")
        self.B, self.N, self.Hq, self.Hkv, self.d, self.kv, self.ks = B, N_global, Hq, Hkv, d, kv, ks
        self.world, self.rank, self.last_q = world, rank, last_q
        self.scale = 1.0 / math.sqrt(d) if scale is None else scale
        dev = torch.device(device)
        C = N_global // (2 * world)
        self.C = C
        L = B_.lib()
        import ctypes
        qg = torch.empty(B, N_global, Hq, d, dtype=torch.bfloat16, device="meta")
        kg = torch.empty(B, N_global, Hkv, d, dtype=torch.bfloat16, device="meta")
        shg = B_.make_shape(qg, kg)
        self.v_idx = torch.empty(B, Hq, kv, dtype=torch.int32, device=dev)
        self.s_idx = torch.empty(B, Hq, ks, dtype=torch.int32, device=dev)
        self.v_score = torch.empty(B, Hq, N_global, dtype=torch.float32, device=dev)
        self.s_score = torch.empty(B, Hq, N_global, dtype=torch.float32, device=dev)
        self.ws_est = torch.zeros(max(256, L.vs_estimate_workspace(ctypes.byref(shg), last_q)), dtype=torch.uint8,
                                  device=dev)
        qc = torch.empty(B, C, Hq, d, dtype=torch.bfloat16, device=dev)
        kc = torch.empty(B, C, Hkv, d, dtype=torch.bfloat16, device=dev)
        shc = B_.make_shape(qc, kc)
        # per ring step: the chunk pairs (query chunk i, key chunk j, window)
        self.pairs = []
        for s in range(world):
            src = self.source(s)
            qch, kch = self.chunks(rank), self.chunks(src)
            ps = []
            for i in range(2):
                for j in range(2):
                    if qch[i] >= kch[j]:
                        ps.append((i, j, B_.make_window(qch[i] * C, kch[j] * C, N_global)))
            self.pairs.append(ps)
        self.arenas = [[torch.empty(L.vs_block_index_bytes(ctypes.byref(shc), kv, ks, ctypes.byref(st)),
                                    dtype=torch.uint8, device=dev) for (_, _, st) in ps] for ps in self.pairs]
        self.o = torch.empty(B, 2 * C, Hq, d, dtype=torch.bfloat16, device=dev)
        self.lse = [torch.empty(B, Hq, C, dtype=torch.float32, device=dev) for _ in range(2)]  # per query chunk
        # fp32 accumulators are contiguous [B][C][Hq][d] per query chunk
        self.o_acc = [torch.empty(B, C, Hq, d, dtype=torch.float32, device=dev) for _ in range(2)]
        self.ws_fwd = torch.zeros(256, dtype=torch.uint8, device=dev)
        self.dq = torch.empty_like(self.o)
        self.dq_acc = [torch.empty(B, C, Hq, d, dtype=torch.float32, device=dev) for _ in range(2)]
        self.dk = torch.empty(world, B, 2 * C, Hkv, d, dtype=torch.bfloat16, device=dev)
        self.dv = torch.empty_like(self.dk)
        self.dkv_acc = [torch.empty(2, B, C, Hkv, d, dtype=torch.float32, device=dev) for _ in range(2)]
        self.ws_bwd = torch.zeros(L.vs_attn_bwd_workspace(ctypes.byref(shc), kv), dtype=torch.uint8, device=dev)
        self.events = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(world)]
        self._qkv = None

    def chunks(self, r: int):
        """The two chunks (of C tokens, in sequence order) worker r holds."""
        return (r, 2 * self.world - 1 - r)

    def source(self, s: int) -> int:
        return ring_source(self.rank, s, self.world)

    def _rows(self, t, i):
        return t[:, i * self.C:(i + 1) * self.C]

    def select(self, q_global, k_global, stream=None):
        B_.vs_estimate(q_global, k_global, self.kv, self.ks, self.scale, self.last_q, self.v_idx, self.s_idx,
                       self.v_score, self.s_score, self.ws_est, stream)
        return self.v_idx, self.s_idx

    def build_index(self, q_shard, k_shards, stream=None):
        """One index per chunk pair of every ring step, on global positions."""
        for s in range(self.world):
            src = self.source(s)
            for (i, j, st), arena in zip(self.pairs[s], self.arenas[s]):
                B_.vs_build_block_index(self._rows(q_shard, i), self._rows(k_shards[src], j), self.v_idx, self.s_idx,
                                        st, arena, stream)

    def forward(self, q_shard, k_shards, v_shards, stream=None):
        for l, a in zip(self.lse, self.o_acc):
            l.fill_(-math.inf)
            a.zero_()
        for s in range(self.world):
            src = self.source(s)
            self.events[s][0].record(stream)
            for (i, j, _), arena in zip(self.pairs[s], self.arenas[s]):
                B_.vs_attn_fwd(self._rows(q_shard, i), self._rows(k_shards[src], j), self._rows(v_shards[src], j),
                               arena, self.scale, self._rows(self.o, i), self.lse[i], self.o_acc[i],
                               self.ws_fwd, stream)
            self.events[s][1].record(stream)
        self._qkv = (q_shard, k_shards, v_shards)
        return self.o, self.lse

    def backward(self, dO_shard, stream=None):
        q, ks_, vs_ = self._qkv
        for a in self.dq_acc:
            a.zero_()
        for s in range(self.world):
            src = self.source(s)
            self.events[s][2].record(stream)
            for a in self.dkv_acc:
                a.zero_()
            self.dk[src].zero_()  # key chunks with no causal pair keep zero gradients
            self.dv[src].zero_()
            for (i, j, _), arena in zip(self.pairs[s], self.arenas[s]):
                B_.vs_attn_bwd(self._rows(q, i), self._rows(ks_[src], j), self._rows(vs_[src], j),
                               self._rows(self.o, i), self.lse[i], self._rows(dO_shard, i), arena, self.kv,
                               self.scale, self._rows(self.dq, i), self._rows(self.dk[src], j),
                               self._rows(self.dv[src], j), self.dq_acc[i], self.ws_bwd, stream,
                               dkv_acc=self.dkv_acc[j])
            self.events[s][3].record(stream)
        return self.dq, self.dk, self.dv

    def step_times(self):
        return [(e[0].elapsed_time(e[1]), e[2].elapsed_time(e[3])) for e in self.events]

    def check(self):
        for buf in [self.ws_est, self.ws_fwd, self.ws_bwd] + [a for ar in self.arenas for a in ar]:
            code = B_.vs_check_status(buf)
            if code:
                raise B_.VSError(code, "device status")

    def counts(self) -> np.ndarray:
        """Work units per ring step, summed over the step's chunk pairs: [world, B, Hq, 4]."""
        return np.stack([sum((B_.vs_index_counts(a) for a in ar), np.zeros((self.B, self.Hq, 4), np.int64))
                         for ar in self.arenas])
