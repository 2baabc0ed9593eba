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
    kv / ks.  All tensors are BSHD bf16 on the device.
    """

    def __init__(self, B: int, N: int, Hq: int, Hkv: int, d: int, kv: int, ks: int,
                 device="cuda", last_q: int = 64, scale: Optional[float] = None):
        self.B, self.N, self.Hq, self.Hkv, self.d, self.kv, self.ks = B, N, Hq, Hkv, d, kv, ks
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
        self._qkv = None

    def forward(self, q, k, v, stream=None):
        B_.vs_estimate(q, k, self.kv, self.ks, self.scale, self.last_q, self.v_idx, self.s_idx, self.v_score,
                       self.s_score, self.ws_est, stream)
        B_.vs_build_block_index(q, k, self.v_idx, self.s_idx, None, self.arena, stream)
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
