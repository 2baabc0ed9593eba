"""CPU oracle for MTraining's dynamic Vertical-Slash sparse attention.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's ``cpu_baseline`` / ``--impl reference`` legs may import this
package.  The product path (the CUDA library and its binding) never does.

Plain, slow and fp64: the arithmetic lives in ``vs_oracle.c`` (loaded with
ctypes) plus a few numpy helpers here that follow the pages' definitions
directly:

* ``estimate`` / ``topk`` / ``select`` / ``select_group`` / ``topp_budget`` /
  ``select_topp`` --
  Algorithm 1 of *MTraining:
  Distributed Dynamic Sparse Attention for Efficient Ultra-Long Context
  Training*: the last-``last_q`` observation window, ``sum_v`` / ``sum_s`` and
  ``argtopk`` (fixed budgets; ties go to the lower index).
* ``rows`` / ``keys`` / ``attention`` -- masked softmax attention on the VS
  mask and its gradients by Eq. 1 (dS) and Eq. 2 (dV, dQ, dK).
* ``merge`` -- ``merge_out_and_lse`` of Algorithm 2.
* ``stripe_positions`` / ``striped_permute`` -- 64-token block-level
  striping (section 4.2 (ii)).
* ``ring_owners`` / ``ring_positions`` / ``ring_permute`` / ``ring_work`` --
  the striped and ZigZag ring layouts and the mask entries per (query
  worker, key worker) under them (sections 2, 3.3, 4.2).

Inputs are converted to float64 (bf16 values widen exactly); all arithmetic is fp64.
"""
from __future__ import annotations

import ctypes
import math
import os

import numpy as np

from . import build as _build

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        L.ora_topk.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p]
        L.ora_estimate.argtypes = [ctypes.c_int] * 5 + [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                                                          ctypes.c_double, ctypes.c_void_p, ctypes.c_void_p]
        L.ora_rows.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                               ctypes.c_void_p]
        L.ora_keys.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
        L.ora_mask_count.argtypes = [ctypes.c_void_p]
        L.ora_mask_count.restype = ctypes.c_int64
        L.ora_mask_dense.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
        L.ora_stripe_positions.argtypes = [ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                           ctypes.c_void_p]
        L.ora_merge.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_double, ctypes.c_void_p, ctypes.c_double,
                                ctypes.c_void_p, ctypes.c_void_p]
        L.ora_num_threads.restype = ctypes.c_int
        L.ora_row_stats.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                                    ctypes.c_void_p]
        _lib = L
    return _lib


def num_threads() -> int:
    return int(lib().ora_num_threads())


def _p(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


# ------------------------------------------------------------------ selection
def estimate(q: np.ndarray, k: np.ndarray, last_q: int, scale: float):
    """sum_v and sum_s of the last-``last_q`` causal softmax (Algorithm 1).

    q: [B, N, Hq, d], k: [B, N, Hkv, d].
    Returns (v, s), each float64 [B, Hq, N]: v[m] = sum_i A_hat[i, m],
    s[o] = sum_i A_hat[i, n_i - o] with n_i = N - last_q + i.
    """
    q, k = _f64(q), _f64(k)
    B, N, Hq, d = q.shape
    Hkv = k.shape[2]
    v = np.zeros((B, Hq, N), np.float64)
    s = np.zeros((B, Hq, N), np.float64)
    lib().ora_estimate(B, N, Hq, Hkv, d, _p(q), _p(k), int(last_q), float(scale), _p(v), _p(s))
    return v, s


def topk(score: np.ndarray, k: int) -> np.ndarray:
    """argtopk under the total order (score descending, index ascending),
    returned sorted ascending.  Float32 scores widen to fp64 exactly, so the
    same routine replays a selection made on float32 scores."""
    score = np.ascontiguousarray(score, dtype=np.float64)
    out = np.zeros(int(k), np.int32)
    lib().ora_topk(int(score.shape[0]), _p(score), int(k), _p(out))
    return out


def select(v: np.ndarray, s: np.ndarray, kv: int, ks: int):
    """Per (b, h): iv = argtopk(v, kv), is = argtopk(s, ks)."""
    B, H, N = v.shape
    iv = np.zeros((B, H, kv), np.int32)
    is_ = np.zeros((B, H, ks), np.int32)
    for b in range(B):
        for h in range(H):
            iv[b, h] = topk(v[b, h], kv)
            is_[b, h] = topk(s[b, h], ks)
    return iv, is_


def select_group(v: np.ndarray, s: np.ndarray, kv: int, ks: int, g: int, dtype=np.float64):
    """Per-KV-group shared selection (a variant of Algorithm 1's per-head
    selection: the g query heads that share a KV head use one index): the
    group's scores are the sum of its heads' scores, added in head order in
    `dtype` (the precision in which the sum decides the selection), and every
    head of the group gets iv = argtopk(sum v, kv), is = argtopk(sum s, ks)."""
    B, H, N = v.shape
    G = H // g
    iv = np.zeros((B, H, kv), np.int32)
    is_ = np.zeros((B, H, ks), np.int32)
    vv = np.asarray(v, dtype).reshape(B, G, g, N)
    ss = np.asarray(s, dtype).reshape(B, G, g, N)
    for b in range(B):
        for hk in range(G):
            sv, sl = vv[b, hk, 0].copy(), ss[b, hk, 0].copy()
            for j in range(1, g):
                sv = (sv + vv[b, hk, j]).astype(dtype)
                sl = (sl + ss[b, hk, j]).astype(dtype)
            iv[b, hk * g:(hk + 1) * g] = topk(sv, kv)
            is_[b, hk * g:(hk + 1) * g] = topk(sl, ks)
    return iv, is_


# Top-p budgets decide an integer (a count) from sums of scores, so both this
# oracle and the kernels take the decision in one exact precision: a score x
# counts floor(x * 2^40) mass units, sums of units are exact integers, and the
# target is t = ceil(fl(p * T)) for the list total T (one IEEE double product).
MASS_UNIT_LOG2 = 40


def mass_units(score: np.ndarray) -> np.ndarray:
    """floor(x * 2^40) of each score as int64 (exact: scaling by a power of two)."""
    x = np.asarray(score, np.float64)
    return np.floor(x * float(2 ** MASS_UNIT_LOG2)).astype(np.int64)


def topp_budget(units: np.ndarray, p: float) -> int:
    """``topp`` of Algorithm 1 on integer mass units: the smallest k in [0, n]
    whose k largest units sum to at least t = ceil(p * T), T = sum of all
    units; n when no k reaches t.  (Which of several equal units is counted
    does not change the sum, so ties need no rule here.)"""
    u = np.sort(np.asarray(units, np.int64))[::-1]
    n = u.size
    T = int(u.sum())
    t = math.ceil(float(p) * float(T))
    if t <= 0:
        return 0
    csum = np.cumsum(u)
    k = int(np.searchsorted(csum, t, side="left")) + 1
    return min(k, n)


def pool(units: np.ndarray, block: int = 64) -> np.ndarray:
    """``Pool`` of Algorithm 1: the sum of each run of `block` consecutive
    entries (the last run may be shorter)."""
    u = np.asarray(units, np.int64)
    nb = (u.size + block - 1) // block
    padded = np.zeros(nb * block, np.int64)
    padded[:u.size] = u
    return padded.reshape(nb, block).sum(1)


def select_topp(v: np.ndarray, s: np.ndarray, pv: float, ps: float, kv_max: int, ks_max: int, block: int = 64):
    """Budgets from top-p, then token-level selection (Algorithm 1):
    kv = min(topp(units(v), pv), kv_max); ks = min(block * topp(Pool(units(s),
    block), ps), ks_max, N); iv = argtopk(v, kv), is = argtopk(s, ks).  The
    slash budget pools the slash scores (the listing's ``Pool(sum_v ...)`` is
    read as ``Pool(sum_s ...)``: the budget it sets is spent on sum_s) in
    64-offset blocks, matching the kernel's 64 x 64 slash tiles.
    Returns (iv [B,H,kv_max], is [B,H,ks_max], kv [B,H], ks [B,H]); each list
    holds its budget's indices ascending, then -1."""
    B, H, N = v.shape
    iv = np.full((B, H, kv_max), -1, np.int32)
    is_ = np.full((B, H, ks_max), -1, np.int32)
    kv = np.zeros((B, H), np.int32)
    ks = np.zeros((B, H), np.int32)
    for b in range(B):
        for h in range(H):
            kv[b, h] = min(topp_budget(mass_units(v[b, h]), pv), kv_max)
            ks[b, h] = min(block * topp_budget(pool(mass_units(s[b, h]), block), ps), ks_max, N)
            iv[b, h, :kv[b, h]] = topk(v[b, h], int(kv[b, h]))
            is_[b, h, :ks[b, h]] = topk(s[b, h], int(ks[b, h]))
    return iv, is_, kv, ks


# ------------------------------------------------------------------ attention
class _Problem(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("Nq", ctypes.c_int), ("Nk", ctypes.c_int), ("Hq", ctypes.c_int),
                ("Hkv", ctypes.c_int), ("d", ctypes.c_int), ("n_global", ctypes.c_int64),
                ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("dout", ctypes.c_void_p),
                ("qpos", ctypes.c_void_p), ("kpos", ctypes.c_void_p), ("iv", ctypes.c_void_p),
                ("is_", ctypes.c_void_p), ("kv", ctypes.c_int), ("ks", ctypes.c_int), ("scale", ctypes.c_double),
                ("block", ctypes.c_int)]


class Problem:
    """One VS attention problem.

    q [B, Nq, Hq, d], k/v [B, Nk, Hkv, d], dout [B, Nq, Hq, d] or None;
    iv [B, Hq, kv] and is_ [B, Hq, ks] index the global sequence of length
    ``n_global``; qpos / kpos give each local row's / key's global position
    (identity when None).  block=True selects the block-cover reading of the
    slashes (section 4.1 (ii): the slash budget works on 64 x 64 blocks): every
    causal entry of a 64 x 64 block (on global positions) that a selected
    slash passes through is in the mask, besides the selected columns.
    """

    def __init__(self, q, k, v, iv, is_, scale, dout=None, qpos=None, kpos=None, n_global=None, block=False):
        self.q, self.k, self.v = _f64(q), _f64(k), _f64(v)
        self.dout = None if dout is None else _f64(dout)
        B, Nq, Hq, d = self.q.shape
        Nk, Hkv = self.k.shape[1], self.k.shape[2]
        self.iv = np.ascontiguousarray(iv, dtype=np.int32)
        self.is_ = np.ascontiguousarray(is_, dtype=np.int32)
        self.qpos = np.arange(Nq, dtype=np.int64) if qpos is None else np.ascontiguousarray(qpos, np.int64)
        self.kpos = np.arange(Nk, dtype=np.int64) if kpos is None else np.ascontiguousarray(kpos, np.int64)
        self.n_global = int(n_global if n_global is not None else max(Nq, Nk))
        assert self.iv.shape[:2] == (B, Hq) and self.is_.shape[:2] == (B, Hq)
        assert Hq % Hkv == 0
        self.shape = (B, Nq, Nk, Hq, Hkv, d)
        self.scale = float(scale)
        self._c = _Problem(B, Nq, Nk, Hq, Hkv, d, self.n_global, self.q.ctypes.data, self.k.ctypes.data,
                           self.v.ctypes.data, None if self.dout is None else self.dout.ctypes.data,
                           self.qpos.ctypes.data, self.kpos.ctypes.data, self.iv.ctypes.data, self.is_.ctypes.data,
                           self.iv.shape[2], self.is_.shape[2], self.scale, int(bool(block)))

    def ref(self):
        return ctypes.byref(self._c)


def rows(p: Problem, rows_bhn: np.ndarray):
    """Forward (O, LSE) and, when dout is set, dQ for the given (b, h, n) rows."""
    rows_bhn = np.ascontiguousarray(rows_bhn, dtype=np.int32).reshape(-1, 3)
    R, d = rows_bhn.shape[0], p.shape[5]
    o = np.zeros((R, d), np.float64)
    lse = np.zeros(R, np.float64)
    dq = np.zeros((R, d), np.float64) if p.dout is not None else None
    lib().ora_rows(p.ref(), R, _p(rows_bhn), _p(o), _p(lse), None if dq is None else _p(dq))
    return o, lse, dq


def row_stats(p: Problem, rows_bhn: np.ndarray):
    """LSE_n and D_n = sum_m dA_nm A_nm (Eq. 1's row sum) for (b, h, n) rows."""
    rows_bhn = np.ascontiguousarray(rows_bhn, dtype=np.int32).reshape(-1, 3)
    R = rows_bhn.shape[0]
    lse = np.zeros(R, np.float64)
    D = np.zeros(R, np.float64)
    lib().ora_row_stats(p.ref(), R, _p(rows_bhn), _p(lse), _p(D))
    return lse, D


def keys(p: Problem, keys_bkm: np.ndarray):
    """dK, dV (summed over the query heads of the KV group) for (b, hk, m) keys."""
    assert p.dout is not None
    keys_bkm = np.ascontiguousarray(keys_bkm, dtype=np.int32).reshape(-1, 3)
    R, d = keys_bkm.shape[0], p.shape[5]
    dk = np.zeros((R, d), np.float64)
    dv = np.zeros((R, d), np.float64)
    lib().ora_keys(p.ref(), R, _p(keys_bkm), _p(dk), _p(dv))
    return dk, dv


def attention(p: Problem):
    """Every output of the problem: O [B,Nq,Hq,d], LSE [B,Hq,Nq] and, with
    dout, dQ [B,Nq,Hq,d], dK / dV [B,Nk,Hkv,d].  Small cases only."""
    B, Nq, Nk, Hq, Hkv, d = p.shape
    bb, hh, nn = np.meshgrid(np.arange(B), np.arange(Hq), np.arange(Nq), indexing="ij")
    r = np.stack([bb.ravel(), hh.ravel(), nn.ravel()], 1)
    o, lse, dq = rows(p, r)
    O = o.reshape(B, Hq, Nq, d).transpose(0, 2, 1, 3).copy()
    LSE = lse.reshape(B, Hq, Nq)
    out = {"o": O, "lse": LSE}
    if p.dout is not None:
        out["dq"] = dq.reshape(B, Hq, Nq, d).transpose(0, 2, 1, 3).copy()
        bb, hh, mm = np.meshgrid(np.arange(B), np.arange(Hkv), np.arange(Nk), indexing="ij")
        kk = np.stack([bb.ravel(), hh.ravel(), mm.ravel()], 1)
        dk, dv = keys(p, kk)
        out["dk"] = dk.reshape(B, Hkv, Nk, d).transpose(0, 2, 1, 3).copy()
        out["dv"] = dv.reshape(B, Hkv, Nk, d).transpose(0, 2, 1, 3).copy()
    return out


def mask_dense(p: Problem, b: int, h: int) -> np.ndarray:
    """The VS mask of one head as a dense bool [Nq, Nk] (small cases only)."""
    B, Nq, Nk = p.shape[:3]
    out = np.zeros((Nq, Nk), np.uint8)
    lib().ora_mask_dense(p.ref(), int(b), int(h), _p(out))
    return out.astype(bool)


def mask_count(p: Problem) -> int:
    """|M| summed over (b, h, n): the effective mask area."""
    return int(lib().ora_mask_count(p.ref()))


# ------------------------------------------------------- striping and merging
def stripe_positions(N: int, W: int, stripe: int, r: int) -> np.ndarray:
    """Global positions of worker r's tokens under block-level striping."""
    pos = np.zeros(N // W, np.int64)
    lib().ora_stripe_positions(int(N), int(W), int(stripe), int(r), _p(pos))
    return pos


def striped_permute(x: np.ndarray, W: int, stripe: int, inverse: bool = False) -> np.ndarray:
    """x [B, N, H, d] -> [W, B, N/W, H, d] shards (or back with inverse=True):
    global block j goes to shard j mod W, local block j // W."""
    if not inverse:
        B, N = x.shape[:2]
        out = np.empty((W, B, N // W) + x.shape[2:], x.dtype)
        for j in range(N // stripe):
            out[j % W, :, (j // W) * stripe:(j // W + 1) * stripe] = x[:, j * stripe:(j + 1) * stripe]
        return out
    W_, B, Nl = x.shape[:3]
    N = Nl * W_
    out = np.empty((B, N) + x.shape[3:], x.dtype)
    for j in range(N // stripe):
        out[:, j * stripe:(j + 1) * stripe] = x[j % W_, :, (j // W_) * stripe:(j // W_ + 1) * stripe]
    return out


def ring_owners(N: int, W: int, layout: str, stripe: int = 64) -> np.ndarray:
    """Worker that holds each global token of a context-parallel ring.

    striped: block j = n // stripe lives on worker j mod W (Block-level
      Striped Sparse Ring Attention, section 4.2 (ii));
    zigzag: the sequence is cut into 2W chunks of N / (2W) tokens and worker
      r holds chunks r and 2W - 1 - r (the folded, mirrored layout of ZigZag
      Ring Attention, section 2 and Figure 1)."""
    n = np.arange(N, dtype=np.int64)
    if layout == "striped":
        return (n // stripe) % W
    if layout == "zigzag":
        c = n // (N // (2 * W))
        return np.where(c < W, c, 2 * W - 1 - c)
    raise ValueError(layout)


def ring_positions(N: int, W: int, r: int, layout: str, stripe: int = 64) -> np.ndarray:
    """Global positions of worker r's tokens in its shard's (local) order.
    striped: stripe_positions; zigzag: chunk r then chunk 2W - 1 - r of the
    2W chunks of N / (2W) tokens (section 2, Figure 1)."""
    if layout == "striped":
        return stripe_positions(N, W, stripe, r)
    if layout == "zigzag":
        C = N // (2 * W)
        first, second = r, 2 * W - 1 - r
        return np.concatenate([np.arange(first * C, (first + 1) * C), np.arange(second * C, (second + 1) * C)])
    raise ValueError(layout)


def ring_permute(x: np.ndarray, W: int, layout: str) -> np.ndarray:
    """x [B, N, H, d] -> [W, B, N/W, H, d]: shard r holds x at ring_positions(r)."""
    N = x.shape[1]
    return np.stack([x[:, ring_positions(N, W, r, layout)] for r in range(W)])


def ring_work(iv, is_, N: int, W: int, layout: str, stripe: int = 64) -> np.ndarray:
    """Effective work of every (query worker, key worker) pair: the number of
    entries of the VS mask on the global sequence whose query token lives on
    worker r and whose key token lives on worker q, summed over (b, h);
    int64 [W, W].  At ring step s worker r attends to the keys of worker
    (r - s) mod W, so its work at that step is out[r, (r - s) % W]."""
    iv = np.asarray(iv, np.int32)
    is_ = np.asarray(is_, np.int32)
    B, H = iv.shape[:2]
    own = ring_owners(N, W, layout, stripe)
    z = np.zeros((B, N, H, 1))
    p = Problem(z, np.zeros((B, N, 1, 1)), np.zeros((B, N, 1, 1)), iv, is_, 1.0)
    out = np.zeros((W, W), np.int64)
    for b in range(B):
        for h in range(H):
            n, m = np.nonzero(mask_dense(p, b, h))
            np.add.at(out, (own[n], own[m]), 1)
    return out


def merge(o1, l1, o2, l2):
    """merge_out_and_lse of Algorithm 2 for one row (fp64)."""
    o1 = np.ascontiguousarray(o1, np.float64)
    o2 = np.ascontiguousarray(o2, np.float64)
    o = np.zeros_like(o1)
    l = ctypes.c_double(0.0)
    lib().ora_merge(int(o1.shape[0]), _p(o1), float(l1), _p(o2), float(l2), _p(o), ctypes.byref(l))
    return o, l.value
