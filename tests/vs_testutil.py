"""Helpers shared by the tests: seeded inputs on both sides, error norms, and a
host-side decoder of the device index arena (for mask-coverage checks)."""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle
import synth

HDR_FIELDS = ["status", "magic", "B", "Hq", "Nq", "Nk", "kv", "ks", "world", "stripe", "q_rank", "kv_rank"]


def dev_bf16(bits: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def host_f64(t_or_bits) -> np.ndarray:
    if isinstance(t_or_bits, torch.Tensor):
        return t_or_bits.detach().float().cpu().numpy().astype(np.float64)
    return synth.bf16_to_f32(t_or_bits).astype(np.float64)


def rel_l2(x, y) -> float:
    x = np.asarray(x, np.float64)
    y = np.asarray(y, np.float64)
    den = np.linalg.norm(y)
    return float(np.linalg.norm(x - y) / den) if den > 0 else float(np.linalg.norm(x))


def random_selection(B, Hq, N_global, kv, ks, seed):
    rng = np.random.default_rng(seed)
    iv = np.stack([np.stack([np.sort(rng.choice(N_global, kv, replace=False)) for _ in range(Hq)])
                   for _ in range(B)]).astype(np.int32)
    is_ = np.stack([np.stack([np.sort(rng.choice(N_global, ks, replace=False)) for _ in range(Hq)])
                    for _ in range(B)]).astype(np.int32)
    return iv, is_


def make_inputs(B, N, Hq, Hkv, d, seed, n_out=0, n_slash=0, band=0):
    w = synth.small_workload(N=N, Hq=Hq, Hkv=Hkv, d=d, kv=1, ks=1, seed=seed, n_out=n_out, n_slash=n_slash,
                             band=band, B=B)
    return w, synth.make_batch(w)


# ------------------------------------------------------------- arena decoding
class Arena:
    """Host copy of an index arena with the documented layout."""

    def __init__(self, arena: torch.Tensor):
        raw = arena.cpu().numpy()
        i32 = raw[:256].view(np.int32)
        self.h = dict(zip(HDR_FIELDS, i32[:12].tolist()))
        i64 = raw[:256].view(np.int64)
        self.N_global = int(i64[6])
        self.WG, self.WL, self.EMAX, self.KVP, self.sheared, self.block_cover = [int(x) for x in i32[14:20]]
        offs = i64[10:22]
        names = ["offbits", "colbits", "elist", "ecount", "flist", "fcount", "vlist", "vcount", "vlocbits",
                 "vlocpre", "counts", "total"]
        self.off = dict(zip(names, [int(x) for x in offs]))
        BH = self.h["B"] * self.h["Hq"]
        self.raw = raw
        g = lambda name, dt, n: raw[self.off[name]: self.off[name] + n * np.dtype(dt).itemsize].view(dt)
        self.offbits = g("offbits", np.uint64, BH * self.WG).reshape(BH, self.WG)
        self.colbits = g("colbits", np.uint64, BH * self.WG).reshape(BH, self.WG)
        self.elist = g("elist", np.int32, BH * self.EMAX).reshape(BH, self.EMAX)
        self.ecount = g("ecount", np.int32, BH)
        self.flist = g("flist", np.int32, BH * self.EMAX).reshape(BH, self.EMAX)
        self.fcount = g("fcount", np.int32, BH)
        self.vlist = g("vlist", np.int32, BH * self.KVP).reshape(BH, self.KVP)
        self.vcount = g("vcount", np.int32, BH)
        self.counts = g("counts", np.int64, BH * 4).reshape(BH, 4)
        self.off["bdbits"] = int(i64[22])
        self.bdbits = g("bdbits", np.uint64, BH * self.WG).reshape(BH, self.WG)

    def bit(self, bm_row, pos):
        pos = np.asarray(pos, np.int64)
        ok = (pos >= 0) & (pos < 64 * bm_row.size)
        p = np.where(ok, pos, 0)
        return ok & (((bm_row[p >> 6] >> (p & 63).astype(np.uint64)) & np.uint64(1)) == 1)

    def qpos(self, l):
        W, r = self.h["world"], self.h["q_rank"]
        l = np.asarray(l, np.int64)
        return (W * (l >> 6) + r) * 64 + (l & 63)

    def kpos(self, l):
        W, r = self.h["world"], self.h["kv_rank"]
        l = np.asarray(l, np.int64)
        return (W * (l >> 6) + r) * 64 + (l & 63)

    def _slash(self, bh, ng, mg):
        """Slash part of the mask at global (row, key) positions: the offset
        selected (exact), or the block diagonal active (block cover)."""
        off = ng - mg
        if self.block_cover:
            return self.bit(self.bdbits[bh], (ng >> 6) - (mg >> 6)) & (off >= 0)
        return self.bit(self.offbits[bh], off) & (off >= 0)

    def coverage_query_major(self, bh):
        """Times each (row, key) entry is computed by the query-major passes."""
        Nq, Nk = self.h["Nq"], self.h["Nk"]
        cov = np.zeros((Nq, Nk), np.int32)
        T = (Nq + 127) // 128
        e = self.elist[bh, : self.ecount[bh]]
        vl = self.vlist[bh, : self.vcount[bh]]
        for t in range(T):
            rows = np.arange(128 * t, min(128 * t + 128, Nq))
            ng = self.qpos(rows)
            for ee in e[e <= 128 * t + 127]:
                c = 128 * t + 64 - int(ee)
                keys = np.arange(c, c + 64)
                kk = keys[(keys >= 0) & (keys < Nk)]
                mg = self.kpos(kk) if c >= 0 else kk
                off = ng[:, None] - mg[None, :]
                sel = self._slash(bh, ng[:, None], mg[None, :]) & ~self.bit(self.colbits[bh], mg)[None, :]
                cov[np.ix_(rows, kk)] += sel
            nb = 0
            while nb * 64 < vl.size and vl[nb * 64] <= 128 * t + 127:
                nb += 1
            for c in range(nb):
                kk = vl[c * 64:(c + 1) * 64]
                sel = self.kpos(kk)[None, :] <= ng[:, None]
                cov[np.ix_(rows, kk)] += sel
        return cov

    def coverage_key_major(self, bh):
        """Times each entry is computed by the key-major (dK / dV) passes."""
        Nq, Nk = self.h["Nq"], self.h["Nk"]
        cov = np.zeros((Nq, Nk), np.int32)
        f = self.flist[bh, : self.fcount[bh]]
        vl = self.vlist[bh, : self.vcount[bh]]
        vset = np.zeros(Nk, bool)
        vset[vl] = True
        for k0 in range(0, Nk, 128):
            keys = np.arange(k0, min(k0 + 128, Nk))
            mg = self.kpos(keys)
            for ff in f[k0 + f <= Nq - 1]:
                r0 = k0 + int(ff)
                rows = np.arange(r0, min(r0 + 64, Nq))
                sel = self._slash(bh, self.qpos(rows)[:, None], mg[None, :]) & ~vset[keys][None, :]
                cov[np.ix_(rows, keys)] += sel
        for c in range(0, vl.size, 128):
            kk = vl[c:c + 128]
            rs = (kk[0] // 64) * 64
            rows = np.arange(rs, Nq)
            sel = self.kpos(kk)[None, :] <= self.qpos(rows)[:, None]
            cov[np.ix_(rows, kk)] += sel
        return cov
