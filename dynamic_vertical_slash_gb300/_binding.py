"""ctypes binding of libvs.so (the C ABI in include/vs.h).

Argument marshalling only: every step of the path runs in the library's CUDA
kernels.  Torch tensors provide device memory and the current stream; outputs
and workspaces not passed in are allocated with torch.  A missing library is
an error, never a fallback.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional, Tuple

import numpy as np
import torch

from . import _build

VS_OK, VS_ERR_ARG, VS_ERR_SHAPE, VS_ERR_WORKSPACE, VS_ERR_INDEX, VS_ERR_TIMEOUT, VS_ERR_CUDA, VS_ERR_SCORE = range(8)


class VSError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__("%s: %s" % (where, status_string(code)))


class vs_shape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("Nq", ctypes.c_int), ("Nk", ctypes.c_int), ("Hq", ctypes.c_int),
                ("Hkv", ctypes.c_int), ("d", ctypes.c_int), ("sq", ctypes.c_int64 * 3), ("sk", ctypes.c_int64 * 3),
                ("sv", ctypes.c_int64 * 3), ("so", ctypes.c_int64 * 3)]


class vs_stripe(ctypes.Structure):
    _fields_ = [("world", ctypes.c_int), ("stripe", ctypes.c_int), ("q_rank", ctypes.c_int),
                ("kv_rank", ctypes.c_int), ("N_global", ctypes.c_int64)]


_lib = None
_P = ctypes.c_void_p
_S = ctypes.POINTER(vs_shape)


def lib_path() -> str:
    return _build.LIB


def lib(build_if_missing: bool = True):
    """The loaded libvs.so.  Raises if it is missing and cannot be built."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB
    if build_if_missing:
        path = _build.build()
    if not os.path.exists(path):
        raise RuntimeError("libvs.so is not built (%s); run __graft_entry__.build()" % path)
    L = ctypes.CDLL(path)
    L.vs_estimate_workspace.argtypes = [_S, ctypes.c_int]
    L.vs_estimate_workspace.restype = ctypes.c_size_t
    L.vs_estimate.argtypes = [_S, _P, _P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_float, _P, _P, _P, _P,
                              _P, ctypes.c_size_t, _P]
    L.vs_estimate_group.argtypes = [_S, _P, _P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_float, _P, _P,
                                    _P, _P, _P, ctypes.c_size_t, _P]
    L.vs_estimate_topp.argtypes = [_S, _P, _P, ctypes.c_int, ctypes.c_double, ctypes.c_double, ctypes.c_int,
                                   ctypes.c_int, ctypes.c_float, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]
    L.vs_select_topp.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, _P, _P, ctypes.c_double, ctypes.c_double,
                                 ctypes.c_int, ctypes.c_int, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]
    L.vs_block_index_bytes.argtypes = [_S, ctypes.c_int, ctypes.c_int, ctypes.POINTER(vs_stripe)]
    L.vs_block_index_bytes.restype = ctypes.c_size_t
    L.vs_build_block_index.argtypes = [_S, _P, _P, ctypes.c_int, ctypes.c_int, ctypes.POINTER(vs_stripe), _P,
                                       ctypes.c_size_t, _P]
    L.vs_build_block_index_ex.argtypes = [_S, _P, _P, ctypes.c_int, ctypes.c_int, ctypes.POINTER(vs_stripe),
                                          ctypes.c_int, _P, ctypes.c_size_t, _P]
    L.vs_index_counts.argtypes = [_P, _P, _P]
    L.vs_attn_fwd_workspace.argtypes = [_S]
    L.vs_attn_fwd_workspace.restype = ctypes.c_size_t
    L.vs_attn_fwd.argtypes = [_S, _P, _P, _P, _P, ctypes.c_float, _P, _P, _P, _P, ctypes.c_size_t, _P]
    L.vs_attn_bwd_workspace.argtypes = [_S, ctypes.c_int]
    L.vs_attn_bwd_workspace.restype = ctypes.c_size_t
    L.vs_attn_bwd.argtypes = [_S, _P, _P, _P, _P, _P, _P, _P, ctypes.c_float, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]
    L.vs_attn_bwd_ex.argtypes = [_S, _P, _P, _P, _P, _P, _P, _P, ctypes.c_float, _P, _P, _P, _P, _P, _P,
                                 ctypes.c_size_t, _P]
    L.vs_ring_permute.argtypes = [_P, _P, ctypes.c_int, ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                  ctypes.c_int, ctypes.c_int, ctypes.c_int, _P]
    L.striped_permute.argtypes = [_P, _P, ctypes.c_int, ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                  ctypes.c_int, ctypes.c_int, ctypes.c_int, _P]
    L.vs_ring_work.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int64, _P, ctypes.c_int, _P, ctypes.c_int,
                               ctypes.c_int, ctypes.c_int, _P, _P, ctypes.c_size_t, _P]
    L.vs_check_status.argtypes = [_P, _P]
    L.vs_selftest_wait_timeout.argtypes = [_P, ctypes.c_size_t, _P]
    L.vs_estimate_noalloc.argtypes = [_S, _P, _P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_float, _P, _P,
                                      _P, _P, _P]
    L.vs_estimate_noalloc_status.argtypes = [_P]
    L.vs_estimate_noalloc_selftest_plant.argtypes = [ctypes.c_int, _P]
    L.vs_status_string.argtypes = [ctypes.c_int]
    L.vs_status_string.restype = ctypes.c_char_p
    L.vs_launch_count.restype = ctypes.c_int64
    for name in ("vs_estimate", "vs_build_block_index", "vs_index_counts", "vs_attn_fwd", "vs_attn_bwd",
                 "striped_permute", "vs_check_status", "vs_selftest_wait_timeout", "vs_estimate_group",
                 "vs_estimate_topp", "vs_select_topp", "vs_build_block_index_ex", "vs_ring_work",
                 "vs_estimate_noalloc", "vs_estimate_noalloc_status", "vs_estimate_noalloc_selftest_plant",
                 "vs_attn_bwd_ex", "vs_ring_permute"):
        getattr(L, name).restype = ctypes.c_int
    _lib = L
    return L


def status_string(code: int) -> str:
    return lib().vs_status_string(int(code)).decode()


def launch_count() -> int:
    return int(lib().vs_launch_count())


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(code: int, where: str):
    if code != VS_OK:
        raise VSError(code, where)


def make_shape(q: torch.Tensor, k: torch.Tensor, v: Optional[torch.Tensor] = None,
               o: Optional[torch.Tensor] = None) -> vs_shape:
    """vs_shape from BSHD tensors q [B,Nq,Hq,d], k/v [B,Nk,Hkv,d], o like q."""
    v = k if v is None else v
    o = q if o is None else o
    B, Nq, Hq, d = q.shape
    Nk, Hkv = k.shape[1], k.shape[2]
    sh = vs_shape(B, Nq, Nk, Hq, Hkv, d)
    for name, t in (("sq", q), ("sk", k), ("sv", v), ("so", o)):
        if t.stride(3) != 1:
            raise ValueError("channel dimension of %s must be contiguous" % name)
        getattr(sh, name)[:] = [t.stride(0), t.stride(1), t.stride(2)]
    return sh


def _ws(nbytes: int, device) -> torch.Tensor:
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device)


# ------------------------------------------------------------------ entry points
def vs_estimate(q, k, kv: int, ks: int, scale: Optional[float] = None, last_q: int = 64, v_idx=None, s_idx=None,
                v_score=None, s_score=None, ws=None, stream=None, shared: bool = False):
    """Vertical and slash selection (Algorithm 1).  Returns (v_idx, s_idx) int32
    [B, Hq, kv] / [B, Hq, ks], sorted ascending.  shared=True: one selection
    per KV group (vs_estimate_group)."""
    sh = make_shape(q, k)
    B, N, Hq, d = q.shape
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    v_idx = torch.empty(B, Hq, kv, dtype=torch.int32, device=q.device) if v_idx is None else v_idx
    s_idx = torch.empty(B, Hq, ks, dtype=torch.int32, device=q.device) if s_idx is None else s_idx
    need = lib().vs_estimate_workspace(ctypes.byref(sh), last_q)
    ws = _ws(need, q.device) if ws is None else ws
    fn = lib().vs_estimate_group if shared else lib().vs_estimate
    _check(fn(ctypes.byref(sh), _ptr(q), _ptr(k), last_q, kv, ks, scale, _ptr(v_idx), _ptr(s_idx), _ptr(v_score),
              _ptr(s_score), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)), "vs_estimate")
    return v_idx, s_idx


def vs_estimate_topp(q, k, pv: float, ps: float, kv_max: int, ks_max: int, scale: Optional[float] = None,
                     last_q: int = 64, v_idx=None, s_idx=None, kv=None, ks=None, v_score=None, s_score=None, ws=None,
                     stream=None):
    """Vertical and slash selection with top-p budgets (Algorithm 1).  Returns
    (v_idx [B,Hq,kv_max], s_idx [B,Hq,ks_max], kv [B,Hq], ks [B,Hq]), int32;
    each list ascending, padded with -1 past its budget."""
    sh = make_shape(q, k)
    B, N, Hq, d = q.shape
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    dev = q.device
    v_idx = torch.empty(B, Hq, kv_max, dtype=torch.int32, device=dev) if v_idx is None else v_idx
    s_idx = torch.empty(B, Hq, ks_max, dtype=torch.int32, device=dev) if s_idx is None else s_idx
    kv = torch.empty(B, Hq, dtype=torch.int32, device=dev) if kv is None else kv
    ks = torch.empty(B, Hq, dtype=torch.int32, device=dev) if ks is None else ks
    need = lib().vs_estimate_workspace(ctypes.byref(sh), last_q)
    ws = _ws(need, dev) if ws is None else ws
    _check(lib().vs_estimate_topp(ctypes.byref(sh), _ptr(q), _ptr(k), last_q, float(pv), float(ps), kv_max, ks_max,
                                  scale, _ptr(v_idx), _ptr(s_idx), _ptr(kv), _ptr(ks), _ptr(v_score), _ptr(s_score),
                                  _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)), "vs_estimate_topp")
    return v_idx, s_idx, kv, ks


def vs_select_topp(v_score, s_score, pv: float, ps: float, kv_max: int, ks_max: int, v_idx=None, s_idx=None,
                   kv=None, ks=None, ws=None, stream=None):
    """Top-p budgets and selection on given fp32 scores [B, H, N]."""
    B, H, N = v_score.shape
    assert v_score.dtype == torch.float32 and s_score.dtype == torch.float32
    assert v_score.is_contiguous() and s_score.is_contiguous() and s_score.shape == v_score.shape
    dev = v_score.device
    v_idx = torch.empty(B, H, kv_max, dtype=torch.int32, device=dev) if v_idx is None else v_idx
    s_idx = torch.empty(B, H, ks_max, dtype=torch.int32, device=dev) if s_idx is None else s_idx
    kv = torch.empty(B, H, dtype=torch.int32, device=dev) if kv is None else kv
    ks = torch.empty(B, H, dtype=torch.int32, device=dev) if ks is None else ks
    ws = _ws(256, dev) if ws is None else ws
    _check(lib().vs_select_topp(B, H, N, _ptr(v_score), _ptr(s_score), float(pv), float(ps), kv_max, ks_max,
                                _ptr(v_idx), _ptr(s_idx), _ptr(kv), _ptr(ks), _ptr(ws),
                                ws.numel() * ws.element_size(), _stream(stream)), "vs_select_topp")
    return v_idx, s_idx, kv, ks


VS_LAYOUT_STRIPED, VS_LAYOUT_ZIGZAG = 0, 1


def vs_ring_work(v_idx, s_idx, N: int, world: int, layout: str = "striped", out=None, ws=None, stream=None):
    """Mask entries per (query worker, key worker) of a ring over the global
    lists: int64 device tensor [world, world] (see include/vs.h)."""
    B, H, kv = v_idx.shape
    ks = s_idx.shape[-1]
    lay = {"striped": VS_LAYOUT_STRIPED, "zigzag": VS_LAYOUT_ZIGZAG}[layout]
    out = torch.empty(world, world, dtype=torch.int64, device=v_idx.device) if out is None else out
    ws = _ws(256, v_idx.device) if ws is None else ws
    _check(lib().vs_ring_work(B, H, int(N), _ptr(v_idx), kv, _ptr(s_idx), ks, world, lay, _ptr(out), _ptr(ws),
                              ws.numel() * ws.element_size(), _stream(stream)), "vs_ring_work")
    return out


def make_stripe(world: int, q_rank: int, kv_rank: int, N_global: int, stripe: int = 64) -> vs_stripe:
    return vs_stripe(world, stripe, q_rank, kv_rank, N_global)


def make_window(q_start: int, k_start: int, N_global: int) -> vs_stripe:
    """Query rows and keys that are contiguous windows of the global sequence
    starting at tokens q_start / k_start (multiples of 64)."""
    if q_start % 64 or k_start % 64:
        raise ValueError("windows start on 64-token blocks")
    return vs_stripe(1, 64, q_start // 64, k_start // 64, N_global)


VS_INDEX_BLOCK_COVER, VS_INDEX_PACK_GQA = 1, 2


def vs_build_block_index(q, k, v_idx, s_idx, stripe: Optional[vs_stripe] = None, arena=None, stream=None,
                         block_cover: bool = False, pack_gqa: bool = False):
    """Sparse index arena (uint8 device tensor) for the shape of q / k;
    block_cover selects the block-cover reading of the slashes, pack_gqa the
    head-packed query-major tiles (lists equal within each KV group)."""
    sh = make_shape(q, k)
    kv, ks = v_idx.shape[-1], s_idx.shape[-1]
    sp = ctypes.byref(stripe) if stripe is not None else None
    need = lib().vs_block_index_bytes(ctypes.byref(sh), kv, ks, sp)
    if need == 0:
        raise VSError(VS_ERR_SHAPE, "vs_block_index_bytes")
    arena = torch.empty(need, dtype=torch.uint8, device=q.device) if arena is None else arena
    _check(lib().vs_build_block_index_ex(ctypes.byref(sh), _ptr(v_idx), _ptr(s_idx), kv, ks, sp,
                                         (VS_INDEX_BLOCK_COVER if block_cover else 0) |
                                         (VS_INDEX_PACK_GQA if pack_gqa else 0), _ptr(arena), arena.numel(),
                                         _stream(stream)), "vs_build_block_index")
    return arena


def vs_index_counts(arena, stream=None) -> np.ndarray:
    """Work units per (b, h): [B, Hq, 4] int64 (see include/vs.h)."""
    hdr = arena[:64].cpu().numpy().view(np.int32)
    B, Hq = int(hdr[2]), int(hdr[3])
    out = np.zeros((B, Hq, 4), np.int64)
    _check(lib().vs_index_counts(_ptr(arena), ctypes.c_void_p(out.ctypes.data), _stream(stream)), "vs_index_counts")
    return out


def vs_attn_fwd(q, k, v, arena, scale: Optional[float] = None, o=None, lse=None, o_acc=None, ws=None, stream=None):
    """Sparse forward.  Returns (o bf16 [B,Nq,Hq,d], lse fp32 [B,Hq,Nq])."""
    B, Nq, Hq, d = q.shape
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    o = torch.empty_like(q) if o is None else o
    lse = torch.empty(B, Hq, Nq, dtype=torch.float32, device=q.device) if lse is None else lse
    sh = make_shape(q, k, v, o)
    ws = _ws(lib().vs_attn_fwd_workspace(ctypes.byref(sh)), q.device) if ws is None else ws
    _check(lib().vs_attn_fwd(ctypes.byref(sh), _ptr(q), _ptr(k), _ptr(v), _ptr(arena), scale, _ptr(o), _ptr(lse),
                             _ptr(o_acc), _ptr(ws), ws.numel(), _stream(stream)), "vs_attn_fwd")
    return o, lse


def vs_attn_bwd(q, k, v, o, lse, dO, arena, kv: int, scale: Optional[float] = None, dq=None, dk=None, dv=None,
                dq_acc=None, ws=None, stream=None, dkv_acc=None):
    """Sparse backward.  Returns (dq, dk, dv) bf16.  dq_acc / dkv_acc: fp32
    accumulate modes (dkv_acc [2, B, Nk, Hkv, d], vs_attn_bwd_ex)."""
    d = q.shape[-1]
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if dO.stride() != o.stride():
        raise ValueError("dO must have the layout of o")
    sh = make_shape(q, k, v, o)
    ws = _ws(lib().vs_attn_bwd_workspace(ctypes.byref(sh), kv), q.device) if ws is None else ws
    if dkv_acc is None:
        _check(lib().vs_attn_bwd(ctypes.byref(sh), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dO),
                                 _ptr(arena), scale, _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dq_acc), _ptr(ws), ws.numel(),
                                 _stream(stream)), "vs_attn_bwd")
    else:
        _check(lib().vs_attn_bwd_ex(ctypes.byref(sh), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dO),
                                    _ptr(arena), scale, _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dq_acc), _ptr(dkv_acc),
                                    _ptr(ws), ws.numel(), _stream(stream)), "vs_attn_bwd_ex")
    return dq, dk, dv


def striped_permute(x, world: int, stripe: int = 64, inverse: bool = False, only_rank: int = -1, y=None,
                    stream=None):
    """Block-level striping of x [B, N, H, d] into [world, B, N/world, H, d]
    (or one shard with only_rank >= 0), or back with inverse=True."""
    if not inverse:
        B, N, H, d = x.shape
        shape = (B, N // world, H, d) if only_rank >= 0 else (world, B, N // world, H, d)
    else:
        W_, B, Nl, H, d = x.shape
        N = Nl * W_
        shape = (B, N, H, d)
    y = torch.empty(shape, dtype=x.dtype, device=x.device) if y is None else y
    _check(lib().striped_permute(_ptr(x), _ptr(y), B, N, H, d, world, stripe, int(inverse), only_rank,
                                 _stream(stream)), "striped_permute")
    return y


def ring_permute(x, world: int, layout: str = "zigzag", inverse: bool = False, only_rank: int = -1, y=None,
                 stream=None):
    """x [B, N, H, d] -> [world, B, N/world, H, d] shards of a striped or
    ZigZag ring (or one shard with only_rank >= 0), or back with inverse=True
    (vs_ring_permute)."""
    lay = {"striped": VS_LAYOUT_STRIPED, "zigzag": VS_LAYOUT_ZIGZAG}[layout]
    if not inverse:
        B, N, H, d = x.shape
        shape = (B, N // world, H, d) if only_rank >= 0 else (world, B, N // world, H, d)
    else:
        W_, B, Nl, H, d = x.shape
        N = Nl * W_
        shape = (B, N, H, d)
    y = torch.empty(shape, dtype=x.dtype, device=x.device) if y is None else y
    _check(lib().vs_ring_permute(_ptr(x), _ptr(y), B, N, H, d, world, lay, int(inverse), only_rank, _stream(stream)),
           "vs_ring_permute")
    return y


def vs_selftest_wait_timeout(ws, stream=None):
    """Launches the failure-detection self-test kernel (a bounded wait that
    runs out) on a uint8 workspace of at least 256 bytes."""
    _check(lib().vs_selftest_wait_timeout(_ptr(ws), ws.numel(), _stream(stream)), "vs_selftest_wait_timeout")


def vs_check_status(buf, stream=None) -> int:
    """Device status word of a workspace or arena (reset to VS_OK)."""
    return int(lib().vs_check_status(_ptr(buf), _stream(stream)))


# ------------------------------------------------------------------ tracing
def trace_enable(on: bool = True):
    lib().vs_trace_enable(1 if on else 0)


def trace_reset():
    lib().vs_trace_reset()


def trace_report() -> dict:
    """{kernel name: (launches, total ms)} since the last reset (synchronises)."""
    L = lib()
    L.vs_trace_report.argtypes = [ctypes.c_char_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
    L.vs_trace_report.restype = ctypes.c_int
    n_max = 64
    names = ctypes.create_string_buffer(4096)
    counts = np.zeros(n_max, np.int64)
    ms = np.zeros(n_max, np.float64)
    n = L.vs_trace_report(names, 4096, ctypes.c_void_p(counts.ctypes.data), ctypes.c_void_p(ms.ctypes.data), n_max)
    if n < 0:
        raise VSError(VS_ERR_CUDA, "vs_trace_report")
    keys = names.raw.split(b"\0")[:n]
    return {k.decode(): (int(c), float(t)) for k, c, t in zip(keys, counts[:n], ms[:n])}
