"""The C ABI without a GPU: the library loads, exports every function that
include/vs.h declares, and rejects bad arguments on the host before any
launch."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^\s*(?:[A-Za-z_][\w\s\*]*?)\b([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "return", "sizeof")))


@pytest.fixture(scope="module")
def L():
    from dynamic_vertical_slash_gb300 import _binding

    return _binding.lib()


def test_every_declared_symbol_is_exported(L):
    names = _declared()
    assert {"vs_estimate", "vs_build_block_index", "vs_attn_fwd", "vs_attn_bwd", "striped_permute",
            "vs_check_status", "vs_status_string"} <= set(names)
    for n in names:
        assert hasattr(L, n), n


def _shape(B=1, N=1024, Hq=2, Hkv=1, d=64):
    from dynamic_vertical_slash_gb300._binding import vs_shape

    sh = vs_shape(B, N, N, Hq, Hkv, d)
    sh.sq[:] = [N * Hq * d, Hq * d, d]
    sh.so[:] = [N * Hq * d, Hq * d, d]
    sh.sk[:] = [N * Hkv * d, Hkv * d, d]
    sh.sv[:] = [N * Hkv * d, Hkv * d, d]
    return sh


def test_status_strings(L):
    for code in range(8):
        assert L.vs_status_string(code)
    assert b"VS_ERR_SHAPE" in L.vs_status_string(2)


def test_host_validation_rejects_before_launch(L):
    from dynamic_vertical_slash_gb300._binding import VS_ERR_ARG, VS_ERR_SHAPE, VS_ERR_WORKSPACE

    fake = ctypes.c_void_p(0x10000)  # never dereferenced: validation fails first
    sh = _shape(d=96)
    assert L.vs_attn_fwd(ctypes.byref(sh), fake, fake, fake, fake, 0.1, fake, fake, None, fake, 256, None) == VS_ERR_SHAPE
    sh = _shape(N=1000)
    assert L.vs_attn_fwd(ctypes.byref(sh), fake, fake, fake, fake, 0.1, fake, fake, None, fake, 256, None) == VS_ERR_SHAPE
    sh = _shape(Hq=3, Hkv=2)
    assert L.vs_attn_bwd(ctypes.byref(sh), fake, fake, fake, fake, fake, fake, fake, 0.1, fake, fake, fake, None,
                         fake, 1 << 30, None) == VS_ERR_SHAPE
    sh = _shape()
    assert L.vs_attn_fwd(ctypes.byref(sh), None, fake, fake, fake, 0.1, fake, fake, None, fake, 256, None) == VS_ERR_ARG
    assert L.vs_attn_fwd(ctypes.byref(sh), fake, fake, fake, fake, -1.0, fake, fake, None, fake, 256, None) == VS_ERR_ARG
    assert L.vs_attn_fwd(ctypes.byref(sh), fake, fake, fake, fake, 0.1, fake, fake, None, fake, 16, None) == VS_ERR_WORKSPACE
    assert L.vs_estimate(ctypes.byref(sh), fake, fake, 32, 8, 8, 0.1, fake, fake, None, None, fake, 1 << 30, None) == VS_ERR_ARG
    assert L.vs_estimate(ctypes.byref(sh), fake, fake, 64, 0, 8, 0.1, fake, fake, None, None, fake, 1 << 30, None) == VS_ERR_ARG
    assert L.vs_estimate(ctypes.byref(sh), fake, fake, 64, 8, 8, 0.1, fake, fake, None, None, fake, 16, None) == VS_ERR_WORKSPACE
    need = L.vs_block_index_bytes(ctypes.byref(sh), 32, 32, None)
    assert need > 256
    assert L.vs_build_block_index(ctypes.byref(sh), fake, fake, 32, 2000, None, fake, need, None) == VS_ERR_ARG
    assert L.vs_build_block_index(ctypes.byref(sh), fake, fake, 32, 32, None, fake, need - 1, None) == VS_ERR_WORKSPACE
    sh.sq[1] = 13  # stride not a multiple of 8 elements
    assert L.vs_attn_fwd(ctypes.byref(sh), fake, fake, fake, fake, 0.1, fake, fake, None, fake, 256, None) == VS_ERR_SHAPE
    assert L.striped_permute(fake, fake, 1, 1000, 1, 64, 4, 64, 0, -1, None) == VS_ERR_SHAPE
    assert L.striped_permute(fake, fake, 1, 1024, 1, 64, 4, 32, 0, -1, None) == VS_ERR_SHAPE
    assert L.striped_permute(fake, fake, 1, 1024, 1, 64, 4, 64, 1, 2, None) == VS_ERR_ARG


def test_workspace_queries(L):
    sh = _shape(N=4096, Hq=16, Hkv=2, d=128)
    assert L.vs_estimate_workspace(ctypes.byref(sh), 64) > 0
    assert L.vs_attn_fwd_workspace(ctypes.byref(sh)) == 256
    a = L.vs_attn_bwd_workspace(ctypes.byref(sh), 128)
    b = L.vs_attn_bwd_workspace(ctypes.byref(sh), 1024)
    assert b > a > 0


def test_estimator_entry_points_refuse_the_same_arguments(L):
    # vs_estimate_noalloc validates exactly what vs_estimate validates (one
    # shared routine), on the host, before any CUDA call
    fake = ctypes.c_void_p(0x10000)
    cases = []
    for kw in (dict(d=96), dict(N=1000), dict(Hq=3, Hkv=2), dict(Hq=130, Hkv=2), dict(B=0)):
        cases.append((_shape(**kw), 64, 8, 8, 0.1))
    sh = _shape()
    sh.sq[2] = 32  # head stride below d
    cases.append((sh, 64, 8, 8, 0.1))
    sh = _shape()
    sh.sk[1] = 12  # token stride not a multiple of 8 elements
    cases.append((sh, 64, 8, 8, 0.1))
    sh = _shape()
    sh.Nk = 512  # Nq != Nk
    cases.append((sh, 64, 8, 8, 0.1))
    for args in ((_shape(), 32, 8, 8, 0.1), (_shape(), 64, 0, 8, 0.1), (_shape(), 64, 8, 2000, 0.1),
                 (_shape(), 64, 8, 8, -1.0)):
        cases.append(args)
    for sh, last_q, kv, ks, scale in cases:
        a = L.vs_estimate(ctypes.byref(sh), fake, fake, last_q, kv, ks, scale, fake, fake, None, None, fake, 1 << 40,
                          None)
        b = L.vs_estimate_noalloc(ctypes.byref(sh), fake, fake, last_q, kv, ks, scale, fake, fake, fake, fake, None)
        assert a == b != 0, (a, b)
    # missing score buffers are refused by the no-alloc entry point (it keeps no scores of its own)
    sh = _shape()
    assert L.vs_estimate_noalloc(ctypes.byref(sh), fake, fake, 64, 8, 8, 0.1, fake, fake, None, fake, None) == 1


def test_packed_index_host_validation(L):
    from dynamic_vertical_slash_gb300._binding import VS_ERR_ARG, VS_ERR_SHAPE, make_stripe

    fake = ctypes.c_void_p(0x10000)
    PACK, BLOCK = 2, 1
    sh = _shape(Hq=8, Hkv=1)
    need = L.vs_block_index_bytes(ctypes.byref(sh), 32, 32, None)
    st = make_stripe(2, 0, 1, 2048)
    assert L.vs_build_block_index_ex(ctypes.byref(sh), fake, fake, 32, 32, ctypes.byref(st), PACK, fake, 1 << 30,
                                     None) == VS_ERR_ARG
    assert L.vs_build_block_index_ex(ctypes.byref(sh), fake, fake, 32, 32, None, PACK | BLOCK, fake, need,
                                     None) == VS_ERR_ARG
    sh1 = _shape(Hq=2, Hkv=2)  # g = 1: nothing to pack
    assert L.vs_build_block_index_ex(ctypes.byref(sh1), fake, fake, 32, 32, None, PACK, fake, need, None) == VS_ERR_SHAPE
    sh3 = _shape(Hq=3, Hkv=1)  # g = 3 does not divide a 128-row tile
    assert L.vs_build_block_index_ex(ctypes.byref(sh3), fake, fake, 32, 32, None, PACK, fake, need, None) == VS_ERR_SHAPE
    assert L.vs_build_block_index_ex(ctypes.byref(sh), fake, fake, 32, 32, None, 4, fake, need, None) == VS_ERR_ARG
