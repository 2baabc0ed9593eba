"""vs_estimate_noalloc: the estimator entry point for callers that cannot
allocate device memory while they run (an engine that owns all device memory,
or a latency-critical loop that cannot afford cudaMalloc's device-wide
synchronisation).  Its scratch is a fixed array in the library's static device
memory; this test checks, through the C ABI, that two calls in a row give the
same selection and scores as vs_estimate with a caller workspace, that the
status reader of the fixed scratch reports a clean run and a recorded device
error (planted through the self-test hook), and that a problem too large for
the fixed scratch is refused before any launch.

Kept in a file of its own, named to be collected last."""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def _lib():
    import dynamic_vertical_slash_gb300 as vs

    L = vs.lib()
    L.vs_estimate_noalloc.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                      ctypes.c_int, ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                      ctypes.c_void_p, ctypes.c_void_p]
    L.vs_estimate_noalloc.restype = ctypes.c_int
    L.vs_estimate_noalloc_status.argtypes = [ctypes.c_void_p]
    L.vs_estimate_noalloc_status.restype = ctypes.c_int
    L.vs_estimate_noalloc_selftest_plant.argtypes = [ctypes.c_int, ctypes.c_void_p]
    L.vs_estimate_noalloc_selftest_plant.restype = ctypes.c_int
    return vs, L


def _inputs(B, N, Hq, Hkv, d, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, N, Hq, d, generator=g).to(torch.bfloat16).cuda()
    k = torch.randn(B, N, Hkv, d, generator=g)
    k[:, torch.randperm(N, generator=g)[:8]] *= 4  # a few outlier columns
    return q, k.to(torch.bfloat16).cuda()


def _noalloc(vs, L, q, k, kv, ks, scale):
    B, N, Hq, d = q.shape
    sh = vs.make_shape(q, k)
    out = [torch.full((B, Hq, kv), -7, dtype=torch.int32, device="cuda"),
           torch.full((B, Hq, ks), -7, dtype=torch.int32, device="cuda"),
           torch.full((B, Hq, N), -1.0, device="cuda"), torch.full((B, Hq, N), -1.0, device="cuda")]
    rc = L.vs_estimate_noalloc(ctypes.byref(sh), q.data_ptr(), k.data_ptr(), 64, kv, ks, scale,
                               *[t.data_ptr() for t in out], torch.cuda.current_stream().cuda_stream)
    return rc, out


def test_noalloc_matches_workspace_entry_point_on_consecutive_calls():
    vs, L = _lib()
    cases = [(1, 1024, 2, 1, 64, 32, 32, 11), (2, 4096, 4, 2, 128, 100, 300, 12)]
    for B, N, Hq, Hkv, d, kv, ks, seed in cases:  # two calls in a row, different shapes
        q, k = _inputs(B, N, Hq, Hkv, d, seed)
        scale = d ** -0.5
        vsc = torch.empty(B, Hq, N, device="cuda")
        ssc = torch.empty(B, Hq, N, device="cuda")
        iv_ref, is_ref = vs.vs_estimate(q, k, kv, ks, scale, 64, v_score=vsc, s_score=ssc)
        rc, (iv, is_, v2, s2) = _noalloc(vs, L, q, k, kv, ks, scale)
        torch.cuda.synchronize()
        assert rc == 0, vs.status_string(rc)
        assert torch.equal(iv, iv_ref) and torch.equal(is_, is_ref)
        for a, b in ((v2, vsc), (s2, ssc)):
            tol = 1e-4 * float(b.abs().max())
            assert float((a - b).abs().max()) <= tol
        # no device error was recorded in the fixed scratch
        assert L.vs_estimate_noalloc_status(torch.cuda.current_stream().cuda_stream) == 0


def test_noalloc_status_word_reports_device_errors_and_is_cleared():
    vs, L = _lib()
    st = torch.cuda.current_stream().cuda_stream
    q, k = _inputs(1, 1024, 2, 1, 64, 14)
    rc, _ = _noalloc(vs, L, q, k, 16, 16, 0.125)
    assert rc == 0
    assert L.vs_estimate_noalloc_status(st) == 0
    # a failing kernel writes its code into the status word; the reader
    # returns it once and resets the word
    assert L.vs_estimate_noalloc_selftest_plant(5, st) == 0  # VS_ERR_TIMEOUT
    assert L.vs_estimate_noalloc_status(st) == 5
    assert L.vs_estimate_noalloc_status(st) == 0
    # the next call clears a word nobody read, and computes again
    assert L.vs_estimate_noalloc_selftest_plant(5, st) == 0
    rc, (iv, is_, v2, s2) = _noalloc(vs, L, q, k, 16, 16, 0.125)
    torch.cuda.synchronize()
    assert rc == 0 and L.vs_estimate_noalloc_status(st) == 0
    iv_ref, is_ref = vs.vs_estimate(q, k, 16, 16, 0.125, 64)
    assert torch.equal(iv, iv_ref) and torch.equal(is_, is_ref)


def test_noalloc_refuses_problems_beyond_its_scratch():
    vs, L = _lib()
    q, k = _inputs(1, 1024, 2, 1, 64, 13)
    sh = vs.make_shape(q, k)
    sh.B, sh.Nq, sh.Nk, sh.Hq = 64, 131072, 131072, 16  # needs far more than 32 MiB; rejected on the host
    dummy = torch.empty(16, dtype=torch.int32, device="cuda")
    rc = L.vs_estimate_noalloc(ctypes.byref(sh), q.data_ptr(), k.data_ptr(), 64, 8, 8, 0.1, dummy.data_ptr(),
                               dummy.data_ptr(), dummy.data_ptr(), dummy.data_ptr(),
                               torch.cuda.current_stream().cuda_stream)
    assert rc == 3  # VS_ERR_WORKSPACE
