"""Pins for the oracle's block-cover mask (MTraining section 4.1 (ii):
slashes taken at the granularity of the kernel's 64 x 64 tiles): closed
forms for single slashes, containment of the exact mask, whole blocks, and
the full causal mask."""
import numpy as np
import pytest

import oracle
from vs_testutil import random_selection


def _p(N, iv, is_, block=True, Hq=1):
    z = np.zeros((1, N, Hq, 1))
    return oracle.Problem(z, np.zeros((1, N, 1, 1)), np.zeros((1, N, 1, 1)), iv, is_, 1.0, block=block)


@pytest.mark.parametrize("D0", [0, 1, 3])
def test_slash_on_a_block_multiple(D0):
    # o = 64 D0 passes only through block diagonal D0: |o - 64 D| <= 63 iff D = D0
    N = 512
    nb = N // 64
    iv = np.full((1, 1, 1), -1, np.int32)
    is_ = np.array([[[64 * D0]]], np.int32)
    want = nb * 2080 if D0 == 0 else (nb - D0) * 4096
    assert oracle.mask_count(_p(N, iv, is_)) == want


def test_slash_between_block_multiples():
    # o = 64 D0 + 32 passes through diagonals D0 and D0 + 1
    N, D0 = 512, 2
    iv = np.full((1, 1, 1), -1, np.int32)
    is_ = np.array([[[64 * D0 + 32]]], np.int32)
    nb = N // 64
    assert oracle.mask_count(_p(N, iv, is_)) == (nb - D0) * 4096 + (nb - D0 - 1) * 4096
    # offset 1 touches diagonals 0 and 1: the causal band of the first two
    is1 = np.array([[[1]]], np.int32)
    assert oracle.mask_count(_p(N, iv, is1)) == nb * 2080 + (nb - 1) * 4096


def test_contains_exact_and_is_whole_blocks():
    N = 640
    iv, is_ = random_selection(1, 2, N, 9, 12, 3)
    pb, pe = _p(N, iv, is_, Hq=2), _p(N, iv, is_, block=False, Hq=2)
    for h in range(2):
        mb, me = oracle.mask_dense(pb, 0, h), oracle.mask_dense(pe, 0, h)
        assert np.all(mb >= me)  # the exact mask is contained
        # outside the selected columns, the mask is a union of whole causal blocks
        cols = np.zeros(N, bool)
        cols[iv[0, h][iv[0, h] >= 0]] = True
        causal = np.tril(np.ones((N, N), bool))
        for I in range(N // 64):
            for J in range(I + 1):
                blk = mb[64 * I:64 * I + 64, 64 * J:64 * J + 64] & ~cols[None, 64 * J:64 * J + 64]
                cz = causal[64 * I:64 * I + 64, 64 * J:64 * J + 64] & ~cols[None, 64 * J:64 * J + 64]
                assert (not blk.any()) or np.array_equal(blk, cz)


def test_every_offset_is_full_causal():
    N = 384
    iv = np.full((1, 1, 1), -1, np.int32)
    is_ = np.arange(0, N, 64, dtype=np.int32).reshape(1, 1, -1)  # one slash per block diagonal
    assert oracle.mask_count(_p(N, iv, is_)) == N * (N + 1) // 2


def test_block_attention_equals_full_causal_when_every_diagonal_is_active():
    # one slash per block diagonal activates every block: the block mask is
    # the full causal mask, so every output (dK / dV included) equals the
    # exact computation with every offset selected
    rng = np.random.default_rng(4)
    N, d = 256, 8
    q, k, v, do = (rng.standard_normal((1, N, 1, d)) for _ in range(4))
    iv = np.full((1, 1, 1), -1, np.int32)
    blk = oracle.attention(oracle.Problem(q, k, v, iv, np.arange(0, N, 64, dtype=np.int32).reshape(1, 1, -1), 0.3,
                                          dout=do, block=True))
    full = oracle.attention(oracle.Problem(q, k, v, iv, np.arange(N, dtype=np.int32).reshape(1, 1, -1), 0.3,
                                           dout=do))
    for key in ("o", "lse", "dq", "dk", "dv"):
        np.testing.assert_allclose(blk[key], full[key], rtol=1e-12, atol=1e-12)
