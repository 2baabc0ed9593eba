"""Pins for the oracle's masked attention and its gradients.

Each test checks the oracle against something other than itself: torch's
scaled-dot-product attention and autograd (library routines), central finite
differences in fp64, the causal-area closed form, and identities the pages
state (softmax rows sum to 1; D = rowsum(dA (.) A) = rowsum(dO (.) O) from the
ring-attention backward; Eq. 1 implies every row of dS sums to 0).
"""
import math

import numpy as np
import pytest
import torch

import oracle


def _problem(N=128, Hq=2, Hkv=1, d=16, kv=8, ks=12, seed=0, B=1, dout=True, dense=False):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, N, Hq, d))
    k = rng.standard_normal((B, N, Hkv, d))
    v = rng.standard_normal((B, N, Hkv, d))
    do = rng.standard_normal((B, N, Hq, d)) if dout else None
    if dense:
        ks = N
    iv = np.stack([np.stack([np.sort(rng.choice(N, kv, replace=False)) for _ in range(Hq)]) for _ in range(B)])
    is_ = np.stack([np.stack([np.sort(rng.choice(N, ks, replace=False)) for _ in range(Hq)]) for _ in range(B)])
    return oracle.Problem(q, k, v, iv, is_, 1 / math.sqrt(d), dout=do)


def _mask_from_definition(p, b, h):
    """M[n, m] = (m <= n) and (m in iv or n - m in is), on global positions."""
    n = p.qpos[:, None]
    m = p.kpos[None, :]
    iv, is_ = p.iv[b, h], p.is_[b, h]
    off = n - m
    return (m <= n) & (np.isin(m, iv) | np.isin(np.where(off >= 0, off, -1), is_))


def _torch_masked(p, dense_mask_fn):
    """Masked softmax attention with torch autograd (float64) for reference."""
    B, Nq, Nk, Hq, Hkv, d = p.shape
    g = Hq // Hkv
    q = torch.tensor(p.q, requires_grad=True)
    k = torch.tensor(p.k, requires_grad=True)
    v = torch.tensor(p.v, requires_grad=True)
    kr = k.repeat_interleave(g, dim=2)
    vr = v.repeat_interleave(g, dim=2)
    S = torch.einsum("bnhc,bmhc->bhnm", q, kr) * p.scale
    M = torch.stack([torch.stack([torch.tensor(dense_mask_fn(p, b, h)) for h in range(Hq)]) for b in range(B)])
    S = S.masked_fill(~M, float("-inf"))
    lse = torch.logsumexp(S, dim=-1)
    A = torch.softmax(S, dim=-1).nan_to_num(0.0)
    O = torch.einsum("bhnm,bmhc->bnhc", A, vr)
    out = {"o": O, "lse": lse}
    if p.dout is not None:
        (O * torch.tensor(p.dout)).sum().backward()
        out.update(dq=q.grad, dk=k.grad, dv=v.grad)
    return out


def test_mask_enumeration_matches_definition():
    p = _problem(N=200, Hq=3, Hkv=1, kv=20, ks=30, seed=1)
    for h in range(3):
        np.testing.assert_array_equal(oracle.mask_dense(p, 0, h), _mask_from_definition(p, 0, h))


def test_causal_area_when_every_offset_is_selected():
    # ks = N covers the full causal mask; its area per head is N(N+1)/2
    N = 192
    p = _problem(N=N, Hq=2, Hkv=2, dense=True, dout=False)
    assert oracle.mask_count(p) == 2 * N * (N + 1) // 2


def test_dense_equals_library_causal_sdpa():
    p = _problem(N=160, Hq=4, Hkv=2, d=32, dense=True, seed=2)
    out = oracle.attention(p)
    q = torch.tensor(p.q).transpose(1, 2)
    k = torch.tensor(p.k).transpose(1, 2).repeat_interleave(2, dim=1)
    v = torch.tensor(p.v).transpose(1, 2).repeat_interleave(2, dim=1)
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True, scale=p.scale)
    np.testing.assert_allclose(out["o"], ref.transpose(1, 2).numpy(), rtol=0, atol=1e-12)


@pytest.mark.parametrize("seed", [3, 4])
def test_vs_mask_matches_library_masked_softmax_and_autograd(seed):
    p = _problem(N=144, Hq=4, Hkv=2, d=16, kv=10, ks=9, seed=seed)
    out = oracle.attention(p)
    ref = _torch_masked(p, _mask_from_definition)
    np.testing.assert_allclose(out["o"], ref["o"].detach().numpy(), rtol=0, atol=1e-12)
    finite = np.isfinite(ref["lse"].detach().numpy())
    np.testing.assert_array_equal(np.isfinite(out["lse"]), finite)
    np.testing.assert_allclose(out["lse"][finite], ref["lse"].detach().numpy()[finite], rtol=0, atol=1e-12)
    for key in ("dq", "dk", "dv"):
        np.testing.assert_allclose(out[key], ref[key].numpy(), rtol=0, atol=1e-11, err_msg=key)


def test_single_entry_row_and_empty_row():
    # row 0 may only see key 0; with 0 selected nowhere it is empty
    N, d = 64, 8
    rng = np.random.default_rng(5)
    q, k, v = (rng.standard_normal((1, N, 1, d)) for _ in range(3))
    do = rng.standard_normal((1, N, 1, d))
    iv = np.array([[[5]]])
    is_ = np.array([[[3]]])
    p = oracle.Problem(q, k, v, iv, is_, 0.5, dout=do)
    out = oracle.attention(p)
    assert np.all(out["o"][0, :3, 0] == 0) and np.all(np.isneginf(out["lse"][0, 0, :3]))
    assert np.all(out["dq"][0, :3, 0] == 0)
    # row 3 sees only key 0 (offset 3): O_3 = v_0 exactly, zero gradient to q_3
    np.testing.assert_array_equal(out["o"][0, 3, 0], v[0, 0, 0])
    np.testing.assert_allclose(out["dq"][0, 3, 0], 0, atol=1e-15)


def test_rows_of_attention_sum_to_one():
    p = _problem(N=128, Hq=2, Hkv=1, kv=9, ks=7, seed=6)
    p1 = oracle.Problem(p.q, p.k, np.ones_like(p.v), p.iv, p.is_, p.scale)
    out = oracle.attention(p1)
    nonempty = np.isfinite(out["lse"]).transpose(0, 2, 1)
    np.testing.assert_allclose(out["o"][nonempty], 1.0, rtol=0, atol=1e-13)


def test_finite_differences():
    # L = <dO, O>; central differences in fp64 for a sample of inputs
    p = _problem(N=96, Hq=2, Hkv=1, d=8, kv=6, ks=7, seed=7)
    out = oracle.attention(p)

    def loss(q, k, v):
        pp = oracle.Problem(q, k, v, p.iv, p.is_, p.scale)
        o = oracle.attention(pp)["o"]
        return float(np.sum(o * p.dout))

    rng = np.random.default_rng(8)
    eps = 1e-6
    for name, grad in (("q", out["dq"]), ("k", out["dk"]), ("v", out["dv"])):
        base = {"q": p.q, "k": p.k, "v": p.v}
        x = base[name]
        for _ in range(6):
            idx = tuple(int(rng.integers(0, s)) for s in x.shape)
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args_p = dict(base, **{name: xp})
            args_m = dict(base, **{name: xm})
            fd = (loss(**args_p) - loss(**args_m)) / (2 * eps)
            assert fd == pytest.approx(grad[idx], rel=1e-6, abs=1e-8), (name, idx)


def test_D_identity_and_gradient_sums():
    p = _problem(N=160, Hq=4, Hkv=2, d=16, kv=12, ks=10, seed=9)
    out = oracle.attention(p)
    B, Nq, Nk, Hq, Hkv, d = p.shape
    rows = np.array([(0, h, n) for h in range(Hq) for n in range(Nq)], np.int32)
    lse, D = oracle.row_stats(p, rows)
    # D_n = rowsum(dA (.) A) equals rowsum(dO (.) O) (ring-attention backward)
    O = out["o"][0].transpose(1, 0, 2).reshape(-1, d)
    dO = p.dout[0].transpose(1, 0, 2).reshape(-1, d)
    np.testing.assert_allclose(D, np.sum(O * dO, -1), rtol=0, atol=1e-12)
    # every row of dS sums to 0, so sum_m dK_m = 0 per KV head
    np.testing.assert_allclose(out["dk"].sum(1), 0, atol=1e-11)
    # sum_m dV_m = sum over the group's heads of dO_n over non-empty rows
    ne = np.isfinite(out["lse"][0])  # [Hq, N]
    g = Hq // Hkv
    for hk in range(Hkv):
        want = sum(p.dout[0, ne[h], h].sum(0) for h in range(hk * g, (hk + 1) * g))
        np.testing.assert_allclose(out["dv"][0, :, hk].sum(0), want, atol=1e-11)


def test_sampled_rows_and_keys_match_full():
    p = _problem(N=128, Hq=4, Hkv=2, d=16, kv=8, ks=8, seed=10, B=2)
    full = oracle.attention(p)
    rows = np.array([(1, 3, 77), (0, 0, 5), (1, 1, 127)], np.int32)
    o, lse, dq = oracle.rows(p, rows)
    for r, (b, h, n) in enumerate(rows):
        np.testing.assert_allclose(o[r], full["o"][b, n, h], atol=1e-14)
        np.testing.assert_allclose(dq[r], full["dq"][b, n, h], atol=1e-14)
    keys = np.array([(1, 0, 3), (0, 1, 100)], np.int32)
    dk, dv = oracle.keys(p, keys)
    for r, (b, hk, m) in enumerate(keys):
        np.testing.assert_allclose(dk[r], full["dk"][b, m, hk], atol=1e-14)
        np.testing.assert_allclose(dv[r], full["dv"][b, m, hk], atol=1e-14)
