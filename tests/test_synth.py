"""Checks of the seeded input generator against the pages' RoPE algebra
(the expansion of z_{n,m} in the proof of Theorem 3.1) and library rounding."""
import math

import numpy as np
import torch

import synth


def test_bf16_rounding_matches_library():
    x = np.random.default_rng(0).standard_normal(100000).astype(np.float32) * 7
    x[:4] = [0.0, -0.0, 1e-40, 3.0e38]
    ours = synth.bf16_round(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)
    np.testing.assert_array_equal(synth.bf16_to_f32(ours), torch.from_numpy(ref.view(np.int16)).view(torch.bfloat16).float().numpy())


def test_rope_dot_product_is_the_theorem_expansion():
    # z_{n,m} = q_lo cos k_lo + q_hi cos k_hi + q_lo sin k_hi - q_hi sin k_lo at angle (n-m) theta
    d, N = 16, 50
    rng = np.random.default_rng(1)
    q = rng.standard_normal((N, 1, d)).astype(np.float32)
    k = rng.standard_normal((N, 1, d)).astype(np.float32)
    cos, sin = synth.rope_tables(N, d)
    qr = synth.apply_rope(q.astype(np.float64).copy(), cos.astype(np.float64), sin.astype(np.float64))
    kr = synth.apply_rope(k.astype(np.float64).copy(), cos.astype(np.float64), sin.astype(np.float64))
    theta = 10000.0 ** (-2.0 * np.arange(d // 2) / d)
    h = d // 2
    for n, m in [(10, 3), (49, 0), (7, 7), (20, 31)]:
        a = (n - m) * theta
        ql, qh, kl, kh = q[n, 0, :h], q[n, 0, h:], k[m, 0, :h], k[m, 0, h:]
        want = np.sum(ql * np.cos(a) * kl + qh * np.cos(a) * kh + ql * np.sin(a) * kh - qh * np.sin(a) * kl)
        assert abs(float(qr[n, 0] @ kr[m, 0]) - want) < 1e-5


def test_rope_relative_position_and_norm():
    d, N = 32, 64
    rng = np.random.default_rng(2)
    x = rng.standard_normal((N, 1, d))
    cos, sin = synth.rope_tables(N, d)
    xr = synth.apply_rope(x.copy(), cos.astype(np.float64), sin.astype(np.float64))
    np.testing.assert_allclose(np.linalg.norm(xr, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-6)
    # same vectors placed at shifted positions give the same dot product
    qv, kv = x[0, 0], x[1, 0]
    def at(vec, pos):
        y = np.tile(vec, (N, 1, 1))
        return synth.apply_rope(y, cos.astype(np.float64), sin.astype(np.float64))[pos, 0]
    assert abs(at(qv, 20) @ at(kv, 5) - at(qv, 40) @ at(kv, 25)) < 1e-5


def test_generator_is_deterministic_and_plants():
    w = synth.small_workload(N=512, Hq=4, Hkv=2, d=32, kv=8, ks=8, seed=3, n_out=5, n_slash=3)
    a = synth.make_batch(w)
    b = synth.make_batch(w)
    for key in ("q", "k", "v", "dout"):
        np.testing.assert_array_equal(a[key], b[key])
    k = synth.bf16_to_f32(a["k"])[0]
    norms = np.linalg.norm(k, axis=-1)  # [N, Hkv]
    for hk in range(2):
        cols = a["planted_cols"][0][hk]
        rest = np.setdiff1d(np.arange(512), cols)
        assert norms[cols, hk].min() > 2.5 * np.median(norms[rest, hk])
    assert a["q"].dtype == np.uint16 and a["q"].shape == (1, 512, 4, 32)


def test_band_plant_matches_direct_sum():
    w = synth.small_workload(N=256, Hq=2, Hkv=1, d=16, kv=4, ks=4, seed=4, band=20)
    x = synth.make_sequence(256, 2, 1, 16, w.seqs[0])
    y = synth.make_sequence(256, 2, 1, 16, synth.SeqSpec(seed=4))
    # undo: q_planted - q_plain ~= gamma/sqrt(w) * sum_{o=1..w} k[n-o]
    qd = synth.bf16_to_f32(x["q"]).astype(np.float64) - synth.bf16_to_f32(y["q"]).astype(np.float64)
    k = synth.bf16_to_f32(y["k"]).astype(np.float64)[:, 0]
    want = np.zeros((256, 16))
    for o in range(1, 21):
        want[o:] += k[: 256 - o]
    want *= synth.SLASH_GAMMA / math.sqrt(20)
    assert np.max(np.abs(qd[:, 0] - want)) < 0.1  # bf16 rounding of q dominates
