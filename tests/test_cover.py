"""The sheared tile cover of the slash part of the mask (host arithmetic, no
GPU), checked by brute force from its definition: E = {u : some selected
offset o in [u - 127, u]}, covered greedily by disjoint 64-wide intervals
starting at u_s; a 128-row query tile at r0 computes, per u_s <= r0 + 127,
keys [r0 + 64 - u_s, r0 + 127 - u_s]; a 128-key tile at k0 computes, per u_s,
rows [k0 + u_s, k0 + u_s + 63].  Claim: every causal entry whose offset n - m
is selected lies in exactly one unit of each cover (the pages' 64 x 64
block cover of the slashes, sheared so that every MMA has M = 128)."""
import numpy as np
import pytest


def greedy_starts(offsets, N):
    """Starts u_s of the greedy cover of E by disjoint 64-wide intervals."""
    sel = np.zeros(N + 256, bool)
    sel[np.asarray(offsets, np.int64)] = True
    in_e = np.zeros(N + 256, bool)
    for o in np.nonzero(sel)[0]:
        in_e[o:o + 128] = True
    starts, u = [], 0
    while u < len(in_e):
        if in_e[u]:
            starts.append(u)
            u += 64
        else:
            u += 1
    return [s for s in starts if s <= N + 126]


def check_cover(offsets, N):
    starts = greedy_starts(offsets, N)
    osel = np.zeros(N, bool)
    osel[np.asarray(offsets, np.int64)] = True
    # query-major: per tile, count the units covering each (row, key)
    for r0 in range(0, N, 128):
        rows = np.arange(r0, min(r0 + 128, N))
        cnt = np.zeros((len(rows), N), np.int32)
        for u in starts:
            if u > r0 + 127:
                continue
            k_lo, k_hi = r0 + 64 - u, r0 + 127 - u
            lo, hi = max(k_lo, 0), min(k_hi, N - 1)
            if lo <= hi:
                cnt[:, lo:hi + 1] += 1
        n = rows[:, None]
        m = np.arange(N)[None, :]
        want = (m <= n) & osel[np.clip(n - m, 0, N - 1)] & (n - m >= 0)
        assert np.all(cnt[want] == 1), ("query-major", r0)
        # units never reach past the causal diagonal of a selected entry's row
        assert np.all(cnt[(m > n + 127)] == 0)
    # key-major: per 128-key tile, count the units covering each (row, key)
    for k0 in range(0, N, 128):
        keys = np.arange(k0, min(k0 + 128, N))
        cnt = np.zeros((N, len(keys)), np.int32)
        for u in starts:
            lo, hi = k0 + u, min(k0 + u + 63, N - 1)
            if lo <= hi:
                cnt[lo:hi + 1, :] += 1
        n = np.arange(N)[:, None]
        m = keys[None, :]
        want = (m <= n) & osel[np.clip(n - m, 0, N - 1)] & (n - m >= 0)
        assert np.all(cnt[want] == 1), ("key-major", k0)


@pytest.mark.parametrize("offsets", [
    [0], [1], [63], [64], [127], [128], [1000], [1023],   # single diagonals
    list(range(0, 64)), list(range(5, 69)),                # 64-wide bands
    [0, 64, 128], [10, 75, 300, 301, 302, 1023],           # mixed
])
def test_fixed_selections(offsets):
    check_cover(offsets, 1024)


@pytest.mark.parametrize("seed", range(8))
def test_random_selections(seed):
    rng = np.random.default_rng(seed)
    N = 1024 + 64 * int(rng.integers(0, 8))  # a multiple of 64: possibly a ragged last 128-row tile
    k = int(rng.choice([4, 32, 200, N // 2]))
    offsets = np.sort(rng.choice(N, size=k, replace=False))
    check_cover(offsets, N)


def test_every_offset_gives_every_causal_tile():
    # ks = N: all offsets selected, the cover must be the full causal mask
    check_cover(list(range(512)), 512)
