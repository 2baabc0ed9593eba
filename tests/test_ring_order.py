"""Ring step order of the striped worker (host arithmetic, no GPU): the flat
ring of Balanced Sparse Ring Attention (MTraining section 4.2) and the
hierarchical order of Algorithm 2 (section 4.3)."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

from dynamic_vertical_slash_gb300.pipeline import ring_source  # noqa: E402


@pytest.mark.parametrize("world,inner", [(1, 0), (2, 0), (8, 0), (8, 2), (8, 4), (8, 8), (12, 3), (16, 4)])
def test_every_step_is_a_permutation_and_every_worker_sees_every_shard(world, inner):
    for s in range(world):
        srcs = [ring_source(r, s, world, inner) for r in range(world)]
        assert sorted(srcs) == list(range(world))  # each shard is read by exactly one worker per step
    for r in range(world):
        seq = [ring_source(r, s, world, inner) for s in range(world)]
        assert seq[0] == r  # the first step uses the worker's own shard
        assert sorted(seq) == list(range(world))  # over the ring every shard is visited once


def test_flat_ring_receives_from_the_previous_worker():
    assert [ring_source(0, s, 8) for s in range(8)] == [0, 7, 6, 5, 4, 3, 2, 1]
    assert [ring_source(3, s, 8) for s in range(8)] == [3, 2, 1, 0, 7, 6, 5, 4]


def test_hierarchical_order_inner_ring_inside_outer_ring():
    # two nodes of four cards: worker 0 runs its node's inner ring first
    # (its own card, then the node's cards 3, 2, 1), then the other node's
    # shards in the same inner order
    assert [ring_source(0, s, 8, 4) for s in range(8)] == [0, 3, 2, 1, 4, 7, 6, 5]
    # worker 5 = node 1, card 1
    assert [ring_source(5, s, 8, 4) for s in range(8)] == [5, 4, 7, 6, 1, 0, 3, 2]
    # inner = world is one node: the flat ring
    assert [ring_source(2, s, 8, 8) for s in range(8)] == [ring_source(2, s, 8) for s in range(8)]
    # inner = 1: every card is its own node, again the flat ring
    assert [ring_source(2, s, 8, 1) for s in range(8)] == [ring_source(2, s, 8) for s in range(8)]
