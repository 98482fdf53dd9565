"""Randomized checks of the GEMM kernel's mbarrier protocol (CPU only).

`pipeline_model` restates each role's waits and arrivals; these tests run
one block of every pipeline configuration the kernel builds, under random
interleavings and random completion orders, and look for deadlocks and for
buffers overwritten while in use.  The configurations are those of the
kernel's configuration table: A buffers NB, accumulators ND, weight stages,
and token slots, per format and token tile."""
import pytest

import pipeline_model as pm

# (format, token tile, groups per step): the counts the kernel's configuration
# derives from the 512 TMEM columns and 227 KB of shared memory; EPI is the
# number of epilogue warps (8; 12 at 96-token tiles; 4 at W8A8 tiles of 32
# and fewer)
CONFIGS = {
    "W4A16 T16 two-group": dict(mode="wo", NB=2, ND=2, stages=8, NX=8),
    "W4A16 T32 two-group": dict(mode="wo", NB=2, ND=2, stages=8, NX=4),
    "W4A16 T64 two-group": dict(mode="wo", NB=2, ND=2, stages=4, NX=4),
    "W4A16 T16": dict(mode="wo", NB=6, ND=2, stages=16, NX=16),
    "W4A16 T64": dict(mode="wo", NB=4, ND=2, stages=16, NX=4),
    "W4A16 T96": dict(mode="wo", NB=2, ND=2, stages=14, NX=4, EPI=12),
    "W8A16 T16": dict(mode="wo", NB=6, ND=2, stages=7, NX=16),
    "W8A8 T16": dict(mode="w8x", NB=4, ND=16, stages=10, NX=4, NXR=16, EPI=4),
    "W8A8 T32": dict(mode="w8x", NB=4, ND=8, stages=9, NX=4, NXR=8, EPI=4),
    "W8A8 T64": dict(mode="w8", NB=2, ND=6, stages=9, NX=4),
    "W8A8 T96": dict(mode="w8", NB=2, ND=4, stages=7, NX=4, EPI=12),
}

# (first step, end step, steps per tile): split tiles at both ends, whole
# tiles in between, short segments, chunks cut by segment ends
RANGES = [(6, 24, 20), (0, 40, 20), (19, 45, 20), (5, 60, 40), (2, 30, 8), (1, 33, 3),
          (0, 30, 2), (130, 170, 136), (7, 8, 20)]
ONE_GROUP = [(3, 11, 1), (0, 9, 1), (0, 24, 1), (5, 40, 1)]


def failures(cfg, ranges, seeds):
    out = {}
    for s0, s1, G in ranges:
        for seed in range(seeds):
            r = pm.run(cfg, s0, s1, G, seed)
            if r:
                out.setdefault((s0, s1, G), (seed, r))
                break
    return out


@pytest.mark.parametrize("name", sorted(CONFIGS))
def test_configurations_have_no_deadlock_or_hazard(name):
    cfg = CONFIGS[name]
    ranges = RANGES + ONE_GROUP
    assert failures(cfg, ranges, 25) == {}


def test_an_odd_a_buffer_count_breaks_the_protocol():
    """With three A buffers consecutive uses of a buffer alternate between
    the two converter groups.  A group then waits on `a_empty` for the use
    before its own previous one, and a parity wait cannot tell "one phase
    done" from "two phases behind": it passes early and overwrites an A
    buffer an MMA still reads.  The kernel keeps the count even."""
    cfg = dict(mode="wo", NB=3, ND=2, stages=8, NX=8)
    assert failures(cfg, [(6, 24, 20), (0, 40, 20)], 60) != {}


@pytest.mark.parametrize("name", ["W4A16 T16", "W4A16 T64", "W8A16 T16"])
def test_releasing_a_chunk_without_waiting_breaks_one_group_tiles(name):
    """Tiles of one 128-wide group make every scale chunk one step long.  If
    a converter warp released a chunk it had no step in without waiting for
    it to land, a group running four chunks ahead would add its releases to
    an earlier chunk's phase: the scale slot would be reloaded under a warp
    that still reads it (or the pipeline would stop).  The kernel's converter
    warps therefore wait for every chunk before they release it; this is the
    protocol without that wait."""
    cfg = dict(CONFIGS[name], release_without_landing=True)
    assert failures(cfg, ONE_GROUP, 60) != {}


@pytest.mark.parametrize("name", ["W4A16 T16", "W4A16 T64", "W8A16 T16"])
def test_one_group_tiles_weight_only(name):
    """The same one-group tiles with the kernel's protocol (wait for the
    chunk to land, then release it): no deadlock and no hazard."""
    assert failures(CONFIGS[name], ONE_GROUP + RANGES[:3], 60) == {}


def test_weights_released_before_a_full_scale_ring_blocks():
    """Weight-only formats hold the weight stream back until the first
    activation tiles are queued (x_go).  With one-step segments the scale
    ring fills first and drains only as the weights flow, so the activation
    producer releases x_go before it waits on a full scale ring; without
    that release the block stops."""
    cfg = dict(CONFIGS["W4A16 T16 two-group"], no_early_x_go=True)
    assert failures(cfg, [(0, 9, 1), (0, 24, 1)], 10) != {}
    assert failures(CONFIGS["W4A16 T16 two-group"], [(0, 9, 1), (0, 24, 1)], 10) == {}
