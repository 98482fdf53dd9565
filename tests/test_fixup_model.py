"""Randomized checks of the GEMM's cross-block split-tile protocol (CPU only).

`fixup_model` restates how blocks publish split-tile partials, count their
arrivals (the first contributor of a tile after its last step, publishing
only if another block finishes the tile), finish a tile in the last arriving
block and reset its counter;
these tests run several consecutive calls sharing one workspace under random
interleavings and random store visibility, over stream-K shapes like the
decode layers' (more blocks than tiles: tiles split across several blocks;
fewer: blocks spanning whole tiles), and check that the mistakes the protocol
guards against are caught."""
import pytest

import fixup_model as fm

# (steps W = tiles * G, groups per tile G, blocks C): 152 blocks over the
# gate/up, q/k/v and down shapes of the decode layer at one token tile, and
# small shapes with ragged block ranges
SHAPES = [(272 * 40, 40, 152), (48 * 40, 40, 152), (40 * 136, 136, 152), (7 * 20, 20, 9),
          (5 * 3, 3, 7), (12 * 8, 8, 5), (3 * 40, 40, 100), (2 * 2, 2, 3)]


def test_block_of_step_closed_form():
    """The kernel's closed form for the block holding step s,
    ceil((s + 1) C / W) - 1, agrees with a search over the ranges."""
    for W, G, C in SHAPES:
        for s in range(0, W, max(1, W // 997)):
            assert ((s + 1) * C + W - 1) // W - 1 == fm.block_of_step(s, W, C)


@pytest.mark.parametrize("W,G,C", SHAPES)
def test_split_tiles_finish_once_with_every_partial(W, G, C):
    for seed in range(6 if W > 2000 else 30):
        assert fm.run(W, G, C, calls=3, seed=seed) is None


@pytest.mark.parametrize("W,G,C", SHAPES[3:])
def test_publishing_before_every_arrival_is_also_correct(W, G, C):
    """The plainer protocol (every contributor publishes, then arrives)."""
    for seed in range(20):
        assert fm.run(W, G, C, calls=2, seed=seed, publish_first_everywhere=True) is None


@pytest.mark.parametrize("flaw", ["skip_flag_wait", "flag_before_flush"])
def test_reading_the_first_contributors_partial_before_its_flag_is_caught(flaw):
    """When the first contributor arrives before another block completes the
    count, it publishes afterwards: a finisher that does not wait for the
    published flag, or a flag raised before the partial is visible, reads a
    stale slot."""
    bad = [fm.run(W, G, C, calls=2, seed=s, **{flaw: True})
           for W, G, C in SHAPES[3:] for s in range(60)]
    assert any(r is not None and "read block" in r for r in bad)


@pytest.mark.parametrize("flaw", ["arrive_before_publish", "relaxed_arrival"])
def test_counting_an_arrival_before_its_partial_is_visible_is_caught(flaw):
    """The partial must be visible before the arrival that makes a block the
    last one: arriving first, or arriving without release semantics, lets the
    finisher read a stale slot."""
    bad = [fm.run(W, G, C, calls=2, seed=s, **{flaw: True})
           for W, G, C in SHAPES[3:] for s in range(40)]
    assert any(r is not None and "read block" in r for r in bad)


def test_a_counter_not_reset_is_caught():
    bad = [fm.run(W, G, C, calls=2, seed=s, no_reset=True) for W, G, C in SHAPES[3:] for s in range(3)]
    assert all(r is not None for r in bad)


def test_a_call_that_does_not_wait_for_the_previous_one_is_caught():
    """Without the grid dependency a block of the next call can overwrite a
    partial slot, or bump a counter, while the previous call still finishes
    its tiles."""
    bad = [fm.run(W, G, C, calls=2, seed=s, no_grid_wait=True)
           for W, G, C in SHAPES[3:] for s in range(60)]
    assert any(r is not None for r in bad)
