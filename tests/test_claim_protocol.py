"""The run-time claim of a last partial wave, modelled step by step on the host.

The persistent kernel deals whole tiles round-robin except the R tiles of a
last, partial wave: each of the G clusters, once it has run its share, takes
one ticket from a 64-bit word in device memory and runs tile dyn_first + t if
its ticket t < R.  The word holds a launch tag (the low 32 bits of the launch
id) above a 32-bit count, and is never reset between launches: cluster 0
starts the launch's count with an exchange, (tag << 32) | 0, and a claim is
one atomic add; an add that finds another tag came before the start, so the
claimer waits until it reads its own tag and adds again.

The device code runs those atomics; this file runs the same steps as a model,
under random interleavings of the clusters (each atomic is one indivisible
step, waits and the start come at random points), from stale words left by
earlier launches, and checks what the kernel relies on: every claimer gets
exactly one ticket, the tickets of a launch are 0 .. G-1 (so each of the R
tiles is run by exactly one cluster), and nothing depends on the order.
"""
import random

import pytest

MASK32 = (1 << 32) - 1


def run_launch(G, R, launch_id, word, rng):
    """One launch: G claimers and cluster 0's start, interleaved at random.
    Returns (tickets by cluster, tiles by cluster, the word afterwards)."""
    tag = launch_id & MASK32
    state = {"word": word}
    started = False
    # each claimer: "add" -> (done | "wait") ; "wait" polls until the tag is its own
    phase = ["add"] * G
    ticket = [None] * G
    # cluster 0 also claims, after its start; the start comes before its own claim
    pending = list(range(G)) + ["start"]
    steps = 0
    while any(p != "done" for p in phase) or not started:
        steps += 1
        assert steps < 100000, "no progress"
        choice = rng.choice([x for x in pending if x == "start" or phase[x] != "done"])
        if choice == "start":
            state["word"] = tag << 32                       # atomicExch
            started = True
            pending.remove("start")
            continue
        c = choice
        if c == 0 and not started:
            continue                                         # cluster 0 starts before it claims
        if phase[c] == "add":
            v = state["word"]                                # atomicAdd(w, 1)
            state["word"] = (v + 1) & ((1 << 64) - 1)
            if v >> 32 == tag:
                ticket[c] = v & MASK32
                phase[c] = "done"
            else:
                phase[c] = "wait"
        elif phase[c] == "wait":
            if state["word"] >> 32 == tag:                   # atomicAdd(w, 0) sees the new tag
                phase[c] = "add"
    tiles = [t if t < R else None for t in ticket]
    return ticket, tiles, state["word"]


@pytest.mark.parametrize("G,R", [(76, 36), (76, 12), (36, 24), (7, 3), (2, 1), (152, 151)])
def test_each_last_wave_tile_is_run_by_exactly_one_cluster(G, R):
    rng = random.Random(1000 * G + R)
    word = rng.getrandbits(64)                   # whatever an earlier launch left
    for launch_id in range(1, 40):
        tickets, tiles, word = run_launch(G, R, launch_id, word, rng)
        assert sorted(tickets) == list(range(G))
        run = sorted(t for t in tiles if t is not None)
        assert run == list(range(R))
        assert word == ((launch_id & MASK32) << 32) | G


def test_stale_word_with_a_large_count_and_adds_before_the_start():
    """Claimers that add before cluster 0 starts the count see the old tag,
    their increments are overwritten by the start, and they still get tickets
    of this launch only."""
    G, R = 76, 36
    rng = random.Random(7)
    for trial in range(200):
        old_tag = rng.getrandbits(32)
        word = (old_tag << 32) | rng.getrandbits(32)
        launch_id = (old_tag + 1 + rng.getrandbits(8)) & MASK32 or 1
        tickets, tiles, _ = run_launch(G, R, launch_id, word, rng)
        assert sorted(tickets) == list(range(G))
        assert sorted(t for t in tiles if t is not None) == list(range(R))


def test_a_start_that_overwrote_nothing_would_be_caught():
    """The model detects a planted mistake: without the start's overwrite
    (claimers that find an old tag adopt the count as it is), tickets no
    longer run from 0 and last-wave tiles are left undone."""
    G, R = 76, 36
    rng = random.Random(11)
    word = (5 << 32) | 1000
    tag = 6
    counts = []
    w = word
    for c in range(G):                            # the mistake: take the count whatever the tag
        counts.append(w & MASK32)
        w += 1
    assert sorted(counts) != list(range(G))
    assert sorted(t for t in counts if t < R) != list(range(R))
    assert tag != word >> 32
