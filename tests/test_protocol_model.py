"""The cross-rank buffer-reuse rules, checked on a model of the ranks.

No GPU and no library call: each rank is a program of events in stream
order -- the layer writing its partial, the barrier's post and wait (a
flag per rank holding the last epoch posted, as the signal pads do), and
the reads and writes of the epilogue and of the two stages.  A random
scheduler interleaves the ranks in every way stream order and the barriers
allow, and the test looks for a write into a buffer while an earlier call
of some rank is still reading it.

What it checks is the argument the library's documentation makes:
* one-shot calls with two partials used in turn need no end barrier (the
  group object's calls, also mixed with two-shot calls), while one partial
  without the end barrier races;
* the one-shot call with its end barrier is safe with one partial;
* the two-shot call, with a barrier before stage 1 and one between the
  stages, is safe with one partial and one set of temporaries; without the
  first barrier a fast rank's stage 1 reads a partial its owner is still
  writing;
* a CUDA graph of the group object's calls, replayed back to back, needs
  an even number of captured calls or a barrier at its end.
"""
import random

import pytest


def _one_shot(rank, world, k, partial, end_barrier):
    """Events of rank `rank` for one-shot call k reading partial set `partial`."""
    ev = [("write", ("P", partial, rank)), ("post", k), ("wait", k),
          ("read_begin", [("P", partial, q) for q in range(world)])]
    ev.append(("read_end", None))
    if end_barrier:
        ev += [("post", ("end", k)), ("wait", ("end", k))]
    return ev


def _two_shot(rank, world, k, partial, temp, first_barrier=True):
    """Events of rank `rank` for two-shot call k: a barrier (every partial
    written), stage 1 reading every rank's partial (its slice) and storing
    into every rank's temporary, a barrier, stage 2 reading its own
    temporary.  first_barrier=False leaves the first barrier out."""
    ev = [("write", ("P", partial, rank))]
    if first_barrier:
        ev += [("post", ("first", k)), ("wait", ("first", k))]
    return ev + [("read_begin", [("P", partial, q) for q in range(world)]),
                 ("write_all", [("T", temp, q) for q in range(world)]),
                 ("read_end", None),
                 ("post", k), ("wait", k),
                 ("read_begin", [("T", temp, rank)]), ("read_end", None)]


def _programs(world, calls, kind, partial_sets, temp_sets, end_barrier, first_barrier=True):
    """`kind` is "one_shot", "two_shot" or a list naming each call's path."""
    progs = []
    for r in range(world):
        ev, two = [], 0
        for k in range(calls):
            p = k % partial_sets
            if (kind if isinstance(kind, str) else kind[k]) == "one_shot":
                ev += _one_shot(r, world, k, p, end_barrier)
            else:
                ev += _two_shot(r, world, k, p, two % temp_sets, first_barrier)
                two += 1
        progs.append(ev)
    return progs


def _run(progs, rng):
    """Interleave the programs at random; return the first race found."""
    world = len(progs)
    pc = [0] * world
    posted = [set() for _ in range(world)]      # epochs rank r has posted
    reading = {}                                 # rank -> buffers it reads now
    while any(pc[r] < len(progs[r]) for r in range(world)):
        ready = []
        for r in range(world):
            if pc[r] >= len(progs[r]):
                continue
            op, arg = progs[r][pc[r]]
            if op == "wait" and not all(arg in posted[q] for q in range(world)):
                continue
            ready.append(r)
        assert ready, "deadlock: every rank waits"
        r = rng.choice(ready)
        op, arg = progs[r][pc[r]]
        pc[r] += 1
        if op in ("write", "write_all"):
            targets = [arg] if op == "write" else arg
            for q, bufs in reading.items():
                for t in targets:
                    if t in bufs:
                        return (r, t, q)
        elif op == "post":
            posted[r].add(arg)
        elif op == "read_begin":
            reading[r] = set(arg)
        elif op == "read_end":
            reading.pop(r, None)
    return None


def _races(world, calls, kind, partial_sets, temp_sets=1, end_barrier=False, first_barrier=True,
           trials=400, seed=0):
    rng = random.Random(seed)
    progs = _programs(world, calls, kind, partial_sets, temp_sets, end_barrier, first_barrier)
    return sum(_run(progs, rng) is not None for _ in range(trials))


@pytest.mark.parametrize("world", [2, 3, 4])
def test_one_shot_with_two_partials_in_turn_needs_no_end_barrier(world):
    assert _races(world, 6, "one_shot", partial_sets=2) == 0


@pytest.mark.parametrize("world", [2, 4])
def test_one_shot_with_one_partial_needs_the_end_barrier(world):
    assert _races(world, 6, "one_shot", partial_sets=1) > 0          # the model sees the race
    assert _races(world, 6, "one_shot", partial_sets=1, end_barrier=True) == 0


@pytest.mark.parametrize("world", [2, 3, 4])
def test_two_shot_with_both_barriers_needs_one_partial_and_one_temporary(world):
    assert _races(world, 6, "two_shot", partial_sets=1, temp_sets=1) == 0


@pytest.mark.parametrize("world", [2, 4])
def test_two_shot_without_the_first_barrier_races(world):
    """Stage 1 reads a slice of every rank's partial: without a barrier
    before it, a fast rank reads a partial its owner is still writing --
    whatever the buffers' rotation."""
    for sets in (1, 2):
        assert _races(world, 6, "two_shot", partial_sets=sets, temp_sets=sets,
                      first_barrier=False) > 0


@pytest.mark.parametrize("world", [2, 3, 4])
def test_the_group_objects_mixed_calls_are_safe(world):
    """The group object's sequence: one- and two-shot calls mixed, two
    partials in turn, one-shot calls without the end barrier, one set of
    temporaries."""
    kinds = ["one_shot", "two_shot", "two_shot", "one_shot", "one_shot", "two_shot", "one_shot",
             "two_shot"]
    assert _races(world, len(kinds), kinds, partial_sets=2, temp_sets=1) == 0
    assert _races(world, len(kinds), kinds, partial_sets=1, temp_sets=1) > 0


def _replayed_one_shots(world, captured, replays, barrier_at_end):
    """The group object's one-shot calls captured once in a CUDA graph and
    replayed: the partial of each captured call is fixed at capture, so
    `captured` calls use partials 0, 1, 0, ... again on every replay."""
    progs = []
    for r in range(world):
        ev, k = [], 0
        for _ in range(replays):
            for i in range(captured):
                ev += _one_shot(r, world, k, i % 2, end_barrier=False)
                k += 1
            if barrier_at_end:
                ev += [("post", ("graph_end", k)), ("wait", ("graph_end", k))]
        progs.append(ev)
    return progs


@pytest.mark.parametrize("world", [2, 3])
def test_a_replayed_graph_needs_an_even_number_of_calls_or_a_final_barrier(world):
    rng = random.Random(1)

    def races(captured, barrier_at_end):
        progs = _replayed_one_shots(world, captured, 4, barrier_at_end)
        return sum(_run(progs, rng) is not None for _ in range(300))

    assert races(2, False) == 0 and races(4, False) == 0
    assert races(3, False) > 0          # the replay boundary reuses a partial back to back
    assert races(3, True) == 0
