"""The copy ring of the band kernels (csrc/gemvband.cu, csrc/w4band.cu), checked
on the CPU against the mbarrier parity semantics.

A consumer (an MMA warp; in the W4A16 kernel a pair of them, whose stage is
free once both have arrived) takes the stages ch = w, w + 4, ... (w = 0..3) and waits on the
stage's slot with `try_wait.parity((ch / stages) & 1)`, which succeeds as soon
as the phase *before* the barrier's current one has that parity; the copy
warp refills slot(ch) after waiting for the consumption of stage ch - stages.
The kernels map stage ch to slot (ch & 3) + 4 * ((ch >> 2) % (stages >> 2))
for 4 or 8 slots (each consumer warp owns its slots) and to slot ch when the
stages fit at once.  The model below runs random interleavings of the copy
warp, the copy engine and the four consumers and checks that every consumer
reads exactly the stage it waited for.  A shared mapping (slot ch % stages,
every warp on every slot) fails the same check.
"""
import random

import pytest


def owned_slot(ch, stages):
    return (ch & 3) + 4 * ((ch >> 2) % (stages >> 2)) if stages >= 4 else ch


def shared_slot(ch, stages):
    return ch % stages


def run_ring(nch, stages, slot_of, seed, consumers=4):
    """One random interleaving; raises AssertionError when a consumer's wait
    passes on a slot that does not hold its stage."""
    rnd = random.Random(seed)
    full = [0] * stages        # completed phases of each slot's FULL barrier
    empty = [0] * stages       # completed phases of each slot's EMPTY barrier (one arrival each)
    data = [None] * stages     # the stage whose copy last landed in the slot
    in_flight = {}             # slot -> stage being copied into it
    issued = 0
    nxt = list(range(consumers))
    consumed = set()
    for _ in range(100000):
        actions = []
        if issued < nch:
            actions.append("copy")
        if in_flight:
            actions.append("land")
        actions += [w for w in range(consumers) if nxt[w] < nch]
        if not actions:
            break
        a = rnd.choice(actions)
        if a == "copy":
            ch = issued
            s = slot_of(ch, stages)
            if ch >= stages:
                parity = ((ch // stages) - 1) & 1
                if (empty[s] & 1) == parity:       # wait: that phase has not completed
                    continue
                assert ch - stages in consumed, "refilled a slot whose stage is unread"
            assert s not in in_flight, "two copies into one slot"
            in_flight[s] = ch
            issued += 1
        elif a == "land":
            s = rnd.choice(sorted(in_flight))
            data[s] = in_flight.pop(s)
            full[s] += 1
        else:
            w = a
            ch = nxt[w]
            s = slot_of(ch, stages)
            parity = (ch // stages) & 1
            if (full[s] & 1) == parity:            # wait: that phase has not completed
                continue
            assert data[s] == ch and s not in in_flight, f"stage {ch} read from a slot holding {data[s]}"
            consumed.add(ch)
            empty[s] += 1
            nxt[w] += consumers
    assert len(consumed) == nch


@pytest.mark.parametrize("nch", list(range(1, 25)) + [40, 64])
def test_owned_slots_never_read_a_wrong_stage(nch):
    stages = 8 if nch > 4 else nch
    for seed in range(60):
        run_ring(nch, stages, owned_slot, seed)


def test_owned_slots_with_four_slots():
    for nch in (5, 9, 16, 33):
        for seed in range(60):
            run_ring(nch, 4, owned_slot, seed)


def test_a_shared_ring_is_caught():
    # six slots shared by all four consumers: some interleaving lets a consumer
    # pass a parity wait two phases behind
    failures = 0
    for seed in range(100):
        try:
            run_ring(16, 6, shared_slot, seed)
        except AssertionError:
            failures += 1
    assert failures > 0
