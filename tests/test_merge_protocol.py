"""The cooperative in-launch merge of the fast decode kernel (merge_coop in
csrc/fast_kernel.cuh) as a protocol, checked on the CPU over random
interleavings of its atomic steps.

The na CTAs of a sequence share three counter words.  Each CTA adds 1 to
word 0 when its partial is written.  The CTA that completes the count reads
word 1 (the give-up bits) and merges its own rows and those of every CTA whose
bit it sees.  Every other CTA waits for the count; if its bounded wait runs
out it sets its bit in word 1 and reads word 0 once more, merging its own rows
only if the count completed meanwhile.  After its reads of words 0 and 1 each
CTA adds 1 to word 2, and the CTA that completes that count resets the three
words for the next launch.  The model checks, for every schedule (with waits
that run out at random), that each partition's rows are merged at least once
and only after every partial is in, that no CTA touches words 0 and 1 after
the reset, and that the words end at zero.  Without the second read of word 0
after a give-up, a partition can be lost, and the check shows it."""
import random

import pytest


def run_schedule(na, rng, recheck=True, p_timeout=0.3):
    w = [0, 0, 0]
    arrived = 0                  # partials written (word 0's true count)
    merged = [0] * na
    bad = []
    reset_done = False
    # per CTA: a generator of atomic steps
    def cta(j):
        nonlocal arrived, reset_done
        yield
        arrived += 1
        old = w[0]
        w[0] += 1
        if reset_done:
            bad.append(("word 0 after the reset", j))
        if old + 1 == na:
            yield
            merge_set = (1 << j) | w[1]
        else:
            merge_set = 0
            while True:
                yield
                if w[0] >= na:
                    merge_set = 1 << j
                    break
                yield  # the clock check: the wait may run out now
                if rng.random() < p_timeout:
                    w[1] |= 1 << j
                    yield
                    if recheck and w[0] >= na:
                        merge_set = 1 << j
                    break
        if reset_done:
            bad.append(("words 0/1 read after the reset", j))
        # the done count (word 2), then the merge of the set's rows
        yield
        old2 = w[2]
        w[2] += 1
        if old2 + 1 == na:
            w[0] = w[1] = w[2] = 0
            reset_done = True
        for k in range(na):
            if merge_set >> k & 1:
                yield
                if arrived < na:
                    bad.append(("merged before every partial was in", j, k))
                merged[k] += 1

    procs = {j: cta(j) for j in range(na)}
    while procs:
        j = rng.choice(list(procs))
        try:
            next(procs[j])
        except StopIteration:
            del procs[j]
    lost = [k for k in range(na) if merged[k] == 0]
    if lost:
        bad.append(("partitions never merged", lost))
    if w != [0, 0, 0]:
        bad.append(("words not reset", w))
    return bad


@pytest.mark.parametrize("na", [1, 2, 3, 5, 19, 32])
def test_every_partition_is_merged_once_all_are_in(na):
    rng = random.Random(na)
    for trial in range(400):
        bad = run_schedule(na, rng, p_timeout=rng.choice([0.0, 0.05, 0.5, 1.0]))
        assert not bad, (na, trial, bad[:3])


def test_a_give_up_without_the_second_read_loses_rows():
    """The red control: a CTA that gives up and does not read the count again
    may miss the completion, and the completing CTA may have read word 1 before
    the give-up bit was set."""
    rng = random.Random(11)
    assert any(run_schedule(3, rng, recheck=False, p_timeout=0.5) for _ in range(3000))
