"""The 32-token rings of the Q4_0 decode (range_body32 in csrc/fast_kernel.cuh)
as a protocol, checked on the CPU over random schedules.

The wph warps of a K/V head share S slots; warp sub reads tiles sub,
sub + wph, ...; tile t sits in slot t % S and the warp that has read tile t
issues tile t + S into the same slot.  Slot s has wph mbarriers used in turn:
tile t completes barrier (t % S, (t // S) % wph), and its reader waits on that
barrier for parity (t // (S * wph)) & 1.  An mbarrier parity wait succeeds
when the phase of that parity has completed -- which, if the barrier is two
phases behind, an older phase satisfies.  The model below plays the warps and
the copies in random order with exactly that wait rule and checks that every
successful wait finds its own tile in the slot, that no barrier takes a second
arrival before its phase completes, and that every schedule finishes.  The
single-barrier form (one barrier per slot, parity (t // S) & 1), which
faulted the GPU once, fails the same check."""
import random

import pytest


class Barrier:
    def __init__(self):
        self.completed = 0      # phases completed
        self.pending = False    # an arrival whose bytes have not all landed

    def ready(self, parity):
        # the wait of mbarrier.try_wait.parity: the phase of that parity is done
        return (self.completed & 1) != parity


def run_schedule(S, wph, n_tiles, rng, rotating=True):
    """One random interleaving; returns a list of violations (empty if none)."""
    bars = {}
    slot = [None] * S           # tile whose bytes the slot holds
    inflight = []               # copies issued and not landed: (barrier key, slot, tile)
    bad = []

    def key(t):
        return (t % S, (t // S) % wph) if rotating else (t % S, 0)

    def parity(t):
        return (t // (S * wph)) & 1 if rotating else (t // S) & 1

    def issue(t):
        b = bars.setdefault(key(t), Barrier())
        if b.pending:
            bad.append(("second arrival before the phase completed", t))
        b.pending = True
        inflight.append((key(t), t % S, t))

    for t in range(min(S, n_tiles)):
        issue(t)
    pos = [0] * wph             # next tile index of each warp
    mine = [list(range(w, n_tiles, wph)) for w in range(wph)]
    while True:
        moves = []
        if inflight:
            moves.append(("land", None))
        for w in range(wph):
            if pos[w] < len(mine[w]):
                t = mine[w][pos[w]]
                b = bars.get(key(t))
                if b is not None and b.ready(parity(t)):
                    moves.append(("read", w))
        if not moves:
            if any(pos[w] < len(mine[w]) for w in range(wph)):
                bad.append(("deadlock", pos[:]))
            return bad
        kind, w = rng.choice(moves)
        if kind == "land":
            k, s, t = inflight.pop(rng.randrange(len(inflight)))
            slot[s] = t
            bars[k].completed += 1
            bars[k].pending = False
        else:
            t = mine[w][pos[w]]
            if slot[t % S] != t:
                bad.append(("read the wrong tile", t, slot[t % S]))
            pos[w] += 1
            if t + S < n_tiles:
                issue(t + S)


@pytest.mark.parametrize("S,wph", [(5, 3), (5, 4), (4, 3), (2, 1), (7, 6), (9, 2)])
def test_rotating_barriers_hold_on_random_schedules(S, wph):
    rng = random.Random(1000 * S + wph)
    for trial in range(300):
        n_tiles = rng.randint(0, 8 * S * wph + 3)
        bad = run_schedule(S, wph, n_tiles, rng)
        assert not bad, (S, wph, n_tiles, trial, bad[:3])


def test_single_barrier_per_slot_fails_the_same_check():
    """The red control: one barrier per slot lets a warp meet the barrier
    still in another warp's phase, and some schedule shows it."""
    rng = random.Random(7)
    found = False
    for trial in range(2000):
        if run_schedule(5, 3, 60, rng, rotating=False):
            found = True
            break
    assert found


def test_one_warp_per_head_needs_no_rotation():
    """With one warp per head the two forms coincide (wph = 1)."""
    rng = random.Random(3)
    for _ in range(200):
        n = rng.randint(0, 40)
        assert not run_schedule(3, 1, n, rng, rotating=False)
        assert not run_schedule(3, 1, n, rng, rotating=True)
