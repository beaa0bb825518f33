"""Model check of the CTA-pair operand-ring drain of the GEMM kernel (gemm.cuh, drain_pair_ring).

In a CTA pair both producers copy their halves of ring use j (stage j % S) into their own shared
memory, and both copies complete on the leader's "full" barrier of that stage, which the leader arms
for both CTAs' bytes.  After an abort the two producers may have issued different numbers of uses;
the leader then balances, per stage, the bytes of the last use below max(own, peer) and waits for its
phase, so that no copy of either CTA is still in flight when the pair leaves.  The device code can
only take this path after a 2-second wait has expired, so it is checked here instead: a model of the
mbarrier (phase count, pending arrivals, transaction count) runs random interleavings of the two
producers, the MMA consumer and copy completions, stops them at random points, applies the drain
rule exactly as the kernel computes it, and requires every wait it performs to be one that completes
and every copy to have landed in a phase the drain waited for."""
import random

import pytest


class Barrier:
    """An mbarrier with one expected arrival per phase and a transaction count."""

    def __init__(self):
        self.phase = 0       # completed phases
        self.pending = 1     # arrivals still expected in the current phase
        self.tx = 0          # expected bytes minus arrived bytes in the current phase

    def _maybe_complete(self):
        if self.pending == 0 and self.tx == 0:
            self.phase += 1
            self.pending, self.tx = 1, 0

    def arrive_expect_tx(self, nbytes):
        self.tx += nbytes
        self.pending -= 1
        assert self.pending >= 0, "more arrivals than the barrier counts"
        self._maybe_complete()

    def complete_tx(self, nbytes):
        self.tx -= nbytes
        self._maybe_complete()

    def done(self, parity):
        """try_wait.parity: the phase with this parity has completed (current phase parity differs)."""
        return (self.phase & 1) != parity


def drain_rule(S, own, peer):
    """The kernel's per-stage decisions: (stage, use j, action, parity waited)."""
    end = max(own, peer)
    out = []
    for s in range(min(S, end)):
        j = s + (end - 1 - s) // S * S
        by_own, by_peer = j < own, j < peer
        action = "balance_peer" if (by_own and not by_peer) else ("arm_peer" if (by_peer and not by_own) else None)
        out.append((s, j, action, (j // S) & 1))
    return out


def simulate(seed, S=6, total=40, B=100):
    rng = random.Random(seed)
    bars = [Barrier() for _ in range(S)]
    own = peer = consumed = 0
    in_flight = []           # (use j, which CTA) copies issued and not landed
    landed_phase = []        # (stage, phase index of the use, which CTA) for every copy
    stop_own = rng.randint(0, total)
    stop_peer = rng.randint(0, total)
    stop_mma = rng.randint(0, total)

    def can_issue(j):
        return j < total and j - S < consumed   # the stage's previous use was consumed

    for _ in range(20 * total):
        moves = []
        if own < stop_own and can_issue(own):
            moves.append("own")
        if peer < stop_peer and can_issue(peer):
            moves.append("peer")
        if consumed < stop_mma and consumed < total and bars[consumed % S].done((consumed // S) & 1):
            moves.append("mma")
        if in_flight:
            moves.append("land")
        if not moves:
            break
        m = rng.choice(moves)
        if m == "own":
            bars[own % S].arrive_expect_tx(2 * B)   # the leader arms both CTAs' bytes
            in_flight.append((own, "own"))
            own += 1
        elif m == "peer":
            in_flight.append((peer, "peer"))
            peer += 1
        elif m == "mma":
            consumed += 1
        else:
            j, who = in_flight.pop(rng.randrange(len(in_flight)))
            # a copy of use j lands in the current phase of its stage, which must be use j's phase
            assert bars[j % S].phase == j // S, "a copy landed in another use's phase"
            landed_phase.append((j % S, j // S, who))
            bars[j % S].complete_tx(B)
    # the producers stopped; copies still in flight land eventually (the hardware completes them)
    for j, who in in_flight:
        assert bars[j % S].phase == j // S
        landed_phase.append((j % S, j // S, who))
        bars[j % S].complete_tx(B)
    # invariants the drain relies on
    assert min(own, peer) >= consumed and max(own, peer) <= consumed + S
    waited = {}
    for s, j, action, parity in drain_rule(S, own, peer):
        if action == "balance_peer":
            bars[s].complete_tx(B)
        elif action == "arm_peer":
            bars[s].arrive_expect_tx(B)
        assert bars[s].done(parity), f"seed {seed}: the drain would wait for a phase that never completes"
        waited[s] = j // S
    # every copy landed in a phase at or before the one the drain waited for on its stage, and no
    # stage is left with arrivals or bytes outstanding
    for s, ph, who in landed_phase:
        assert s in waited and ph <= waited[s]
    for b in bars:
        assert b.pending == 1 and b.tx == 0
    return own, peer, consumed


@pytest.mark.parametrize("S", [5, 6])
def test_drain_balances_and_completes_every_stage(S):
    seen = set()
    for seed in range(3000):
        own, peer, consumed = simulate(seed, S=S)
        seen.add((own > peer, own < peer, own == peer))
    # the random stops covered the leader ahead, the peer ahead and both equal
    assert len(seen) == 3


def test_drain_rule_matches_hand_cases():
    # leader issued uses 0..7, peer 0..9, S = 6: stages 0-3 end at uses 6-9 (4, 5 at uses 4, 5)
    r = {s: (j, a, p) for s, j, a, p in drain_rule(6, 8, 10)}
    assert r[0] == (6, None, 1) and r[1] == (7, None, 1)
    assert r[2] == (8, "arm_peer", 1) and r[3] == (9, "arm_peer", 1)
    assert r[4] == (4, None, 0) and r[5] == (5, None, 0)
    # peer behind: the leader's uses 3, 4 lack the peer's bytes
    r = {s: (j, a, p) for s, j, a, p in drain_rule(6, 5, 3)}
    assert r[3] == (3, "balance_peer", 0) and r[4] == (4, "balance_peer", 0) and 5 not in r
    # nothing issued: nothing to wait for
    assert drain_rule(6, 0, 0) == []
