"""The barrier protocol of the tensor-core FFN passes (csrc/ffn_tc.cu), as a randomised model.

Per pipeline stage the MMA issuer waits on one barrier of the activation ring: it completes
when the stage's activation copies have landed (one arrival with their byte count) and the
stage's dequantiser set (4 warps) has written the A operand.  A stage's A slot is free again
when the MMAs of the stage kKa earlier have completed; its activation slot when those of the
stage kB earlier have.  The model runs the roles in random orders and checks that every phase
of every activation barrier receives only its own stage's arrivals.  With an A ring at least as
deep as the activation ring (the down pass: kKa = 4, kB = 3) a dequantiser set can run ahead
far enough to arrive in the slot's previous, still open phase, unless it first waits for that
phase (the guard the kernel applies there); with kKa = 2 (gate/up) it cannot.
"""
import random

import pytest


def _run(kKa, kB, guard, stages=300, seed=0):
    rnd = random.Random(seed)

    class Bar:
        def __init__(self, count):
            self.count, self.done, self.open = count, 0, []

        def arrive(self, tag, w=1):
            self.open.append((tag, w))
            if sum(x[1] for x in self.open) >= self.count:
                tags = {x[0] for x in self.open}
                self.done += 1
                self.open = []
                return tags
            return None

    full = [Bar(1 + 4) for _ in range(kB)]
    empty_b = [Bar(1) for _ in range(kB)]
    empty_a = [Bar(1) for _ in range(kKa)]
    errors = []

    def arrive_full(slot, tag, w):
        phase = full[slot].done
        tags = full[slot].arrive(tag, w)
        if tags is not None and tags != {phase * kB + slot}:
            errors.append((slot, phase, tags))

    prod, deq, iss, pending = 0, [0, 1], 0, []
    while iss < stages:
        moves = []
        if prod < stages and (prod < kB or empty_b[prod % kB].done >= prod // kB):
            moves.append(("p", 0))
        for k in (0, 1):
            i = deq[k]
            if i < stages and (i < kKa or empty_a[i % kKa].done >= i // kKa):
                if not (guard and kKa >= kB and i >= kB and full[i % kB].done < i // kB):
                    moves.append(("d", k))
        if full[iss % kB].done > iss // kB:
            moves.append(("i", 0))
        if pending:
            moves.append(("m", 0))
        if not moves:
            errors.append(("deadlock", prod, tuple(deq), iss))
            break
        kind, k = rnd.choice(moves)
        if kind == "p":
            arrive_full(prod % kB, prod, 1)
            prod += 1
        elif kind == "i":
            pending.append(iss)
            iss += 1
        elif kind == "m":   # MMAs complete in issue order; their commits free both slots
            i = pending.pop(0)
            empty_b[i % kB].arrive(i)
            empty_a[i % kKa].arrive(i)
        else:
            i = deq[k]
            arrive_full(i % kB, i, 4)
            deq[k] += 2
    return errors


@pytest.mark.parametrize("kKa,kB", [(2, 3), (4, 3)])
def test_merged_stage_barrier_sees_only_its_stage(kKa, kB):
    for seed in range(200):
        assert _run(kKa, kB, guard=True, seed=seed) == [], f"seed {seed}"


def test_deep_a_ring_needs_the_guard():
    """Without the guard the down pass's geometry misplaces arrivals: the check has teeth."""
    assert any(_run(4, 3, guard=False, seed=s) for s in range(20))
    assert not any(_run(2, 3, guard=False, seed=s) for s in range(200))
