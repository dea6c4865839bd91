"""CPU model of the tcgen05 kernel's A-buffer handoff, checking the rule its planner
enforces (`plan_umma` in csrc/wq_umma.cu): Q A buffers are a multiple of the decode
groups and of the issuing threads T.

The protocol, as the kernel runs it:
- quarter h is decoded by group h mod G into buffer h mod Q; before it writes, the group
  waits for the buffer's previous quarter h - Q to be released (a_free);
- issuing thread h mod T waits for quarter h to be written (a_full), then releases the
  buffer after its products (a_free);
- groups and threads each take their own quarters in increasing order, and otherwise run
  freely.

An mbarrier wait in the kernel is a parity test: a waiter for the k-th completion of a
barrier passes when the barrier's completed count has the other parity from k -- that
is, when k + 1 phases are complete, but also when only k - 1 are (two behind). The
model runs random interleavings and records a "stale pass": an issuing thread that
passes its a_full test for quarter h while quarter h - Q, not h, is the last write of
its buffer. A plausible mistake in the rule (Q only >= T, or not a multiple of the
groups) shows stale passes; the planner's rule shows none.
"""
import math
import random

import pytest


def simulate(G, T, Q, quarters, seed, steps=200000):
    rng = random.Random(seed)
    full = [0] * Q    # a_full completions per buffer (one per quarter written)
    free = [0] * Q    # a_free completions per buffer (one per quarter consumed)
    next_dec = list(range(G))          # next quarter of each group
    next_iss = list(range(T))          # next quarter of each issuing thread
    stale = 0
    for _ in range(steps):
        actors = [("d", g) for g in range(G) if next_dec[g] < quarters] + \
                 [("i", t) for t in range(T) if next_iss[t] < quarters]
        if not actors:
            break
        kind, a = rng.choice(actors)
        if kind == "d":
            h = next_dec[a]
            j, k = h % Q, h // Q
            if k >= 1:   # wait for the (k-1)-th release of buffer j (parity test)
                if (free[j] & 1) == ((k - 1) & 1):
                    continue
                assert free[j] == k, "a decode group passed a release it did not wait for"
            full[j] += 1
            next_dec[a] += G
        else:
            h = next_iss[a]
            j, k = h % Q, h // Q
            if (full[j] & 1) == (k & 1):   # the k-th write of buffer j not complete (parity)
                continue
            if full[j] != k + 1:
                stale += 1                 # passed on the write of quarter h - Q
                # the kernel would now read the wrong A and release the buffer early;
                # stop this run here (what follows is undefined)
                break
            free[j] += 1
            next_iss[a] += T
    return stale


def planner_buffers(G, T, room):
    """Q as the planner picks it: the largest multiple of lcm(G, T) within the room."""
    l = G // math.gcd(G, T) * T
    return room // l * l


@pytest.mark.parametrize("T", [1, 2, 3, 4, 6])
@pytest.mark.parametrize("room", [6, 9, 12])
def test_planner_rule_never_passes_a_stale_phase(T, room):
    Q = planner_buffers(3, T, room)
    if Q == 0:
        pytest.skip("no buffer count of the rule fits this room")
    for seed in range(40):
        assert simulate(3, T, Q, quarters=240, seed=seed) == 0, (T, Q, seed)


@pytest.mark.parametrize("T,Q", [(7, 9), (4, 6), (4, 9), (5, 6)])
def test_weaker_rules_can_pass_a_stale_phase(T, Q):
    """Q >= T alone (the rule before the fix) lets a thread meet a buffer two phases
    behind once the groups drift: 7 threads with 9 buffers is the variant that timed out
    on the GPU; 4 with 6 or 9 the default plan's former choice at N_pad = 48..80."""
    assert any(simulate(3, T, Q, quarters=240, seed=seed) for seed in range(200)), (T, Q)
