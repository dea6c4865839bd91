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

A second model adds the rest of the kernel around the handoff: the weight ring, several
tiles per CTA and the read-back between them, with the issuing threads taking each
tile's quarters from t = 0 again. It checks the same rule for stale passes and for
deadlock, and shows that the issuing threads' wait for the previous tile's read-back is
needed where a tile's quarters are not a multiple of T.
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


def simulate_kernel(G, T, Q, n_q, nsteps, nt, S, seed, issuer_waits_readback=True, readback_lag=1):
    """The same handoff with the rest of the kernel around it: the weight ring (three
    producers, S stages, every decode group taking and releasing every K step), tiles
    of nsteps K steps (tq = nsteps * n_q quarters), the read-back at the end of each
    tile (every group waits for all of the tile's products, then arrives), and issuing
    thread t taking the quarters kq = t, t + T, ... of each tile -- so across a tile
    boundary a buffer can change hands when tq is not a multiple of T. Before its first
    quarter of tile lt >= 1 a thread waits for the read-back of tile lt - 1 (the kernel's
    acc_free); `issuer_waits_readback=False` drops that wait and `readback_lag=0` waits
    for the tile's own read-back instead (plausible mistakes). Returns (stale passes,
    deadlocked)."""
    rng = random.Random(seed)
    tq = nsteps * n_q
    steps_total = nt * nsteps
    full, free = [0] * Q, [0] * Q
    loaded = [False] * steps_total
    released = [0] * steps_total      # decode groups that released each K step
    consumed = [0] * nt               # quarters of each tile whose products are done
    readback = [0] * nt               # decode groups that read each tile back
    prod_next = list(range(3))        # producer w loads the steps w, w + 3, ...
    dec = [[0, 0] for _ in range(G)]  # each group: [K step, quarter within it (n_q: release, n_q + 1: read back)]
    iss = [[lt * tq + kq for lt in range(nt) for kq in range(t, tq, T)] for t in range(T)]
    iss_pos = [0] * T
    stale = 0

    def producer(w):
        g = prod_next[w]
        if g >= steps_total or (g >= S and released[g - S] < G):
            return False
        loaded[g] = True
        prod_next[w] += 3
        return True

    def decoder(gq):
        nonlocal stale
        st, q = dec[gq]
        if st >= steps_total or (q == 0 and not loaded[st]):
            return False
        if q < n_q:
            h = st * n_q + q
            if h % G == gq:
                j, k = h % Q, h // Q
                if k >= 1:
                    if (free[j] & 1) == ((k - 1) & 1):
                        return False
                    assert free[j] == k, "a decode group passed a release it did not wait for"
                full[j] += 1
            dec[gq][1] += 1
            return True
        if q == n_q:   # release the step's weight slot
            released[st] += 1
            if st % nsteps == nsteps - 1:
                dec[gq][1] += 1   # the tile's last step: its read-back next
            else:
                dec[gq] = [st + 1, 0]
            return True
        lt = st // nsteps   # read back: wait for all of the tile's products
        if consumed[lt] < tq:
            return False
        readback[lt] += 1
        dec[gq] = [st + 1, 0]
        return True

    def issuer(t):
        nonlocal stale
        if iss_pos[t] >= len(iss[t]):
            return False
        h = iss[t][iss_pos[t]]
        lt = h // tq
        first_of_tile = iss_pos[t] == 0 or iss[t][iss_pos[t] - 1] // tq != lt
        if issuer_waits_readback and first_of_tile and lt >= readback_lag and readback[lt - readback_lag] < G:
            return False
        j, k = h % Q, h // Q
        if (full[j] & 1) == (k & 1):
            return False
        if full[j] != k + 1:
            stale += 1
            return None
        free[j] += 1
        consumed[lt] += 1
        iss_pos[t] += 1
        return True

    actors = [(producer, w) for w in range(3)] + [(decoder, g) for g in range(G)] + \
             [(issuer, t) for t in range(T)]
    while True:
        order = actors[:]
        rng.shuffle(order)
        progressed = False
        for fn, a in order:
            r = fn(a)
            if r is None:
                return stale, False
            if r:
                progressed = True
                break
        if not progressed:
            done = all(p >= steps_total for p in prod_next) and all(d[0] >= steps_total for d in dec) and \
                all(iss_pos[t] >= len(iss[t]) for t in range(T))
            return stale, not done


# (n_q quarters per K step, T, Q, K steps per tile): NVFP4 (4 quarters) and FP8 (2), the
# planner's T = 4 / Q = 12 (N_pad <= 32) and T = 3 / Q = 9 or 6 (N_pad 48..96), with K
# steps per tile that make the tile's quarters a multiple of T or not
KERNEL_CASES = [(4, 4, 12, 5), (4, 3, 9, 5), (4, 3, 6, 7), (2, 4, 12, 3), (2, 3, 9, 5),
                (2, 3, 6, 4), (4, 3, 9, 3), (2, 4, 12, 4)]


@pytest.mark.parametrize("n_q,T,Q,nsteps", KERNEL_CASES)
@pytest.mark.parametrize("S", [3, 6, 12])
def test_kernel_handoff_across_tiles(n_q, T, Q, nsteps, S):
    """Several tiles per CTA with the weight ring and the read-back: no stale pass and
    no deadlock, whether or not a tile's quarters are a multiple of T."""
    assert Q == planner_buffers(3, T, Q)
    for seed in range(12):
        assert simulate_kernel(3, T, Q, n_q, nsteps, nt=3, S=S, seed=seed) == (0, False), (seed,)


@pytest.mark.parametrize("n_q,T,Q,nsteps", [(4, 3, 9, 5), (4, 3, 6, 7), (2, 3, 9, 5), (2, 3, 6, 4)])
def test_readback_wait_keeps_tile_boundaries_safe(n_q, T, Q, nsteps):
    """The planner's T = 3 plans (N_pad 48..96) with tiles whose quarters are not a
    multiple of 3: a tile's first quarters reuse buffers last used in the tile before
    by another thread, and the wait for that tile's read-back is what orders the two.
    Without it a thread can pass a stale phase."""
    assert (n_q * nsteps) % T and Q == planner_buffers(3, T, Q)
    assert any(simulate_kernel(3, T, Q, n_q, nsteps, nt=3, S=12, seed=seed,
                               issuer_waits_readback=False)[0] for seed in range(300))


def test_model_reports_a_deadlock():
    """The deadlock check is live: a thread that waits for its own tile's read-back
    (which needs that thread's products) stops the model."""
    assert simulate_kernel(3, 4, 12, 4, 5, nt=2, S=6, seed=0, readback_lag=0) == (0, True)
