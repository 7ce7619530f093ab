"""A model of the fused merge's arrival-counter protocol (the tcgen05 row kernel), run on the CPU
under random interleavings of the chunk CTAs, including CTAs whose wait gives up.

Protocol, per (group, KV head) counter shared by the group's n chunk CTAs:
  1. store the CTA's records, then count in (+1);
  2. poll the counter up to `spin` times for a value >= n ("all records are stored");
  3. count in a second time, whatever step 2 found; the CTA whose second count-in returns
     2 n - 1 (the last of the 2 n increments) writes 0 back.
What must hold: the counter is 0 after every call, whatever gave up; and when no wait gave up,
no CTA passed step 2 before every CTA had stored its records.
"""

import random


def _run_call(n, spin, rng, cnt=0):
    """One call's n CTAs interleaved at random; returns (final counter, passed, early)."""
    state = [("store", 0) for _ in range(n)]  # (step, polls used)
    stored = [False] * n
    passed = [False] * n
    early = False
    live = list(range(n))
    while live:
        c = rng.choice(live)
        step, polls = state[c]
        if step == "store":
            stored[c] = True
            cnt += 1
            state[c] = ("poll", 0)
        elif step == "poll":
            if polls < spin and cnt >= n:
                passed[c] = True
                early |= not all(stored)
                state[c] = ("second", 0)
            elif polls >= spin:
                state[c] = ("second", 0)  # gave up
            else:
                state[c] = ("poll", polls + 1)
        else:  # second count-in
            old = cnt
            cnt += 1
            if old == 2 * n - 1:
                cnt = 0
            live.remove(c)
    return cnt, passed, early


def test_counter_returns_to_zero_under_any_timeout_pattern():
    rng = random.Random(7)
    for trial in range(3000):
        n = rng.randint(1, 24)
        spin = rng.choice([0, 1, 2, 5, 50, 10 ** 6])
        cnt, passed, early = _run_call(n, spin, rng)
        assert cnt == 0, (trial, n, spin, cnt)
        if all(passed):
            assert not early, (trial, n, spin)


def test_calls_in_sequence_never_see_a_stale_counter():
    """Calls on one workspace run one after another (stream order): a call after a timed-out one
    starts from zero, so its CTAs wait for all of its own records."""
    rng = random.Random(11)
    cnt = 0
    for call in range(500):
        n = rng.randint(1, 20)
        spin = rng.choice([0, 3, 10 ** 6])
        cnt, passed, early = _run_call(n, spin, rng, cnt)
        assert cnt == 0
        if spin == 10 ** 6:
            assert all(passed) and not early, call


def test_a_cta_that_skips_its_second_count_in_would_leave_the_counter_set():
    """Why step 3 is unconditional: the earlier protocol counted in a second time only after a
    successful wait, and one CTA that gave up left the counter part-way for the next call."""
    n = 4
    cnt = 0
    for c in range(n):
        cnt += 1  # every CTA stores and counts in
    # CTAs 0..2 see cnt >= n and count in again; CTA 3 gave up before seeing it (old protocol:
    # no second count-in)
    for c in range(3):
        old = cnt
        cnt += 1
        if old == 2 * n - 1:
            cnt = 0
    assert cnt == 2 * n - 1  # never reset: the next call's first CTA would see >= n at once
