"""Plan changes between runs and the cross-run window, in the policy simulator.

Pinned to the pages' rules ("feat: prefetch streamed layers during compute", Summary:
"evicts residents from the end of the resident prefix", "releases stale residents and
prefetches when the graph plan changes"; "feat: pool VRAM for streamed layer", Summary:
"reuses a sufficiently large pool", "remembers reduced runtime caps"), to the budget
invariants and to the brute-force slot replay. No GPU.
"""
import random

import pytest

from oracle import brute
from oracle.policy import (ACTIVATE, EVICT, LOAD_RESIDENT, LOAD_SYNC, OK, PREFETCH,
                           WARN_MANDATORY_SLOT, plan_slots, simulate, simulate_script)

S = 100


def _ev(sim, run, kinds=None):
    return [e for e in sim.events if e[0] == run and (kinds is None or e[2] in kinds)]


def _between(sim, run):
    """Events of a run before its first step (plan-change releases, resident loads)."""
    return [(e[2], e[3], e[4]) for e in sim.events if e[0] == run and e[1] == -1]


@pytest.mark.parametrize("pool", [0, 1])
def test_shrink_releases_residents_from_the_end_of_the_prefix(pool):
    sim, st = simulate_script([S] * 6, depth=1, max_vram=5 * S, use_pool=pool,
                              script=[("run",), ("replan", 1, -1, 3 * S), ("run",)])
    assert st == [OK, OK, OK]
    assert (sim.plan.R, sim.plan.d, sim.plan.P) == (1, 1, 3)
    if pool:  # the pool changes from 5 to 3 slots: every slot empties, the kept prefix reloads
        assert _between(sim, 1) == [(EVICT, 2, 2), (EVICT, 1, 1), (EVICT, 0, 0), (LOAD_RESIDENT, 0, 0)]
    else:     # buffers of the kept residents stay
        assert _between(sim, 1) == [(EVICT, 2, 2), (EVICT, 1, 1)]
    assert sim.plan.shared_total + sim.plan.P * S <= 3 * S
    assert brute.replay(sim.events, 6, {0: 5, 1: 3}) == 5   # each run checked against its own pool


@pytest.mark.parametrize("pool", [0, 1])
def test_growth_loads_the_new_residents_at_the_next_run(pool):
    sim, st = simulate_script([S] * 6, depth=1, max_vram=3 * S, use_pool=pool,
                              script=[("run",), ("replan", 1, -1, 5 * S), ("run",), ("run",)])
    assert st == [OK, OK, OK, OK]
    assert sim.plan.R == 3
    if pool:
        assert _between(sim, 1) == [(EVICT, 0, 0)] + [(LOAD_RESIDENT, i, i) for i in range(3)]
    else:
        assert _between(sim, 1) == [(LOAD_RESIDENT, 1, 1), (LOAD_RESIDENT, 2, 2)]
    assert _between(sim, 2) == []          # residents persist
    assert brute.replay(sim.events, 6, {0: 3, 1: 5, 2: 5}) == 5


def test_same_slot_count_keeps_the_pool_and_the_kept_residents():
    # depth 1 -> 2 at 5 slots: R 3 -> 2, P stays 5: only resident 2 goes
    sim, st = simulate_script([S] * 8, depth=1, max_vram=5 * S, use_pool=1,
                              script=[("run",), ("replan", 2, -1, 5 * S), ("run",)])
    assert st == [OK, OK, OK]
    assert (sim.plan.R, sim.plan.d, sim.plan.P) == (2, 2, 5)
    assert _between(sim, 1) == [(EVICT, 2, 2)]
    assert sim.stats.pool_degradations == 0


def test_replan_to_the_same_controls_changes_nothing():
    sim, _ = simulate_script([S] * 6, depth=1, max_vram=4 * S, use_pool=1,
                             script=[("run",), ("replan", 1, -1, 4 * S), ("run",)])
    ref, _ = simulate([S] * 6, depth=1, max_vram=4 * S, use_pool=1, runs=2)
    assert sim.events == ref.events


def test_reduced_pool_cap_is_remembered():
    # the allocator holds 4 slots: registration degrades 5 -> 4; a larger budget later
    # plans for at most 4 slots and tries no bigger pool
    sim, st = simulate_script([S] * 8, depth=1, max_vram=5 * S, use_pool=1, alloc_cap=4 * S,
                              script=[("run",), ("replan", 1, -1, 8 * S), ("run",)])
    assert st == [OK, OK, OK]
    assert sim.slot_cap == 4 and sim.plan.P == 4
    assert sim.stats.pool_degradations == 1


def test_sync_fallback_is_remembered_across_a_replan():
    sim, st = simulate_script([S] * 6, depth=1, max_vram=6 * S, resident=0, use_pool=1,
                              fail_async=True, script=[("run",), ("replan", 3, 0, 6 * S), ("run",)])
    assert st[0] == 2  # WARN_SYNC_FALLBACK
    assert sim.d == 0
    assert not _ev(sim, 1, {PREFETCH})


def test_replan_below_one_slot_takes_the_mandatory_slot():
    sim, st = simulate_script([S] * 4, depth=1, max_vram=3 * S, use_pool=1,
                              script=[("run",), ("replan", 1, -1, S // 2), ("run",)])
    assert st == [OK, WARN_MANDATORY_SLOT, OK]
    assert (sim.plan.P, sim.plan.R, sim.plan.d) == (1, 0, 0)
    assert not _ev(sim, 1, {PREFETCH})


# ------------------------------------------------------------------ cross-run window
@pytest.mark.parametrize("N", [5, 6])
def test_cross_run_window_prefetches_the_next_runs_first_segment(N):
    sim, st = simulate([S] * N, depth=1, max_vram=2 * S, use_pool=1, runs=3, cross_run=True)
    assert st == [OK] * 3
    # run 0 issues its own N loads plus the next run's first
    pf0 = _ev(sim, 0, {PREFETCH})
    assert [e[3] for e in pf0] == list(range(N)) + [0]
    assert pf0[-1][1] == N - 1                  # from the last step's window
    for r in (1, 2):
        assert len(_ev(sim, r, {PREFETCH})) == N  # N - R per steady-state run, as without the window
        assert not _ev(sim, r, {LOAD_SYNC})
        first = _ev(sim, r, {ACTIVATE})[0]
        assert first[3] == 0 and first[4] == pf0[-1][4] if r == 1 else True
    # load numbers continue across runs: slots alternate without a break
    slots = [e[4] for e in sim.events if e[2] == ACTIVATE]
    assert slots == [j % 2 for j in range(3 * N)]
    assert brute.replay(sim.events, N, 2) == 2
    assert sim.stats.prefetch_activated == 3 * N


def test_cross_run_off_matches_the_run_boundary_rule():
    a, _ = simulate([S] * 6, depth=1, max_vram=2 * S, use_pool=1, runs=3)
    for r in range(3):
        assert _ev(a, r, {PREFETCH})[0][1] == 0   # every run's first prefetch at its own step 0


def test_cross_run_needs_a_full_ring():
    # 2 streamed segments, depth 3: the ring is 2 slots (< d + 1): the window stops at the run end
    sim, _ = simulate([S] * 4, depth=3, max_vram=4 * S, resident=2, use_pool=1, runs=2, cross_run=True)
    assert sim.plan.Q == 2 and not sim.carried
    assert [e[3] for e in _ev(sim, 0, {PREFETCH})] == [2, 3]


def test_replan_releases_stale_cross_run_prefetches():
    sim, st = simulate_script([S] * 6, depth=1, max_vram=2 * S, use_pool=1, cross_run=True,
                              script=[("run",), ("replan", 1, -1, 3 * S), ("run",)])
    assert st == [OK, OK, OK]
    carried = _ev(sim, 0, {PREFETCH})[-1]
    assert _between(sim, 1)[0] == (EVICT, carried[3], carried[4])
    assert brute.replay(sim.events, 6, {0: 2, 1: 3}) == 3


def test_pool_off_cross_run_loads_never_evict():
    # room for the ring only once resident 0 is gone: the next run's load is not issued early
    sim, _ = simulate([S] * 5, depth=1, max_vram=3 * S, use_pool=0, runs=2, cross_run=True,
                      alloc_cap=3 * S)
    assert not [e for e in sim.events if e[2] == EVICT]
    assert brute.replay(sim.events, 5, sim.plan.P) <= sim.plan.P


# ------------------------------------------------------------------ brute force
def test_random_scripts_replay_and_budgets():
    rng = random.Random(7)
    for _ in range(400):
        N = rng.randint(1, 7)
        sizes = [rng.choice([64, 100, 128]) for _ in range(N)]
        Smax = max(sizes)
        pool = rng.randint(0, 1)
        cross = rng.random() < 0.5
        cap = None if rng.random() < 0.6 else rng.randint(1, N + 2) * Smax
        def controls():
            return (rng.randint(0, N), rng.randint(-1, N), rng.choice([0, rng.randint(1, N + 2) * Smax,
                                                                        rng.randint(0, (N + 2) * Smax)]))
        d0, r0, b0 = controls()
        script = []
        for _ in range(rng.randint(1, 6)):
            script.append(("run",) if rng.random() < 0.6 else ("replan",) + controls())
        script.append(("run",))
        sim, st = simulate_script(sizes, depth=d0, resident=r0, max_vram=b0, use_pool=pool,
                                  script=script, alloc_cap=cap, cross_run=cross)
        if st and st[-1] < 0:
            continue
        # replay the same script step by step, recording the pool size each run used
        hist, r = {}, 0
        sim3, _ = simulate_script(sizes, depth=d0, resident=r0, max_vram=b0, use_pool=pool,
                                  script=[], alloc_cap=cap, cross_run=cross)
        for step in script:
            if step[0] == "run":
                hist[r] = sim3.plan.P if pool else N
                sim3.run_once()
                r += 1
            else:
                sim3.replan(*step[1:])
            p = sim3.plan
            if pool and not p.warn_mandatory and sim3.max_vram > 0:
                assert p.shared_total + p.P * p.S <= sim3.max_vram   # the budget bounds the pool
            cap_r = p.N if sim3.resident < 0 else min(sim3.resident, p.N)
            assert p.R <= cap_r or sim3.max_vram == 0   # budget 0: segmentation off, all resident
        assert sim3.events == sim.events
        brute.replay(sim.events, N, hist)
