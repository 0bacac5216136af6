"""The policy simulator against the pages' tables, worked numbers, invariants and
brute force."""
import itertools
import os

import numpy as np
import pytest

from oracle import brute
from oracle import policy as pol

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    out = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            left, right = line.split("|")
            exp = dict(kv.split("=") for kv in right.split())
            out.append((left.split(), {k: float(v) for k, v in exp.items()}))
    return out


def _kinds(sim, run, kind):
    return [e for e in sim.events if e[0] == run and e[2] == kind]


def _check_plan_fields(sim, exp):
    """R and d as they stand after the runs (fallback and eviction lower them),
    P and S as planned."""
    p = sim.plan
    for key, val in exp.items():
        if key == "R":
            assert sim.R == val, (key, p)
        elif key == "d":
            assert min(sim.d, p.N - sim.R) == val, (key, p, sim.d)
        elif key == "P":
            assert p.P == val, (key, p)
        elif key == "S":
            assert p.S == val, (key, p)


@pytest.mark.parametrize("row", _rows("sd1905_effective_behavior.txt"), ids=lambda r: r[0][0])
def test_sd1905_effective_behavior(row):
    (name, N, depth, resident, budget), exp = row
    S = 1000
    sim, st = pol.simulate([S] * int(N), [], int(depth), int(resident), int(float(budget) * S),
                           use_pool=1, runs=2)
    assert all(s >= 0 for s in st)
    _check_plan_fields(sim, exp)
    assert len(_kinds(sim, 0, pol.PREFETCH)) == exp["prefetch"]
    assert len(_kinds(sim, 0, pol.LOAD_SYNC)) == exp["sync"]
    if exp["d"] == 0:
        # depth 0 is plain synchronous streaming: no prefetch at all, in any run
        assert not [e for e in sim.events if e[2] == pol.PREFETCH]
    assert brute.replay(sim.events, int(N), sim.plan.P) == sim.plan.P


@pytest.mark.parametrize("row", _rows("sd1906_pool_behavior.txt"), ids=lambda r: r[0][0])
def test_sd1906_pool_behavior(row):
    (name, pool, depth, resident, budget, cap, fail_async), exp = row
    S, N = 1000, 6
    alloc_cap = None if cap == "-" else int(float(cap) * S)
    sim, st = pol.simulate([S] * N, [], int(depth), int(resident), int(float(budget) * S),
                           use_pool=int(pool), runs=2, alloc_cap=alloc_cap,
                           fail_async=bool(int(fail_async)))
    if exp["status"] < 0:
        assert st == [int(exp["status"])]
        return
    first = sim.status if sim.status != 0 else st[0]
    assert first == exp["status"], (sim.status, st)
    _check_plan_fields(sim, exp)
    if "degradations" in exp:
        assert sim.stats.pool_degradations == exp["degradations"]
    if "prefetch" in exp:
        assert len(_kinds(sim, 0, pol.PREFETCH)) == exp["prefetch"]
        assert len(_kinds(sim, 0, pol.LOAD_SYNC)) == exp["sync"]
    if exp.get("alternate"):
        for run in (0, 1):
            slots = [e[4] for e in _kinds(sim, run, pol.ACTIVATE)]
            assert slots == [i % 2 for i in range(N)]
    if exp.get("same_as_pool"):
        ref, _ = pol.simulate([S] * N, [], int(depth), int(resident), int(float(budget) * S),
                              use_pool=1, runs=2)
        assert ref.events == sim.events
    assert brute.replay(sim.events, N, sim.plan.P) <= sim.plan.P


@pytest.mark.parametrize("row", _rows("worked_numbers.txt"), ids=lambda r: r[0][0])
def test_worked_numbers(row):
    (name, N, S, budget, depth, resident), exp = row
    sim, st = pol.simulate([int(S)] * int(N), [], int(depth), int(resident), int(budget),
                           use_pool=1, runs=1)
    _check_plan_fields(sim, exp)
    if "prefetch" in exp:
        assert sim.stats.prefetch_queued == exp["prefetch"]
        assert sim.stats.prefetch_activated == exp["activated"]
    if "status" in exp:
        assert sim.status == exp["status"]
    if "pool_bytes" in exp:
        assert sim.plan.P * sim.plan.S == exp["pool_bytes"]


def _grid():
    sizes = ([100] * 5, [100, 60, 100, 40], [80, 100, 100, 100, 20, 100], [100])
    for seg, depth, resident, budget, pool in itertools.product(
            sizes, range(0, 5), range(-1, 6), (0, 50, 100, 150, 200, 300, 450, 700), (0, 1)):
        if resident > len(seg):
            continue
        yield seg, depth, resident, budget, pool


def test_invariants_and_brute_force_grid():
    n = 0
    for seg, depth, resident, budget, pool in _grid():
        for shared in ([], [(7, 30)]):
            sh_total = sum(pol.align_up(b) for _, b in shared)
            sim, st = pol.simulate(seg, shared, depth, resident, budget, use_pool=pool, runs=2)
            p = sim.plan
            N, S = len(seg), max(seg)
            # exhaustive choice of (depth, residents), depth first
            bd, br, mand = brute.brute_plan(N, S, sh_total, depth, resident, budget)
            assert (p.d_req, p.R) == (bd, br), (seg, depth, resident, budget, p, (bd, br))
            assert p.warn_mandatory == mand
            # the positive budget is never exceeded, except by the one mandatory slot
            if budget > 0:
                if mand:
                    assert p.P == 1 and p.d == 0 and p.R == 0
                else:
                    assert sh_total + p.P * S <= budget
            # the resident prefix respects its cap (max-vram 0 turns segmentation off)
            if budget > 0:
                assert p.R <= (N if resident < 0 else resident)
            # P is exactly the peak number of occupied slots
            assert brute.replay(sim.events, N, p.P) == p.P
            # depth 0 is synchronous streaming
            if p.d == 0:
                assert all(e[2] != pol.PREFETCH for e in sim.events)
            # resident 0 / depth 1 alternates two slots
            if p.R == 0 and p.d == 1 and N >= 2:
                acts = [e[4] for e in sim.events if e[2] == pol.ACTIVATE and e[0] == 1]
                assert acts == [i % 2 for i in range(N)]
            # every streamed segment is queued once per run when d >= 1
            if p.d >= 1:
                assert len(_kinds(sim, 1, pol.PREFETCH)) == N - p.R
            # the window, counted from the events: full, never past the run
            brute.check_window(sim.events, N, p.R, p.d)
            n += 1
    assert n > 1000


def test_window_counted_from_the_events_grid():
    """Every plan of up to 7 segments, with and without the cross-run window: each streamed
    segment is loaded once per run before its activation, and the loads ahead of the active
    segment number min(d, streamed segments left), or d across the run boundary."""
    n = 0
    for N in range(1, 8):
        for depth, resident, slots, cross, pool in itertools.product(
                range(0, 6), range(-1, N + 1), range(1, N + 3), (False, True), (0, 1)):
            sim, st = pol.simulate([100] * N, [], depth, resident, slots * 100, use_pool=pool, runs=3,
                                   cross_run=cross)
            assert all(s >= 0 for s in st)
            p = sim.plan
            brute.check_window(sim.events, N, p.R, p.d, cross)
            assert brute.replay(sim.events, N, p.P) == p.P
            n += 1
    assert n > 6000


def test_window_worked_example():
    """N = 6, two residents, depth 2 (a hand-worked schedule): loads 0 and 1 of the ring
    (segments 2 and 3) are issued at step 0, in the resident prefix; segment 4 enters the
    window when segment 2 activates (step 2), segment 5 at step 3; the ring of three slots
    2, 3, 4 is taken in turn."""
    sim, st = pol.simulate([100] * 6, [], depth=2, resident=2, max_vram=500, use_pool=1, runs=1)
    assert (sim.plan.R, sim.plan.d, sim.plan.Q, sim.plan.P) == (2, 2, 3, 5)
    got = [(e[1], pol.KIND_NAMES[e[2]], e[3], e[4]) for e in sim.events]
    assert got == [
        (-1, "LOAD_RESIDENT", 0, 0), (-1, "LOAD_RESIDENT", 1, 1),
        (0, "PREFETCH", 2, 2), (0, "PREFETCH", 3, 3), (0, "ACTIVATE", 0, 0),
        (1, "ACTIVATE", 1, 1),
        (2, "PREFETCH", 4, 4), (2, "ACTIVATE", 2, 2),
        (3, "PREFETCH", 5, 2), (3, "ACTIVATE", 3, 3),
        (4, "ACTIVATE", 4, 4),
        (5, "ACTIVATE", 5, 2)]


def test_runtime_pressure_evicts_from_the_end_of_the_prefix():
    """Pool off: a prefetch that does not fit evicts the last resident already
    computed, never the active one; when nothing can go, streaming turns
    synchronous and stays so."""
    seg = [100] * 6
    # 3 residents + the active streamed segment fill the 400-byte cap: the prefetch
    # issued at step 3 must evict resident 2 (computed at step 2)
    sim, st = pol.simulate(seg, [], depth=1, resident=3, max_vram=1000, use_pool=0, runs=3,
                           alloc_cap=400)
    ev = [e for e in sim.events if e[2] == pol.EVICT]
    assert ev, sim.events
    for (_, step, _, s, slot, _) in ev:
        assert s < step
    assert [e[3] for e in ev] == sorted([e[3] for e in ev], reverse=True)
    brute.replay(sim.events, 6, sim.plan.P)
    # nothing evictable at step 0 of run 0: prefetch of segment 3 with 3 residents live
    sim2, st2 = pol.simulate(seg, [], depth=1, resident=3, max_vram=1000, use_pool=0, runs=2,
                             alloc_cap=300)
    assert st2[0] == pol.WARN_SYNC_FALLBACK
    assert all(e[2] != pol.PREFETCH for e in sim2.events if e[0] == 1)


def test_run_boundary_and_residents_persist():
    sim, _ = pol.simulate([100] * 5, [(3, 64), (1, 10)], depth=2, resident=2, max_vram=10_000,
                          runs=3)
    kinds0 = [e[2] for e in sim.events if e[0] == 0]
    assert kinds0[:2] == [pol.SHARED_LOAD, pol.SHARED_LOAD]
    assert [e[3] for e in sim.events if e[2] == pol.SHARED_LOAD] == [1, 3]
    assert [e[3] for e in sim.events if e[2] == pol.LOAD_RESIDENT] == [0, 1]
    for run in (1, 2):
        kinds = [e[2] for e in sim.events if e[0] == run]
        assert pol.SHARED_LOAD not in kinds and pol.LOAD_RESIDENT not in kinds
    # the window starts afresh in each run: run r's first prefetch is issued at step 0
    for run in range(3):
        first = [e for e in sim.events if e[0] == run and e[2] == pol.PREFETCH][0]
        assert first[1] == 0 and first[3] == 2
