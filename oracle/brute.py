"""Brute-force checks that pin the policy simulator (oracle; test infrastructure only).

``brute_plan`` enumerates every (depth, residents) pair that respects the
budget, the requested depth and the resident cap, and picks the lexicographic
maximum by (depth, residents): the prefetch window has priority over optional
residents ("feat: prefetch streamed layers during compute", Summary, first
bullet; "feat: pool VRAM for streamed layer", Summary, second bullet).

``replay`` walks an event list slot by slot and checks what the pages require
of any schedule: a load only lands in a free slot, every activation finds its
segment in its slot, the active segment is never evicted, residents keep their
slot across runs, and the number of slots ever occupied at once never exceeds
the pool ("allocates only the peak slot count", "feat: pool VRAM for streamed
layer", Summary). It returns the peak occupancy, which must equal P.
"""
from __future__ import annotations

from .policy import ACTIVATE, EVICT, LOAD_RESIDENT, LOAD_SYNC, PREFETCH, SHARED_LOAD


def brute_plan(N: int, S: int, shared_total: int, depth: int, resident: int, max_vram: int):
    """Return (depth, residents, mandatory) chosen by exhaustive search."""
    if max_vram == 0:
        return 0, N, False
    cap = N if resident < 0 else min(resident, N)
    room = max_vram - shared_total
    best = None
    for dp in range(depth + 1):
        for rp in range(cap + 1):
            streamed = N - rp
            ring = min(dp + 1, streamed) if streamed > 0 else 0
            if (rp + ring) * S <= room:
                if best is None or (dp, rp) > best:
                    best = (dp, rp)
    if best is None:
        return 0, 0, True
    return best[0], best[1], False


def replay(events: list, n_segments: int, n_slots) -> int:
    """Check slot ownership along the schedule; return the peak occupied slots.

    ``n_slots`` is the pool size, or {run: pool size} when the plan changes between
    runs. A streamed load may be activated in a later run (cross-run window); such a
    load, and any resident, may be released at a plan change (EVICT at step -1)."""
    owner: dict = {}
    residents: set = set()
    pending: set = set()          # loaded, not yet activated (may cross a run boundary)
    peak = 0
    by_run: dict = {}
    for ev in events:
        by_run.setdefault(ev[0], []).append(ev)
    for run in sorted(by_run):
        slots = n_slots[run] if isinstance(n_slots, dict) else n_slots
        activated = []
        run_peak = 0
        for (_, step, kind, seg, slot, _nb) in by_run[run]:
            if kind == SHARED_LOAD:
                assert slot == -1
                continue
            # a release at a plan change names a slot of the pool before the change
            if not (kind == EVICT and step == -1):
                assert 0 <= slot < slots, f"slot {slot} outside the pool of {slots}"
            if kind == LOAD_RESIDENT:
                assert slot not in owner, f"resident {seg} lands on occupied slot {slot}"
                assert step == -1, "residents load before the run's first step"
                owner[slot] = seg
                residents.add(seg)
            elif kind in (PREFETCH, LOAD_SYNC):
                assert seg not in residents, f"resident {seg} loaded again"
                assert seg not in pending, f"{seg} loaded twice before its activation"
                assert slot not in owner, \
                    f"run {run} step {step}: load of {seg} overwrites slot {slot} held by {owner[slot]}"
                owner[slot] = seg
                pending.add(seg)
            elif kind == EVICT:
                assert owner.get(slot) == seg, f"evict {seg} finds slot {slot} holding {owner.get(slot)}"
                if seg in residents:
                    # the segment active at step k is k: only ones computed earlier may go
                    assert step == -1 or seg < step, "evicted the active segment or one not yet computed"
                    residents.discard(seg)
                else:
                    assert seg in pending and step == -1, "only a stale prefetch is released, between runs"
                    pending.discard(seg)
                del owner[slot]
            elif kind == ACTIVATE:
                assert owner.get(slot) == seg, f"activate {seg} finds slot {slot} holding {owner.get(slot)}"
                assert seg in residents or seg in pending
                activated.append(seg)
            if not (kind == EVICT and step == -1):   # occupancy once the plan change is done
                run_peak = max(run_peak, len(owner))
            if kind == ACTIVATE and seg not in residents:
                pending.discard(seg)
                del owner[slot]          # a streamed slot is free once its segment computed
        assert run_peak <= slots
        peak = max(peak, run_peak)
        assert activated == list(range(len(activated))), "segments activate in order"
    return peak


def check_window(events: list, n_segments: int, R: int, d: int, cross_run: bool = False) -> None:
    """Check the prefetch window along a schedule without failures, run by run.

    What the pages fix for any schedule ("feat: prefetch streamed layers during compute",
    Summary: the next d segments are loaded while the active one computes; depth 0 is
    synchronous streaming):
      * each streamed segment (index >= R) is loaded exactly once per run, before its
        activation, by a PREFETCH or LOAD_SYNC of this run or (cross-run window) by a
        PREFETCH of the run before, issued after that run had activated the segment;
      * residents are never loaded during a run;
      * when segment k activates, the streamed segments loaded and not yet activated,
        k excluded, number min(d, streamed segments after k): the window is full but
        never reaches past the run. With a cross-run window on a full ring (N - R > d)
        the next run's first segments count too, so the number is d at every step.
    The window here is not computed the simulator's way: it is counted from the events."""
    M = n_segments - R
    crossing = cross_run and M > d
    by_run: dict = {}
    for ev in events:
        by_run.setdefault(ev[0], []).append(ev)
    ahead: set = set()                 # loaded for this run, not yet activated
    for run in sorted(by_run):
        nxt: set = set()               # loaded in this run for the next run
        done: set = set()
        loads: dict = {s: 0 for s in ahead}
        for (_, step, kind, seg, slot, _nb) in by_run[run]:
            if kind in (PREFETCH, LOAD_SYNC):
                assert seg >= R, f"run {run}: resident {seg} loaded during the run"
                if seg in done:
                    assert cross_run and kind == PREFETCH, f"run {run}: {seg} loaded after its activation"
                    assert seg not in nxt, f"run {run}: {seg} loaded twice for the next run"
                    nxt.add(seg)
                else:
                    loads[seg] = loads.get(seg, 0) + 1
                    assert loads[seg] == 1, f"run {run}: {seg} loaded twice"
                    ahead.add(seg)
            elif kind == ACTIVATE:
                k = seg
                assert k == step and k == len(done), "segments activate in order"
                if k >= R:
                    assert k in ahead, f"run {run}: streamed segment {k} activated without a load"
                    ahead.discard(k)
                want = min(d, M if k < R else n_segments - 1 - k)
                if crossing:
                    want = d
                got = len(ahead) + len(nxt)
                assert got == want, f"run {run} step {k}: {got} loads ahead of the active segment, want {want}"
                done.add(k)
        assert len(done) == n_segments
        assert not ahead, f"run {run}: loads never activated: {sorted(ahead)}"
        ahead = nxt
