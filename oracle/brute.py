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


def replay(events: list, n_segments: int, n_slots: int) -> int:
    """Check slot ownership along the schedule; return the peak occupied slots."""
    owner: dict = {}
    residents: set = set()
    peak = 0
    by_run: dict = {}
    for ev in events:
        by_run.setdefault(ev[0], []).append(ev)
    for run in sorted(by_run):
        activated = []
        loaded_this_run = set()
        for (_, step, kind, seg, slot, _nb) in by_run[run]:
            if kind == SHARED_LOAD:
                assert slot == -1
                continue
            assert 0 <= slot < n_slots, f"slot {slot} outside the pool of {n_slots}"
            if kind == LOAD_RESIDENT:
                assert slot not in owner, f"resident {seg} lands on occupied slot {slot}"
                owner[slot] = seg
                residents.add(seg)
                loaded_this_run.add(seg)
            elif kind in (PREFETCH, LOAD_SYNC):
                assert seg not in residents, f"resident {seg} loaded again"
                assert slot not in owner, \
                    f"run {run} step {step}: load of {seg} overwrites slot {slot} held by {owner[slot]}"
                owner[slot] = seg
                loaded_this_run.add(seg)
            elif kind == EVICT:
                assert seg in residents and owner.get(slot) == seg
                # the segment active at step k is k: only ones computed earlier may go
                assert seg < step, "evicted the active segment or one not yet computed"
                del owner[slot]
                residents.discard(seg)
            elif kind == ACTIVATE:
                assert owner.get(slot) == seg, f"activate {seg} finds slot {slot} holding {owner.get(slot)}"
                assert seg in residents or seg in loaded_this_run
                activated.append(seg)
            peak = max(peak, len(owner))
            if kind == ACTIVATE and seg not in residents:
                del owner[slot]          # a streamed slot is free once its segment computed
        assert activated == list(range(len(activated))), "segments activate in order"
    return peak
