"""Event-level simulator of the streaming policy (oracle; test infrastructure only).

It computes, from integers alone, the plan (slot size S, residents R, prefetch
depth d, ring slots Q, pool slots P) and the exact list of schedule events the
runtime must execute. The runtime's own scheduler is separate code; tests
compare the two event lists for equality.

The simulator is written as rules, each a function of its own:
  * ``plan_slots``  the plan in closed form: depth first, then the longest
                    resident prefix that still fits;
  * ``issue_step``  the prefetch window: the step at which each streamed load of
                    a run is issued, as a formula of (R, d) and the load's number;
  * ``ring_slot``   the slot of each streamed load, as a formula of its number;
  * memory and failure rules, applied on top of the window's schedule: the
    pool's degradation to fewer slots, runtime pressure with the pool off
    (eviction from the end of the resident prefix), the synchronous fallback
    when asynchronous transfer is unavailable, and plan changes between runs.

Sources:
  "feat: prefetch streamed layers during compute" (sd.cpp #1905), Summary and
  the Effective behavior table: depth 0 is synchronous streaming, depth N asks
  for N future segments reduced to fit the budget; a positive budget is never
  exceeded by prefetch; the active segment is never evicted; residents are a
  maximum (auto = -1 keeps as many leading segments as the budget allows);
  the prefetch window has priority over optional residents; shared parameters
  are deduplicated; residents are evicted from the end of the prefix under
  runtime memory pressure; when asynchronous transfer is unavailable or a
  prefetch allocation fails, execution continues synchronously; max-vram 0
  disables segmentation.
  "feat: pool VRAM for streamed layer" (sd.cpp #1906), Summary and the pool
  behavior table: one contiguous allocation of fixed slots sized for the
  largest private-parameter footprint; only the peak slot count is allocated;
  a failing pool is retried with fewer slots of the same size, down to one;
  the one-slot pool is mandatory execution memory (attempted, with a warning,
  even above the budget); reduced caps are remembered.

Readings where the pages are silent (each one listed with its reason in the
design notes of the repository):
  * budgets are bytes; the budget counts parameter memory only (shared
    region + pool slots);
  * tensors are packed at 256-byte aligned offsets; S = max over segments of the
    aligned sum of private tensor bytes; shared tensors count once;
  * the prefetch window at step k is the active segment plus the next d
    streamed (non-resident) segments; residents never consume depth; the window
    does not cross run boundaries (no cross-forward state, maintainer review);
  * every streamed segment is loaded through the copy queue when d >= 1,
    including the first one of a run;
  * shared parameters are resident (deduplicated) and loaded once in run 0,
    followed by the resident prefix, both synchronously;
  * load j of a run goes to ring slot R + (j mod Q) with Q = min(d + 1, N - R).

Plan changes between runs and the cross-run window (the pages' "releases stale
residents and prefetches when the graph plan changes", "evicts residents from
the end of the resident prefix", "reuses a sufficiently large pool ... and
remembers reduced runtime caps", sd.cpp #1905 and #1906, Summary):
  * ``replan`` takes new controls (depth, resident cap, budget) between runs. It
    plans with the same rules, under the remembered reduced slot cap, and keeps
    a remembered synchronous fallback;
  * prefetches issued for a run that has not started are stale: each one is
    released (EVICT of that segment and slot) first;
  * residents that the new plan no longer holds are released from the end of
    the prefix (EVICT, descending), before the next run's first step;
  * pool on: the pool is kept while the slot count stays the same. Otherwise it
    is given back and a pool of the new count is allocated (smaller counts tried
    on failure, as at registration). That empties every slot, so every old
    resident is released and the whole new prefix is loaded again. Pool off: the
    kept residents' buffers stay;
  * a run loads, synchronously before its first step, the residents that hold no
    data yet (LOAD_RESIDENT), so a grown prefix is filled at the next run;
  * cross-run window (opt-in; off matches the maintainer's removal of cross-forward
    state): the window of the last steps reaches into the next run's first
    streamed segments, so their prefetches are issued before the run ends. Load
    numbers then continue across runs (slot R + (J mod Q), J counted from the
    last plan change). The window crosses the boundary only when the ring is a
    full d + 1 slots (N - R > d).
"""
from __future__ import annotations

from dataclasses import dataclass, field

# event kinds (values shared with the C ABI's ls_event_kind)
SHARED_LOAD, LOAD_RESIDENT, LOAD_SYNC, PREFETCH, ACTIVATE, EVICT = range(6)
KIND_NAMES = ["SHARED_LOAD", "LOAD_RESIDENT", "LOAD_SYNC", "PREFETCH", "ACTIVATE", "EVICT"]

# status codes (values shared with the C ABI's ls_status)
OK, WARN_MANDATORY_SLOT, WARN_SYNC_FALLBACK = 0, 1, 2
ERR_INVALID_ARG, ERR_VERSION, ERR_OOM = -1, -2, -3

ALIGN = 256


def align_up(n: int, a: int = ALIGN) -> int:
    return (n + a - 1) // a * a


@dataclass
class Plan:
    N: int
    S: int
    shared_total: int
    avail: int          # slots the budget (or a reduced cap) allows
    d_req: int          # depth that fits the budget (before capping by streamed count)
    R: int
    Q: int
    P: int
    warn_mandatory: bool = False

    @property
    def M(self) -> int:
        return self.N - self.R

    @property
    def d(self) -> int:
        return min(self.d_req, self.M)


# ------------------------------------------------------------------ the plan
def plan_slots(seg_slot_bytes: list, shared_bytes: list, depth: int, resident: int,
               max_vram: int, slot_cap: int | None = None) -> Plan:
    """Plan from the budget (sd.cpp #1905 Summary and table; #1906 Summary and table).

    ``slot_cap`` is a remembered reduced slot count. In closed form:
      avail = slots the budget holds beside the shared region (all N when the budget
              is 0 but a cap is remembered), at most ``slot_cap``;
      d     = the requested depth, at most avail - 1 unless every segment fits
              (prefetch first: the ring of d + 1 slots must fit with no residents);
      R     = the resident cap, at most what is left beside that ring."""
    N = len(seg_slot_bytes)
    S = max(seg_slot_bytes)
    shared_total = sum(align_up(b) for b in shared_bytes)
    if max_vram == 0 and slot_cap is None:          # segmentation off: everything resident
        return Plan(N, S, shared_total, N, 0, N, 0, N)
    if max_vram == 0:
        avail, mandatory = N, False
    else:
        avail = max(0, max_vram - shared_total) // S
        mandatory = avail < 1
        if mandatory:
            # below one slot: only the mandatory execution slot, no residency, no prefetch
            return Plan(N, S, shared_total, 1, 0, 0, 1, 1, True)
    if slot_cap is not None:
        avail = min(avail, slot_cap)
    cap = N if resident < 0 else min(resident, N)
    if avail >= N:
        d, R = depth, cap                        # every segment fits whatever the depth
    else:
        d = min(depth, avail - 1)
        R = min(cap, avail - d - 1)
    M = N - R
    Q = min(d + 1, M) if M > 0 else 0
    return Plan(N, S, shared_total, avail, d, R, Q, R + Q, mandatory)


# ------------------------------------------------------------------ the window and the ring
def issue_step(j: int, R: int, d: int) -> int:
    """Step of a run at which its streamed load number j (from 0) enters the prefetch window.

    The window holds the active segment and the next d streamed segments (reading 3). At
    the steps of the resident prefix no streamed segment is active yet, so the window is
    streamed loads 0..d-1, all issued at step 0. Later, load j enters when streamed
    segment j - d (segment R + j - d) becomes active. Numbers j >= N - R are the next
    run's loads (cross-run window): the same rule puts them in the last d steps."""
    return 0 if j < d else R + j - d


def ring_slot(J: int, R: int, Q: int) -> int:
    """Pool slot of streamed load number J, counted over the runs that share one ring:
    the Q ring slots follow the R resident slots and are taken in turn."""
    return R + J % Q


def windows(R: int, d: int, first: int, reach: int) -> dict:
    """{step: [load numbers issued at that step, ascending]} for loads first..reach-1."""
    out: dict = {}
    for j in range(first, reach):
        out.setdefault(issue_step(j, R, d), []).append(j)
    return out


# ------------------------------------------------------------------ state across runs
@dataclass
class Stats:
    prefetch_queued: int = 0
    prefetch_activated: int = 0
    sync_loads: int = 0
    resident_loads: int = 0
    shared_loads: int = 0
    evictions: int = 0
    sync_fallbacks: int = 0
    pool_degradations: int = 0
    bytes_loaded: int = 0


@dataclass
class Sim:
    """Streaming context state mirrored by the simulator."""
    seg_slot_bytes: list
    shared: list                        # [(shared_id, bytes)], distinct ids
    depth: int
    resident: int
    max_vram: int
    use_pool: int
    alloc_cap: int | None = None        # parameter allocator refuses beyond this many live bytes
    fail_async: bool = False            # the first prefetch finds async transfer unavailable
    cross_run: bool = False             # the prefetch window crosses the run boundary
    plan: Plan | None = None
    slot_cap: int | None = None         # remembered reduced pool slot count
    loaded_R: int = 0                   # leading residents whose slots hold their data
    J: int = 0                          # streamed loads numbered since the last plan change (cross-run)
    carried: list = field(default_factory=list)   # [(seg, slot)] prefetched for the next run
    carried_R: int = 0                  # the resident prefix the carried prefetches were planned for
    status: int = OK
    R: int = 0
    d: int = 0
    run: int = 0
    async_ok: bool = True
    live: int = 0
    cur_R: int = 0
    events: list = field(default_factory=list)
    stats: Stats = field(default_factory=Stats)
    warnings: set = field(default_factory=set)

    # -------------------------------------------------------------- memory rules
    def _alloc(self, nbytes: int) -> bool:
        if nbytes == 0:
            return True
        if self.alloc_cap is not None and self.live + nbytes > self.alloc_cap:
            return False
        self.live += nbytes
        return True

    def _free(self, nbytes: int) -> None:
        self.live -= nbytes

    def _pool_for(self, p: Plan) -> Plan | None:
        """Pool degradation (sd.cpp #1906 table): the pool of plan p, else the plan for at
        most P - 1, P - 2, ..., 1 slots of the same size; each refused allocation counts one
        degradation. None when not even one slot can be had."""
        shared_b = [b for _, b in self.shared]
        for cap in range(p.P, 0, -1):
            q = p if cap == p.P else plan_slots(self.seg_slot_bytes, shared_b, self.depth, self.resident,
                                                self.max_vram, slot_cap=cap)
            q.warn_mandatory = p.warn_mandatory
            if self._alloc(q.P * q.S):
                if q.P < p.P:
                    self.slot_cap = q.P          # a reduced cap is remembered
                return q
            self.stats.pool_degradations += 1
        return None

    def _alloc_evicting(self, nbytes: int, k: int) -> bool:
        """Runtime pressure with the pool off (sd.cpp #1905 Summary): a load issued at step k
        that does not fit evicts residents from the end of the prefix, but only ones already
        computed in this run (index < k), so never the active segment."""
        while not self._alloc(nbytes):
            r = self.cur_R - 1
            if r < 0 or r >= k:
                return False
            self._emit(k, EVICT, r, r, 0)
            self._free(self.seg_slot_bytes[r])
            self.cur_R = r
        return True

    def _fallback(self) -> None:
        """Asynchronous transfer unavailable or a prefetch allocation failed: the rest of
        the run and every later run stream synchronously (remembered)."""
        self.async_ok = False
        self.d = 0
        self.fail_async = False
        self.stats.sync_fallbacks += 1
        self.warnings.add(WARN_SYNC_FALLBACK)

    def _emit(self, step, kind, seg, slot, nbytes):
        self.events.append((self.run, step, kind, seg, slot, nbytes))
        st = self.stats
        if kind in (SHARED_LOAD, LOAD_RESIDENT, LOAD_SYNC, PREFETCH):
            st.bytes_loaded += nbytes
        if kind == SHARED_LOAD:
            st.shared_loads += 1
        elif kind == LOAD_RESIDENT:
            st.resident_loads += 1
        elif kind == LOAD_SYNC:
            st.sync_loads += 1
        elif kind == PREFETCH:
            st.prefetch_queued += 1
        elif kind == EVICT:
            st.evictions += 1

    # -------------------------------------------------------------- register
    def register(self) -> int:
        """Plan, then allocate the shared region and (pool on) the slot pool."""
        p = plan_slots(self.seg_slot_bytes, [b for _, b in self.shared], self.depth, self.resident,
                       self.max_vram)
        if p.warn_mandatory:
            self.warnings.add(WARN_MANDATORY_SLOT)
        if not self._alloc(p.shared_total):
            self.status = ERR_OOM
            return ERR_OOM
        if self.use_pool:
            q = self._pool_for(p)
            if q is None:
                self._free(p.shared_total)
                self.status = ERR_OOM
                return ERR_OOM
            p = q
        self.plan = p
        self.R = p.R
        self.d = p.d_req
        self.status = WARN_MANDATORY_SLOT if p.warn_mandatory else OK
        return self.status

    # -------------------------------------------------------------- one run
    def run_once(self, load_bytes=None) -> int:
        """One pass over all segments; returns the run's status.

        ``load_bytes(seg)`` gives the bytes a load of ``seg`` moves in this run
        (default: its aligned private footprint)."""
        assert self.plan is not None
        N = self.plan.N
        lb = load_bytes or (lambda s: self.seg_slot_bytes[s])
        sz = self.seg_slot_bytes
        pool = bool(self.use_pool)

        # before the first step: shared region (run 0), stale carried loads, residents
        if self.run == 0:
            for sid, b in sorted(self.shared):
                self._emit(-1, SHARED_LOAD, sid, -1, b)
        if self.carried and self.carried_R != self.R:
            self._release_carried()          # planned for another ring: stale
        for i in range(self.loaded_R, self.R):
            if not pool and not self._alloc(sz[i]):
                self.R = i                   # the prefix ends where memory ran out
                break
            self._emit(-1, LOAD_RESIDENT, i, i, lb(i))
        self.loaded_R = self.R

        # this run's ring and window
        R = self.R
        M = N - R
        d = min(self.d, M)
        Q = min(self.d + 1, M) if M > 0 else 0
        J0 = self.J if self.cross_run else 0
        reach = M + d if (self.cross_run and M > d) else M
        carried_in, self.carried = self.carried, []
        prefetched = {seg for seg, _ in carried_in}
        sched = windows(R, d, len(carried_in), reach) if d >= 1 and self.async_ok else {}
        prefetching = bool(sched)
        waiting: list = []                   # load numbers whose window is open, not yet issued
        self.cur_R = R
        status, fell_back = OK, False

        def seg_of(j):
            return R + j % M

        for k in range(N):
            if prefetching:
                waiting += sched.get(k, [])
                issued = 0
                for j in waiting:
                    seg = seg_of(j)
                    if j >= M:
                        # the next run's loads never evict; without memory a load waits for a
                        # later step (its run loads the segment itself if none comes)
                        if not pool and not self._alloc(sz[seg]):
                            break
                    elif self.fail_async or (not pool and not self._alloc_evicting(sz[seg], k)):
                        self._fallback()
                        fell_back, prefetching = True, False
                        break
                    slot = ring_slot(J0 + j, R, Q)
                    self._emit(k, PREFETCH, seg, slot, lb(seg))
                    if j < M:
                        prefetched.add(seg)
                    else:
                        self.carried.append((seg, slot))
                    issued += 1
                waiting = waiting[issued:] if prefetching else []
            streamed = k >= R
            slot = ring_slot(J0 + k - R, R, Q) if streamed else k
            if streamed and k not in prefetched:
                if not pool and not self._alloc_evicting(sz[k], k):
                    status = ERR_OOM
                    break
                self._emit(k, LOAD_SYNC, k, slot, lb(k))
            self._emit(k, ACTIVATE, k, slot, 0)
            if k in prefetched:
                self.stats.prefetch_activated += 1
            if not pool and streamed:
                self._free(sz[k])            # its buffer goes back after its compute

        self.R = self.cur_R
        self.loaded_R = min(self.loaded_R, self.R)
        self.carried_R = R
        if self.cross_run:
            self.J = J0 + M
        self.run += 1
        if status != OK:
            return status
        return WARN_SYNC_FALLBACK if fell_back else OK

    # -------------------------------------------------------------- plan changes
    def replan(self, depth: int, resident: int, max_vram: int) -> int:
        """New controls between runs (the next run uses them). Returns the plan's status."""
        assert self.plan is not None
        self.depth, self.resident, self.max_vram = depth, resident, max_vram
        self._release_carried()
        old = self.plan
        p = plan_slots(self.seg_slot_bytes, [b for _, b in self.shared], depth, resident, max_vram,
                       slot_cap=self.slot_cap)
        if self.use_pool and p.P != old.P:
            # the pool is given back and allocated at the new count: every slot is emptied
            self._evict_residents_down_to(0)
            self._free(old.P * old.S)
            q = self._pool_for(p)
            if q is None:
                self.plan = None
                self.status = ERR_OOM
                return ERR_OOM
            p = q
        else:
            self._evict_residents_down_to(p.R)     # stale residents, from the end of the prefix
        self.plan = p
        self.R = p.R                  # a grown prefix is allocated and loaded at the next run
        self.loaded_R = min(self.loaded_R, p.R)
        self.d = p.d_req if self.async_ok else 0
        self.J = 0
        if p.warn_mandatory:
            self.warnings.add(WARN_MANDATORY_SLOT)
        self.status = WARN_MANDATORY_SLOT if p.warn_mandatory else OK
        return self.status

    def _evict_residents_down_to(self, keep: int) -> None:
        """Release residents keep .. loaded_R - 1, last first (before the next run's first step)."""
        for r in range(self.loaded_R - 1, keep - 1, -1):
            self._emit(-1, EVICT, r, r, 0)
            if not self.use_pool:
                self._free(self.seg_slot_bytes[r])
        self.loaded_R = min(self.loaded_R, keep)

    def _release_carried(self) -> None:
        """Prefetches issued for a run whose plan no longer holds: give back their slots."""
        for seg, slot in self.carried:
            self._emit(-1, EVICT, seg, slot, 0)
            if not self.use_pool:
                self._free(self.seg_slot_bytes[seg])
        self.carried = []


def simulate(seg_slot_bytes, shared=(), depth=0, resident=-1, max_vram=0, use_pool=1, runs=1,
             alloc_cap=None, fail_async=False, load_bytes=None, cross_run=False):
    """Register then run ``runs`` passes. Returns (sim, [status per run]).

    ``load_bytes`` is None or a list (per run) of per-segment byte counts."""
    sim = Sim(list(seg_slot_bytes), list(shared), depth, resident, max_vram, use_pool,
              alloc_cap=alloc_cap, fail_async=fail_async, cross_run=cross_run)
    st = sim.register()
    if st < 0:
        return sim, [st]
    out = []
    for r in range(runs):
        lb = None if load_bytes is None else (lambda s, r=r: load_bytes[r][s])
        out.append(sim.run_once(lb))
    return sim, out


def simulate_script(seg_slot_bytes, shared=(), depth=0, resident=-1, max_vram=0, use_pool=1,
                    script=(), alloc_cap=None, fail_async=False, cross_run=False):
    """Register, then follow ``script``: ("run",) for one pass or ("replan", depth, resident,
    max_vram). Returns (sim, [status per script step]); stops at the first error."""
    sim = Sim(list(seg_slot_bytes), list(shared), depth, resident, max_vram, use_pool,
              alloc_cap=alloc_cap, fail_async=fail_async, cross_run=cross_run)
    st = sim.register()
    if st < 0:
        return sim, [st]
    out = []
    for step in script:
        st = sim.run_once() if step[0] == "run" else sim.replan(*step[1:])
        out.append(st)
        if st < 0:
            break
    return sim, out
