"""Plant plausible mistakes in the policy oracle (on the CPU): its plan, prefetch window,
ring numbering, plan-change, cross-run and expert-cache rules. Each one must be caught by
a pin that does not involve the library's own scheduler: the pages' tables and worked
numbers, brute-force plan search, the slot replay and the window counted from events."""
import numpy as np
import pytest

from oracle import expert_cache as X
from oracle import policy as Pol

import test_expert_cache_oracle as TX
import test_policy_oracle as TP
import test_policy_replan as TR


def _evict_ascending(self, keep):
    for r in range(keep, self.loaded_R):               # from the front of the released range
        self._emit(-1, Pol.EVICT, r, r, 0)
        self.stats.evictions += 1
        if not self.use_pool:
            self._free(self.seg_slot_bytes[r])
    self.loaded_R = min(self.loaded_R, keep)


def _release_silently(self):
    if not self.use_pool:
        for seg, _ in self.carried:
            self._free(self.seg_slot_bytes[seg])
    self.carried = []                                  # no EVICT events for stale prefetches


def _hot_ties_high(counts, K, first_streamed):
    L, E = counts.shape
    cand = [(-int(counts[l, e]), -l, -e) for l in range(first_streamed, L) for e in range(E) if counts[l, e] > 0]
    cand.sort()
    return [(-l, -e) for _, l, e in cand[:K]]


def _cache_no_fill_needed(used, K, first_streamed=0):
    out = _ORIG_CACHE(used, K, first_streamed)
    fixed = []
    for u, (host, hits, fills, hot) in zip(used, out):
        u = np.asarray(u, bool)
        hits = hits | fills                            # a hot expert counts as a hit at once
        fixed.append((u & ~hits, hits, np.zeros_like(fills), hot))
    return fixed


def _cache_counts_this_pass(used, K, first_streamed=0):
    L, E = np.asarray(used[0]).shape
    counts = np.zeros((L, E), np.int64)
    filled, out = set(), []
    for u in used:
        u = np.asarray(u, bool)
        counts[first_streamed:] += u[first_streamed:]  # this pass counted before the hot set
        hot = X.hot_set(counts, K, first_streamed)
        filled &= set(hot)
        hits = np.zeros((L, E), bool)
        fills = np.zeros((L, E), bool)
        for (l, e) in hot:
            if u[l, e] and (l, e) in filled:
                hits[l, e] = True
            elif u[l, e]:
                fills[l, e] = True
        host = u & ~hits
        host[:first_streamed] = False
        filled |= {(int(l), int(e)) for l, e in zip(*np.nonzero(fills))}
        out.append((host, hits, fills, hot))
    return out


def _window_one_short(j, R, d):
    return 0 if j < d - 1 else R + j - d + 1          # a window of d - 1 ahead of the active one


def _window_one_long(j, R, d):
    return 0 if j < d + 1 else R + j - d - 1          # d + 1 ahead: more loads than the ring holds


def _window_ignores_residents(j, R, d):
    return max(0, R + j - d)                          # nothing prefetched during the resident prefix


def _window_counts_residents(j, R, d):
    return max(0, j - d)                              # residents consume depth


def _ring_without_resident_offset(J, R, Q):
    return J % Q                                      # ring slots overlap the resident slots


def _ring_one_slot_short(J, R, Q):
    return R + J % max(1, Q - 1)                      # the ring reuses a slot one load too early


def _plan_residents_first(seg_slot_bytes, shared_bytes, depth, resident, max_vram, slot_cap=None):
    p = _ORIG_PLAN(seg_slot_bytes, shared_bytes, depth, resident, max_vram, slot_cap)
    if p.warn_mandatory or p.avail >= p.N:
        return p
    R = min(p.N if resident < 0 else min(resident, p.N), p.avail - 1)   # residents take the room first
    d = min(depth, p.avail - R - 1)
    M = p.N - R
    Q = min(d + 1, M) if M > 0 else 0
    return Pol.Plan(p.N, p.S, p.shared_total, p.avail, d, R, Q, R + Q, p.warn_mandatory)


def _plan_budget_rounds_up(seg_slot_bytes, shared_bytes, depth, resident, max_vram, slot_cap=None):
    if max_vram > 0:
        S = max(seg_slot_bytes)
        sh = sum(Pol.align_up(b) for b in shared_bytes)
        max_vram = sh + -(-(max_vram - sh) // S) * S if max_vram > sh else max_vram
    return _ORIG_PLAN(seg_slot_bytes, shared_bytes, depth, resident, max_vram, slot_cap)


_ORIG_CACHE = X.cache_passes
_ORIG_PLAN = Pol.plan_slots

MUTATIONS = {
    "window_one_short": (Pol, "issue_step", _window_one_short),
    "window_one_long": (Pol, "issue_step", _window_one_long),
    "window_ignores_resident_prefix": (Pol, "issue_step", _window_ignores_residents),
    "window_counts_residents": (Pol, "issue_step", _window_counts_residents),
    "ring_overlaps_residents": (Pol, "ring_slot", _ring_without_resident_offset),
    "ring_one_slot_short": (Pol, "ring_slot", _ring_one_slot_short),
    "plan_residents_before_depth": (Pol, "plan_slots", _plan_residents_first),
    "plan_budget_rounds_up": (Pol, "plan_slots", _plan_budget_rounds_up),
    "replan_evicts_from_the_front": (Pol.Sim, "_evict_residents_down_to", _evict_ascending),
    "stale_prefetch_not_released": (Pol.Sim, "_release_carried", _release_silently),
    "hot_set_ties_to_high_index": (X, "hot_set", _hot_ties_high),
    "cache_hit_without_fill": (X, "cache_passes", _cache_no_fill_needed),
    "cache_counts_current_pass": (X, "cache_passes", _cache_counts_this_pass),
}


def _pins():
    """Every pin of the two test modules, with the parameters they run with."""
    out = []
    for mod in (TP, TR, TX):
        for name in dir(mod):
            fn = getattr(mod, name)
            if not name.startswith("test_") or not callable(fn):
                continue
            marks = getattr(fn, "pytestmark", [])
            params = [m for m in marks if m.name == "parametrize"]
            if not params:
                out.append((name, fn, {}))
                continue
            argname, values = params[0].args
            for v in values:
                out.append((f"{name}[{v}]", fn, {argname: v}))
    return out


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_policy_mutation_is_caught(name, monkeypatch):
    target, attr, fn = MUTATIONS[name]
    orig = getattr(target, attr)
    monkeypatch.setattr(target, attr, fn)
    # the pin modules that imported the function by name see the planted one too
    for mod in (TP, TR, TX):
        if getattr(mod, attr, None) is orig:
            monkeypatch.setattr(mod, attr, fn)
    caught = []
    for pname, pin, kw in _pins():
        try:
            pin(**kw)
        except (AssertionError, ValueError, KeyError, IndexError):
            caught.append(pname)
    assert caught, f"no pin caught the planted mistake {name}"
