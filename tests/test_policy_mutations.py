"""Plant plausible mistakes in the plan-change, cross-run and expert-cache rules of the
oracle (on the CPU) and check that a pin catches each one."""
import numpy as np
import pytest

from oracle import expert_cache as X
from oracle import policy as Pol

import test_expert_cache_oracle as TX
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


_ORIG_CACHE = X.cache_passes

MUTATIONS = {
    "replan_evicts_from_the_front": (Pol.Sim, "_evict_residents_down_to", _evict_ascending),
    "stale_prefetch_not_released": (Pol.Sim, "_release_carried", _release_silently),
    "hot_set_ties_to_high_index": (X, "hot_set", _hot_ties_high),
    "cache_hit_without_fill": (X, "cache_passes", _cache_no_fill_needed),
    "cache_counts_current_pass": (X, "cache_passes", _cache_counts_this_pass),
}


def _pins():
    """Every pin of the two test modules, with the parameters they run with."""
    out = []
    for mod in (TR, TX):
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
    monkeypatch.setattr(target, attr, fn)
    if target is X:  # the pin modules imported the functions by name
        for mod in (TX,):
            if hasattr(mod, attr):
                monkeypatch.setattr(mod, attr, fn)
    caught = []
    for pname, pin, kw in _pins():
        try:
            pin(**kw)
        except (AssertionError, ValueError, KeyError, IndexError):
            caught.append(pname)
    assert caught, f"no pin caught the planted mistake {name}"
