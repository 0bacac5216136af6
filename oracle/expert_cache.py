"""Expert cache of the streamed MoE layers (oracle; test infrastructure only).

A fixed device region holds up to K expert blobs (one expert's gate, up and down
matrices). In a pass, a streamed layer's routed experts that sit in the cache are
copied from it inside device memory, and only the others cross the host link.
This is the "keep hot experts resident and stream only unseen routed experts"
item; the pages ("layer split: overlap the stages' hand-off" and the pipelined
verify windows page) speak of per-GPU expert caches and streaming the routed
experts of a layer without fixing a policy, so the policy below is this
project's reading, chosen to be deterministic and checkable:

  * counts[l][e] = the number of earlier passes in which expert e of layer l was
    routed (by any token);
  * the hot set of pass r is the K pairs (l, e) of streamed layers (l >= R) with
    the largest counts, counts > 0 only, ties to the lower expert, then the lower
    layer (equal counts spread the cache over the layers, so that every layer's
    host copy shrinks and the prefetch pipeline keeps the link busy);
  * a hot pair is "filled" once its expert has been copied into the cache: when
    it is routed in a pass that starts with it hot and unfilled, its host copy
    in that pass also fills the cache. A pair that leaves the hot set is dropped;
  * in pass r, layer l moves from the host the routed experts that are not hot
    and filled at the start of the pass; the routed, hot and filled ones are cache
    hits.
"""
from __future__ import annotations

import numpy as np


def hot_set(counts: np.ndarray, K: int, first_streamed: int) -> list:
    """The K pairs with the largest counts (> 0) among layers >= first_streamed."""
    L, E = counts.shape
    cand = [(-int(counts[l, e]), e, l) for l in range(first_streamed, L) for e in range(E) if counts[l, e] > 0]
    cand.sort()
    return [(l, e) for _, e, l in cand[:K]]


def cache_passes(used: list, K: int, first_streamed: int = 0):
    """used: per pass a bool array [layers, experts] of routed experts.

    Returns per pass (host, hits, fills, hot): bool arrays [layers, experts] of the
    experts moved from the host, served from the cache, copied into the cache, and
    the hot list of that pass."""
    L, E = np.asarray(used[0]).shape
    counts = np.zeros((L, E), np.int64)
    filled: set = set()
    out = []
    for u in used:
        u = np.asarray(u, bool)
        hot = hot_set(counts, K, first_streamed)
        filled &= set(hot)                              # pairs that left the hot set are dropped
        hits = np.zeros((L, E), bool)
        fills = np.zeros((L, E), bool)
        for (l, e) in hot:
            if u[l, e] and (l, e) in filled:
                hits[l, e] = True
            elif u[l, e]:
                fills[l, e] = True
        host = u & ~hits
        host[:first_streamed] = False                   # residents hold all their experts
        for l, e in zip(*np.nonzero(fills)):
            filled.add((int(l), int(e)))
        counts[first_streamed:] += u[first_streamed:]
        out.append((host, hits, fills, hot))
    return out
