"""Pins of the expert-cache policy (oracle/expert_cache.py): hand-worked cases and
invariants that hold for any routing. No GPU."""
import numpy as np

from oracle.expert_cache import cache_passes, hot_set


def _u(L, E, pairs):
    a = np.zeros((L, E), bool)
    for l, e in pairs:
        a[l, e] = True
    return a


def test_hot_set_ranks_by_count_then_expert_then_layer():
    c = np.array([[2, 0, 1], [2, 3, 0]])
    assert hot_set(c, 2, 0) == [(1, 1), (0, 0)]
    # equal counts: the lower expert first, then the lower layer (spread over the layers)
    assert hot_set(np.ones((3, 2), int), 4, 0) == [(0, 0), (1, 0), (2, 0), (0, 1)]
    assert hot_set(c, 4, 0) == [(1, 1), (0, 0), (1, 0), (0, 2)]
    assert hot_set(c, 9, 0) == [(1, 1), (0, 0), (1, 0), (0, 2)]   # zero counts never enter
    assert hot_set(c, 2, 1) == [(1, 1), (1, 0)]                   # residents excluded


def test_worked_sequence():
    # 1 layer, 3 experts, K = 1
    used = [_u(1, 3, [(0, 0), (0, 1)]),   # pass 0: no history, nothing hot
            _u(1, 3, [(0, 1)]),           # pass 1: counts e0=1,e1=1 -> hot (0,0); not routed: no fill
            _u(1, 3, [(0, 0), (0, 1)]),   # pass 2: counts e0=1,e1=2 -> hot (0,1) unfilled: routed -> fill
            _u(1, 3, [(0, 1), (0, 2)])]   # pass 3: hot (0,1) filled and routed -> hit
    out = cache_passes(used, 1)
    assert [o[3] for o in out] == [[], [(0, 0)], [(0, 1)], [(0, 1)]]
    assert not out[0][1].any() and not out[1][1].any() and not out[2][1].any()
    assert out[2][2][0, 1] and out[3][1][0, 1]
    assert out[3][0].tolist() == [[False, False, True]]              # only e2 crosses the host link


def test_invariants_random():
    rng = np.random.default_rng(3)
    for _ in range(200):
        L, E = rng.integers(1, 5), rng.integers(1, 9)
        K = int(rng.integers(0, L * E + 2))
        R = int(rng.integers(0, L))
        p = rng.random(E) ** 3                                        # skewed popularity
        used = [rng.random((L, E)) < p for _ in range(int(rng.integers(1, 7)))]
        out = cache_passes(used, K, R)
        filled = set()
        counts = np.zeros((L, E), int)
        for u, (host, hits, fills, hot) in zip(used, out):
            assert len(hot) <= K and all(l >= R and counts[l, e] > 0 for l, e in hot)
            filled &= set(hot)
            assert not (hits & ~u).any() and not (hits & host).any()
            for l, e in zip(*np.nonzero(hits)):
                assert (l, e) in filled                              # a hit was filled earlier
            assert ((host | hits)[R:] == u[R:]).all()               # every routed expert arrives
            assert not fills[:R].any() and not (fills & ~host).any()  # fills come with host copies
            filled |= {(int(l), int(e)) for l, e in zip(*np.nonzero(fills))}
            assert len(filled) <= K
            counts[R:] += u[R:]


def test_no_cache_moves_every_routed_expert():
    rng = np.random.default_rng(5)
    used = [rng.random((3, 6)) < 0.5 for _ in range(4)]
    for u, (host, hits, _, _) in zip(used, cache_passes(used, 0)):
        assert (host == u).all() and not hits.any()
