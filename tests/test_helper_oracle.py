"""The idle-stage helper's share rule and expert split (oracle/helper.py) against the
page's rows, the rule's closed form at its corners, and the plain MoE forward."""
import os

import numpy as np
import pytest

from oracle import forward as F
from oracle import helper as Hp

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "helper_share.txt")


def _rows():
    out = []
    for line in open(GOLDEN):
        line = line.strip()
        if line and not line.startswith("#"):
            t, exp = (p.strip() for p in line.split("|"))
            out.append((int(t), exp))
    return out


@pytest.mark.parametrize("tokens,exp", _rows())
def test_page_rows(tokens, exp):
    s = Hp.helper_share(tokens)
    assert (s > 0) == (exp == "on"), (tokens, s)


def test_rule_corners():
    assert Hp.helper_share(0) == 0.45 and Hp.helper_share(819) == 0.45       # capped while 0.5 - T/16384 > 0.45
    assert Hp.helper_share(820) < 0.45
    assert Hp.helper_share(1100) == pytest.approx(0.5 - 1100 / 16384)         # 0.4329...
    assert Hp.helper_share(3276) == 0.5 - 3276 / 16384 == 0.300048828125     # last token count with a share
    assert Hp.helper_share(3277) == 0.0                                       # "off below 0.3 (~3.3K tokens)"
    shares = [Hp.helper_share(t) for t in range(0, 3277)]
    assert all(a >= b for a, b in zip(shares, shares[1:]))                    # falls with the chunk


def test_split_is_a_partition():
    rng = np.random.default_rng(2)
    for _ in range(200):
        routed = sorted(set(rng.integers(0, 128, rng.integers(0, 129)).tolist()))
        share = float(rng.choice([0.0, 0.3, 0.37, 0.45]))
        mine, theirs = Hp.split_experts(routed, share)
        assert sorted(mine + theirs) == routed and not set(mine) & set(theirs)
        assert len(theirs) == int(np.floor(share * len(routed)))
        assert not theirs or not mine or max(mine) < min(theirs)             # the helper takes the top


def test_split_layer_equals_the_plain_layer():
    rng = np.random.default_rng(7)
    T, H, Fd, E, k = 40, 24, 16, 10, 3
    x = rng.standard_normal((T, H))
    logits = rng.standard_normal((T, E)).astype(np.float32)
    W = {e: (rng.standard_normal((Fd, H)) / 5, rng.standard_normal((Fd, H)) / 5, rng.standard_normal((H, Fd)) / 4)
         for e in range(E)}
    ref = F.moe_swiglu(x, logits, W.__getitem__, k)
    for share in (0.0, 0.3, 0.45):
        got = Hp.moe_layer_split(x, logits, W.__getitem__, k, share)
        np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)
    # the helper's rows are exactly the rows of its experts
    sel, _ = F.route_topk(logits, k)
    mine, theirs = Hp.split_experts(np.unique(sel), 0.45)
    rows_h = Hp.expert_rows(x, logits, W.__getitem__, k, theirs)
    assert set(rows_h) == {(t, j) for t in range(T) for j in range(k) if sel[t, j] in set(theirs)}


def test_library_rule_and_split_match_the_oracle():
    """The library's host functions (ls_helper_share, ls_helper_split) against the oracle."""
    from host_offloaded_weight_gb300 import lstream as L
    for t in list(range(0, 4000, 7)) + [819, 820, 3276, 3277, 8000, 100000]:
        assert L.ls_helper_share(t) == Hp.helper_share(t), t
    rng = np.random.default_rng(9)
    for _ in range(300):
        E = int(rng.integers(1, 200))
        routed = (rng.random(E) < rng.random()).astype(np.uint8)
        share = float(rng.choice([0.0, 0.3, 0.4329, 0.45, 1.0]))
        mask = L.ls_helper_split(routed, share)
        _, theirs = Hp.split_experts(np.nonzero(routed)[0], share)
        assert np.nonzero(mask)[0].tolist() == theirs
    import pytest as _p
    with _p.raises(L.LsError):
        L.ls_helper_split(np.ones(4, np.uint8), 1.5)
