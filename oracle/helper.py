"""The idle-stage helper of a layer split (oracle; test infrastructure only).

"prefill: a layer split's idle card streams a share of a one-chunk prompt's experts"
(Strata #663), What: with a model split in two stages over two GPUs, a prompt that fits
one chunk runs the stages one after the other, so while one card computes its layers
the other idles. The idle card takes a share of each layer's routed experts: it streams
those experts over its own host link, computes their rows, and hands the result rows
back through mapped host memory; the active card computes the rest and combines. The
share falls with the chunk, min(0.45, 0.5 - T/16384), and the helper is off when that is
below 0.3 (about 3.3K tokens).

Readings where the page is silent (listed with their reasons in the design notes):
  * the share is a share of the layer's routed experts by count (every expert has the
    same bytes, so it is also the share of the streamed bytes); the helper takes
    floor(share * routed) of them;
  * the helper's experts are the highest-numbered routed experts of the layer, the
    active card keeps the others;
  * each (token, k) row is computed entirely on the card that owns its expert, so the
    combine sees the same rows as without the helper (the page's MMQ grouping rounded
    differently; here the expert GEMM of a row does not depend on the other rows).
"""
from __future__ import annotations

import math

import numpy as np

from . import forward as F

SHARE_CAP = 0.45
SHARE_FLOOR = 0.3
SHARE_TOKENS = 16384


def helper_share(tokens: int) -> float:
    """The share of a layer's routed experts the idle card takes for a one-chunk prompt of
    `tokens` tokens: min(0.45, 0.5 - T/16384), and 0 (off) when that falls below 0.3."""
    s = min(SHARE_CAP, 0.5 - tokens / SHARE_TOKENS)
    return s if s >= SHARE_FLOOR else 0.0


def split_experts(routed, share: float):
    """(active card's experts, helper's experts) of one layer: the helper takes the
    floor(share * n) highest-numbered of the n routed experts."""
    routed = sorted(int(e) for e in routed)
    n_h = int(math.floor(share * len(routed)))
    return routed[:len(routed) - n_h], routed[len(routed) - n_h:]


def expert_rows(x, logits, experts, top_k, owned):
    """{(t, j): w[t, j] * SwiGLU_e(x[t])} for the (token, k) rows whose expert e is in
    `owned`: the rows one card computes and, for the helper, hands back."""
    sel, w = F.route_topk(logits, top_k)
    out = {}
    owned = set(int(e) for e in owned)
    for e in sorted(owned):
        t_idx, k_idx = np.nonzero(sel == e)
        if t_idx.size == 0:
            continue
        g, u, d = experts(e)
        ye = F.swiglu_mlp(x[t_idx], g, u, d)
        for r, (t, j) in enumerate(zip(t_idx, k_idx)):
            out[(int(t), int(j))] = w[t, j] * ye[r]
    return out


def combine(x, rows, top_k):
    """out[t] = x[t] + sum over j = 0..k-1 of the row (t, j), in j order."""
    T, H = x.shape
    acc = np.zeros((T, H), np.float64)
    for t in range(T):
        for j in range(top_k):
            acc[t] += rows[(t, j)]
    return x + acc


def moe_layer_split(x, logits, experts, top_k, share):
    """One MoE layer computed by the active card and the helper with the page's share,
    then combined on the active card."""
    sel, _ = F.route_topk(logits, top_k)
    mine, theirs = split_experts(np.unique(sel), share)
    rows = expert_rows(x, logits, experts, top_k, mine)
    rows.update(expert_rows(x, logits, experts, top_k, theirs))
    return combine(x, rows, top_k)
