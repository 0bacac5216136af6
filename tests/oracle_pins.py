"""Pins for the fp64 oracle: facts fixed by the pages or by mathematics.

Each check takes the oracle's forward module (or a stand-in with a planted
mistake) and raises AssertionError when the oracle disagrees with the fact.
The checks never call the oracle to make their own expected values: they use
closed forms, textbook constants, pure-Python brute force on tiny inputs, or
special cases that reduce to another, independently checked function.
"""
from __future__ import annotations

import math
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _close(a, b, tol=1e-12):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    assert a.shape == b.shape, (a.shape, b.shape)
    err = np.max(np.abs(a - b)) if a.size else 0.0
    scale = max(1.0, float(np.max(np.abs(b))) if b.size else 1.0)
    assert err <= tol * scale, f"max err {err} > {tol} * {scale}"


def load_activation_values():
    rows = []
    with open(os.path.join(GOLDEN, "gelu_silu_values.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            fn, z, v = line.split()
            rows.append((fn, float(z), float(v)))
    return rows


# ---------------------------------------------------------------- activations
def check_activation_values(F):
    for fn, z, v in load_activation_values():
        got = float(getattr(F, fn)(np.array([z]))[0])
        assert abs(got - v) <= 1e-14 * max(1.0, abs(v)), f"{fn}({z}) = {got}, table {v}"


def check_activation_limits(F):
    z = np.array([-40.0, -12.0, 12.0, 40.0, 700.0, -700.0])
    g = F.gelu(z)
    assert abs(g[0]) < 1e-300 and abs(g[1]) < 1e-30, "GELU(-large) must vanish"
    assert abs(g[2] - 12.0) < 1e-30 and g[3] == 40.0, "GELU(large) must be z"
    s = F.silu(z)
    assert np.all(np.isfinite(s)), "SiLU must not overflow"
    assert abs(s[3] - 40.0) < 1e-15 and abs(s[0]) < 1e-15
    # odd-part identities: GELU(z) - GELU(-z) = z, SiLU(z) - SiLU(-z) = z
    w = np.linspace(-5, 5, 41)
    _close(F.gelu(w) - F.gelu(-w), w, 1e-14)
    _close(F.silu(w) - F.silu(-w), w, 1e-14)


# ---------------------------------------------------------------- linear layers
def _brute_linear(x, w, b=None):
    T, K = len(x), len(x[0])
    N = len(w)
    out = []
    for t in range(T):
        row = []
        for n in range(N):
            acc = 0.0
            for k in range(K):
                acc += x[t][k] * w[n][k]
            row.append(acc + (b[n] if b is not None else 0.0))
        out.append(row)
    return out


def _rng(seed):
    return np.random.default_rng(seed)


def check_linear_brute(F):
    r = _rng(1)
    x = r.standard_normal((3, 5))
    w = r.standard_normal((4, 5))        # [out, in], not square: a transpose cannot pass
    b = r.standard_normal(4)
    _close(F.linear(x, w, b), _brute_linear(x.tolist(), w.tolist(), b.tolist()), 1e-13)
    _close(F.linear(x, w), _brute_linear(x.tolist(), w.tolist()), 1e-13)


def check_linear_gelu_scalar(F):
    r = _rng(2)
    x = r.standard_normal((2, 3))
    w = r.standard_normal((5, 3))
    b = r.standard_normal(5)
    pre = _brute_linear(x.tolist(), w.tolist(), b.tolist())
    ref = [[v * 0.5 * (1.0 + math.erf(v / math.sqrt(2.0))) for v in row] for row in pre]
    _close(F.linear_gelu(x, w, b), ref, 1e-13)
    # identity weights, zero bias: elementwise GELU
    _close(F.linear_gelu(x, np.eye(3), np.zeros(3)), F.gelu(x), 0)


def _brute_ffn(x, w1, b1, w2, b2, p=None):
    xin = _brute_linear(x, p) if p is not None else x
    h = _brute_linear(xin, w1, b1)
    h = [[v * 0.5 * (1.0 + math.erf(v / math.sqrt(2.0))) for v in row] for row in h]
    o = _brute_linear(h, w2, b2)
    return [[xi + oi for xi, oi in zip(xr, orow)] for xr, orow in zip(x, o)]


def check_ffn_brute(F):
    r = _rng(3)
    H, Fh, T = 3, 7, 4
    x = r.standard_normal((T, H))
    w1, b1 = r.standard_normal((Fh, H)), r.standard_normal(Fh)
    w2, b2 = r.standard_normal((H, Fh)), r.standard_normal(H)
    _close(F.ffn_gelu(x, w1, b1, w2, b2),
           _brute_ffn(x.tolist(), w1.tolist(), b1.tolist(), w2.tolist(), b2.tolist()), 1e-12)
    # zero weights keep the residual and the output bias: y = x + b2
    _close(F.ffn_gelu(x, 0 * w1, 0 * b1, 0 * w2, b2), x + b2, 0)


def check_ffn_proj(F):
    r = _rng(4)
    H, Fh, T = 3, 6, 5
    x = r.standard_normal((T, H))
    p = r.standard_normal((H, H))
    w1, b1 = r.standard_normal((Fh, H)), r.standard_normal(Fh)
    w2, b2 = r.standard_normal((H, Fh)), r.standard_normal(H)
    _close(F.ffn_gelu_proj(x, p, w1, b1, w2, b2),
           _brute_ffn(x.tolist(), w1.tolist(), b1.tolist(), w2.tolist(), b2.tolist(),
                      p.tolist()), 1e-12)
    # P = I reduces to the plain FFN; P = 2I scales only the FFN input, not the residual
    _close(F.ffn_gelu_proj(x, np.eye(H), w1, b1, w2, b2), F.ffn_gelu(x, w1, b1, w2, b2), 1e-14)
    two = F.ffn_gelu_proj(x, 2 * np.eye(H), w1, b1, w2, b2)
    _close(two, x + (F.ffn_gelu(2 * x, w1, b1, w2, b2) - 2 * x), 1e-12)


def _brute_swiglu(x, g, u, d):
    a = _brute_linear(x, g)
    c = _brute_linear(x, u)
    h = [[ai / (1.0 + math.exp(-ai)) * ci for ai, ci in zip(ar, cr)] for ar, cr in zip(a, c)]
    o = _brute_linear(h, d)
    return [[xi + oi for xi, oi in zip(xr, orow)] for xr, orow in zip(x, o)]


def check_swiglu_brute(F):
    r = _rng(5)
    H, Fh, T = 4, 6, 3
    x = r.standard_normal((T, H))
    g, u, d = r.standard_normal((Fh, H)), r.standard_normal((Fh, H)), r.standard_normal((H, Fh))
    _close(F.swiglu(x, g, u, d), _brute_swiglu(x.tolist(), g.tolist(), u.tolist(), d.tolist()),
           1e-12)
    _close(F.swiglu(x, g, u, 0 * d), x, 0)


# ---------------------------------------------------------------- MoE routing
def _brute_topk(row, k):
    order = sorted(range(len(row)), key=lambda e: (-float(row[e]), e))[:k]
    m = max(float(row[e]) for e in order)
    ex = [math.exp(float(row[e]) - m) for e in order]
    s = sum(ex)
    return order, [v / s for v in ex]


def check_route_topk(F):
    r = _rng(6)
    lg = r.standard_normal((9, 16)).astype(np.float32)
    lg[0, :] = 0.5                        # all tied: lowest indices win, equal weights
    lg[1, [3, 7, 11]] = 4.0               # a three-way tie at the top
    lg[2, 5] = 60.0                       # one dominant expert
    sel, w = F.route_topk(lg, 4)
    for t in range(lg.shape[0]):
        order, ww = _brute_topk(lg[t], 4)
        assert list(sel[t]) == order, (t, list(sel[t]), order)
        _close(w[t], ww, 1e-14)
    assert list(sel[0]) == [0, 1, 2, 3]
    _close(w[0], [0.25] * 4, 1e-15)
    assert list(sel[1][:3]) == [3, 7, 11]
    assert w[2][0] >= 1 - 1e-15 and w[2][1] < 1e-20


def _brute_group(sel, E):
    k = len(sel[0])
    table, bounds = [], [0]
    for e in range(E):
        for t in range(len(sel)):
            for j in range(k):
                if sel[t][j] == e:
                    table.append(t * k + j)
        bounds.append(len(table))
    return table, bounds


def check_group_by_expert(F):
    r = _rng(7)
    for T, k, E in ((1, 1, 1), (5, 2, 3), (13, 3, 8), (32, 8, 16)):
        sel = np.stack([r.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
        table, bounds = F.group_by_expert(sel, E)
        bt, bb = _brute_group(sel.tolist(), E)
        assert list(table) == bt and list(bounds) == bb, (T, k, E)


def check_moe_reductions(F):
    r = _rng(8)
    T, H, Fh, E, k = 6, 4, 5, 6, 3
    x = r.standard_normal((T, H))
    ex = {e: (r.standard_normal((Fh, H)), r.standard_normal((Fh, H)), r.standard_normal((H, Fh)))
          for e in range(E)}
    # (a) all experts equal: the weights sum to one, so the layer is one SwiGLU
    same = ex[0]
    lg = r.standard_normal((T, E)).astype(np.float32)
    _close(F.moe_swiglu(x, lg, lambda e: same, k), F.swiglu(x, *same), 1e-12)
    # (b) one expert far ahead of the rest: its weight is 1 to double precision
    lg2 = r.standard_normal((T, E)).astype(np.float32)
    lg2[:, 4] = 80.0
    _close(F.moe_swiglu(x, lg2, lambda e: ex[e], k), F.swiglu(x, *ex[4]), 1e-12)
    # (c) brute force: per token, the weighted sum of its k experts
    sel_ref = []
    out = []
    for t in range(T):
        order, w = _brute_topk(lg[t], k)
        sel_ref.append(order)
        acc = [0.0] * H
        for e, we in zip(order, w):
            g, u, d = ex[e]
            y = _brute_swiglu([x[t].tolist()], g.tolist(), u.tolist(), d.tolist())[0]
            for i in range(H):
                acc[i] += we * (y[i] - x[t][i])
        out.append([x[t][i] + acc[i] for i in range(H)])
    _close(F.moe_swiglu(x, lg, lambda e: ex[e], k), out, 1e-12)


ALL_CHECKS = [check_activation_values, check_activation_limits, check_linear_brute,
              check_linear_gelu_scalar, check_ffn_brute, check_ffn_proj, check_swiglu_brute,
              check_route_topk, check_group_by_expert, check_moe_reductions]
