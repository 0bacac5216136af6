"""Plant plausible mistakes in the oracle (on the CPU) and check a pin catches each.

A pin set that a dropped term, a wrong sign or index, or a transposed operand
slips through would not be pinning anything.
"""
import math

import numpy as np
import pytest
from scipy.special import erf

from oracle import forward as F

import oracle_pins as P


def _gelu_no_sqrt2(z):
    return 0.5 * z * (1.0 + erf(z))


def _gelu_tanh(z):
    return 0.5 * z * (1 + np.tanh(math.sqrt(2 / math.pi) * (z + 0.044715 * z ** 3)))


def _silu_sign(z):
    return z / (1.0 + np.exp(z))


def _linear_no_bias(x, w, b=None):
    return x @ w.T


def _linear_transposed(x, w, b=None):
    y = w @ x.T                     # [out, T] instead of [T, out]
    return y + (b[:, None] if b is not None else 0)


def _ffn_no_residual(x, w1, b1, w2, b2):
    return F.linear(F.gelu(F.linear(x, w1, b1)), w2, b2)


def _ffn_proj_wrong_residual(x, p, w1, b1, w2, b2):
    u = F.linear(x, p)
    return u + F.linear(F.gelu(F.linear(u, w1, b1)), w2, b2)


def _swiglu_swapped(x, g, u, d):
    return x + F.linear(F.silu(F.linear(x, u)) * F.linear(x, g), d)


def _swiglu_mlp_swapped(x, g, u, d):
    return F.linear(F.silu(F.linear(x, u)) * F.linear(x, g), d)


def _route_ties_high(logits, k):
    lg = np.asarray(logits, np.float32)
    E = lg.shape[1]
    order = (E - 1 - np.argsort(-lg[:, ::-1], axis=1, kind="stable"))[:, :k]
    ch = np.take_along_axis(lg, order, axis=1).astype(np.float64)
    e = np.exp(ch - ch.max(axis=1, keepdims=True))
    return order.astype(np.int32), e / e.sum(axis=1, keepdims=True)


def _route_full_softmax(logits, k):
    lg = np.asarray(logits, np.float32).astype(np.float64)
    order = np.argsort(-lg, axis=1, kind="stable")[:, :k]
    e = np.exp(lg - lg.max(axis=1, keepdims=True))
    w = e / e.sum(axis=1, keepdims=True)
    return order.astype(np.int32), np.take_along_axis(w, order, axis=1)


def _group_reversed(sel, n_experts):
    table, bounds = _ORIG["group_by_expert"](sel, n_experts)
    out = table.copy()
    for e in range(n_experts):
        out[bounds[e]:bounds[e + 1]] = table[bounds[e]:bounds[e + 1]][::-1]
    return out, bounds


def _moe_unweighted(x, logits, experts, top_k):
    sel, _ = _ORIG["route_topk"](logits, top_k)
    out = x.copy()
    for t in range(x.shape[0]):
        for e in sel[t]:
            out[t] += F.swiglu_mlp(x[t:t + 1], *experts(int(e)))[0]
    return out


_ORIG = {n: getattr(F, n) for n in ("gelu", "silu", "linear", "ffn_gelu", "ffn_gelu_proj",
                                    "swiglu", "swiglu_mlp", "route_topk", "group_by_expert",
                                    "moe_swiglu")}

MUTATIONS = {
    "gelu_missing_sqrt2": {"gelu": _gelu_no_sqrt2},
    "gelu_tanh_approx": {"gelu": _gelu_tanh},
    "silu_sign": {"silu": _silu_sign},
    "linear_drops_bias": {"linear": _linear_no_bias},
    "linear_transposed": {"linear": _linear_transposed},
    "ffn_drops_residual": {"ffn_gelu": _ffn_no_residual},
    "proj_residual_from_u": {"ffn_gelu_proj": _ffn_proj_wrong_residual},
    "swiglu_gate_up_swapped": {"swiglu": _swiglu_swapped, "swiglu_mlp": _swiglu_mlp_swapped},
    "topk_ties_to_high_index": {"route_topk": _route_ties_high},
    "softmax_over_all_experts": {"route_topk": _route_full_softmax},
    "grouping_not_stable": {"group_by_expert": _group_reversed},
    "moe_drops_weights": {"moe_swiglu": _moe_unweighted},
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_mutation_is_caught(name, monkeypatch):
    for attr, fn in MUTATIONS[name].items():
        monkeypatch.setattr(F, attr, fn)
    caught = []
    for check in P.ALL_CHECKS:
        try:
            check(F)
        except (AssertionError, ValueError) as e:
            caught.append(check.__name__)
    assert caught, f"no pin caught the planted mistake {name}"
