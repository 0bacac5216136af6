"""Plain fp64 forward of the streamed segment kinds (oracle; test infrastructure only).

Layer streaming changes where the weights live, not what is computed: the pages
check pool against non-pool runs with zero differing output channels
("feat: pool VRAM for streamed layer", Verification) and matching output hashes
across residency and prefetch settings ("feat: prefetch streamed layers during
compute", Verification). So the oracle is the all-resident forward written out
from its definition, in float64, with no intermediate rounding.

Segment functions (weights row-major [out, in], activations [tokens, hidden]):
  linear_gelu    y = GELU(x W^T + b)                             (fp32 tiny stack)
  ffn_gelu       y = x + GELU(x W1^T + b1) W2^T + b2             (DiT-style FFN)
  ffn_gelu_proj  y = x + GELU((x P^T) W1^T + b1) W2^T + b2       (shared projection P)
  swiglu         y = x + (SiLU(x G^T) * (x U^T)) D^T             (gate / up / down)
  moe_swiglu     y = x + sum_k w_k * SwiGLU_{e_k}(x)            (top-k routed experts)

GELU is the exact erf form, SiLU(z) = z / (1 + e^-z). MoE routing follows the
expert grouping of "prefill: a layer split's idle card streams a share of a
one-chunk prompt's experts" (What): top-k experts per token from the router
logits, a row table and group bounds that group the (token, k) rows by expert,
one SwiGLU per expert over its rows, then a weighted combine. The softmax is
taken over the k selected logits; the k order is descending logit with ties to
the lower expert index.
"""
from __future__ import annotations

import math

import numpy as np
from scipy.special import erf

_INV_SQRT2 = 1.0 / math.sqrt(2.0)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) to float64, exactly."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def as_f64(a: np.ndarray, dtype: str) -> np.ndarray:
    """Exact float64 view of a stored tensor ("f32" array or "bf16" bit patterns)."""
    return bf16_bits_to_f64(a) if dtype == "bf16" else np.asarray(a, np.float32).astype(np.float64)


def gelu(z: np.ndarray) -> np.ndarray:
    """GELU(z) = z * Phi(z) = z/2 * (1 + erf(z / sqrt 2))."""
    return 0.5 * z * (1.0 + erf(z * _INV_SQRT2))


def silu(z: np.ndarray) -> np.ndarray:
    """SiLU(z) = z / (1 + exp(-z)), computed without overflow for large |z|."""
    z = np.asarray(z, np.float64)
    out = np.empty_like(z)
    pos = z >= 0
    out[pos] = z[pos] / (1.0 + np.exp(-z[pos]))
    ez = np.exp(z[~pos])
    out[~pos] = z[~pos] * ez / (1.0 + ez)
    return out


def linear(x: np.ndarray, w: np.ndarray, b: np.ndarray | None = None) -> np.ndarray:
    """x W^T (+ b) with W stored [out, in]."""
    y = x @ w.T
    if b is not None:
        y = y + b
    return y


def linear_gelu(x, w, b):
    """Tiny fp32 stack segment: GELU(x W^T + b)."""
    return gelu(linear(x, w, b))


def ffn_gelu(x, w1, b1, w2, b2):
    """DiT-style FFN segment with residual: x + GELU(x W1^T + b1) W2^T + b2."""
    return x + linear(gelu(linear(x, w1, b1)), w2, b2)


def ffn_gelu_proj(x, p, w1, b1, w2, b2):
    """FFN segment behind a shared projection P (applied first, no bias):
    x + GELU((x P^T) W1^T + b1) W2^T + b2."""
    u = linear(x, p)
    return x + linear(gelu(linear(u, w1, b1)), w2, b2)


def swiglu_mlp(x, g, u, d):
    """(SiLU(x G^T) * (x U^T)) D^T — the gate / up / down MLP without residual."""
    return linear(silu(linear(x, g)) * linear(x, u), d)


def swiglu(x, g, u, d):
    """Gate/up/down segment with residual: x + (SiLU(x G^T) * (x U^T)) D^T."""
    return x + swiglu_mlp(x, g, u, d)


def route_topk(logits: np.ndarray, k: int):
    """Top-k experts per token and their softmax weights.

    Selection compares the float32 logits as given (descending, ties to the
    lower expert index); the weights are a float64 softmax over the k selected
    logits, in selection order. Returns (sel int32 [T, k], w float64 [T, k]).
    """
    lg = np.asarray(logits, np.float32)
    order = np.argsort(-lg, axis=1, kind="stable")[:, :k]
    sel = order.astype(np.int32)
    chosen = np.take_along_axis(lg, order, axis=1).astype(np.float64)
    m = chosen.max(axis=1, keepdims=True)
    e = np.exp(chosen - m)
    return sel, e / e.sum(axis=1, keepdims=True)


def group_by_expert(sel: np.ndarray, n_experts: int):
    """Row table and group bounds: the (token, k) rows, numbered t*k_total + k,
    grouped by expert with a stable counting sort (rows of one expert stay in
    (t, k) order). Returns (row_table int32 [T*k], group_bounds int32 [E+1])."""
    flat = np.asarray(sel, np.int64).reshape(-1)
    row_table = np.argsort(flat, kind="stable").astype(np.int32)
    counts = np.bincount(flat, minlength=n_experts)
    bounds = np.zeros(n_experts + 1, np.int64)
    np.cumsum(counts, out=bounds[1:])
    return row_table, bounds.astype(np.int32)


def moe_swiglu(x, logits, experts, top_k):
    """MoE SwiGLU layer with residual.

    ``experts(e)`` returns (G_e, U_e, D_e) as float64. Steps in the order the
    expert-grouping description gives them: route, group rows by expert, run
    each expert's MLP over its rows, combine with the routing weights.
    """
    T = x.shape[0]
    sel, w = route_topk(logits, top_k)
    row_table, bounds = group_by_expert(sel, logits.shape[1])
    contrib = np.zeros((T, top_k, x.shape[1]), np.float64)
    for e in range(logits.shape[1]):
        rows = row_table[bounds[e]:bounds[e + 1]]
        if rows.size == 0:
            continue
        t_idx, k_idx = rows // top_k, rows % top_k
        g, u, d = experts(e)
        ye = swiglu_mlp(x[t_idx], g, u, d)
        contrib[t_idx, k_idx] = w[t_idx, k_idx][:, None] * ye
    return x + contrib.sum(axis=1)
