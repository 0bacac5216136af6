"""Whole-stack fp64 forward over a sample of token rows (oracle; test infrastructure only).

Every segment kind here acts on each token row independently (the MoE router
logits are inputs, not functions of the activations), so the forward of a row
subset equals those rows of the full forward. That lets the oracle check the
full-size stacks on sampled rows.
"""
from __future__ import annotations

import numpy as np

import synth
from . import forward as F


def segment_f64(cfg, seg: int):
    """Draw one segment's private tensors and widen them to float64."""
    specs = synth.segment_tensors(cfg)
    return [F.as_f64(a, s.dtype) for a, s in zip(synth.draw_segment(cfg, seg), specs)]


def shared_f64(cfg):
    return [F.as_f64(a, s.dtype) for a, s in zip(synth.draw_shared(cfg), synth.shared_tensors(cfg))]


def apply_segment(cfg, seg: int, x: np.ndarray, rows=None, tensors=None, shared=None, logits=None):
    """y = segment_seg(x) for the given rows of the stack's token set. ``logits``: this
    MoE layer's router logits for all tokens (default: the drawn ones)."""
    k = cfg.kind
    if k == synth.KIND_MOE_SWIGLU_BF16:
        if logits is None:
            logits = synth.draw_logits(cfg, seg)
        if rows is not None:
            logits = logits[rows]
        cache: dict = {}

        def expert(e):
            if e not in cache:
                specs = synth.segment_tensors(cfg)[3 * e:3 * e + 3]
                cache[e] = [F.as_f64(a, s.dtype) for a, s in
                            zip(synth.draw_expert(cfg, seg, e), specs)]
            return cache[e]
        return F.moe_swiglu(x, logits, expert, cfg.top_k)
    t = tensors if tensors is not None else segment_f64(cfg, seg)
    if k == synth.KIND_LINEAR_GELU_F32:
        return F.linear_gelu(x, *t)
    if k == synth.KIND_FFN_GELU_BF16:
        return F.ffn_gelu(x, *t)
    if k == synth.KIND_FFN_GELU_SHARED_BF16:
        p = shared if shared is not None else shared_f64(cfg)[0]
        return F.ffn_gelu_proj(x, p, *t)
    if k == synth.KIND_SWIGLU_BF16:
        return F.swiglu(x, *t)
    raise ValueError(k)


def stack_forward(cfg, rows=None, x=None, n_segments=None, logits=None):
    """fp64 output of the stack for token ``rows`` (all rows when None).

    ``x`` overrides the drawn input (float64 [len(rows), hidden]); ``logits`` the MoE router
    logits ([layers] of [tokens, experts])."""
    if x is None:
        xa = synth.draw_x(cfg)
        if rows is not None:
            xa = xa[rows]
        x = F.as_f64(xa, cfg.dtype)
    shared = shared_f64(cfg)[0] if cfg.kind == synth.KIND_FFN_GELU_SHARED_BF16 else None
    for s in range(cfg.n_segments if n_segments is None else n_segments):
        x = apply_segment(cfg, s, x, rows=rows, shared=shared,
                          logits=None if logits is None else logits[s])
    return x
