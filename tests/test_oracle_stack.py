"""The oracle's whole-stack composition (oracle/stack.py) against a loop written out by
hand over the segment functions of oracle/forward.py, for all five kinds.

The hand loop takes each segment's tensors from one draw of the whole segment, and each
MoE layer's router logits straight from the documented stream (seed, 1_000_000 + layer),
so a composition that reuses one segment's tensors or one layer's logits, skips or
reorders segments, or applies the shared projection wrongly does not match it. Planted
mistakes below check that. No GPU.
"""
import types

import numpy as np
import pytest

import synth
from oracle import forward as F
from oracle import stack as S

KINDS = {
    "linear_gelu_f32": synth.TINY.with_(n_segments=3, tokens=5, hidden=12, ffn=12),
    "ffn_gelu": synth.DIT.with_(n_segments=3, tokens=5, hidden=16, ffn=24),
    "ffn_gelu_shared": synth.SHARED.with_(n_segments=3, tokens=5, hidden=16, ffn=24),
    "swiglu": synth.LARGE.with_(n_segments=3, tokens=5, hidden=16, ffn=24),
    "moe": synth.MOE.with_(n_segments=3, tokens=9, hidden=16, ffn=8, n_experts=5, top_k=2),
}


def _logits(cfg, layer):
    rng = np.random.default_rng(np.random.SeedSequence([cfg.seed, 1_000_000 + layer]))
    return rng.standard_normal((cfg.tokens, cfg.n_experts), dtype=np.float32)


def _hand_stack(cfg):
    """y = seg_{N-1}( ... seg_1(seg_0(x)) ), each segment with its own tensors."""
    specs = synth.segment_tensors(cfg)
    x = F.as_f64(synth.draw_x(cfg), cfg.dtype)
    if cfg.kind == synth.KIND_FFN_GELU_SHARED_BF16:
        P = F.as_f64(synth.draw_shared(cfg)[0], "bf16")
    for s in range(cfg.n_segments):
        t = [F.as_f64(a, sp.dtype) for a, sp in zip(synth.draw_segment(cfg, s, threads=1), specs)]
        if cfg.kind == synth.KIND_LINEAR_GELU_F32:
            x = F.linear_gelu(x, t[0], t[1])
        elif cfg.kind == synth.KIND_FFN_GELU_BF16:
            x = F.ffn_gelu(x, t[0], t[1], t[2], t[3])
        elif cfg.kind == synth.KIND_FFN_GELU_SHARED_BF16:
            x = F.ffn_gelu_proj(x, P, t[0], t[1], t[2], t[3])
        elif cfg.kind == synth.KIND_SWIGLU_BF16:
            x = F.swiglu(x, t[0], t[1], t[2])
        else:
            x = F.moe_swiglu(x, _logits(cfg, s), lambda e: t[3 * e:3 * e + 3], cfg.top_k)
    return x


@pytest.mark.parametrize("name", sorted(KINDS))
def test_stack_equals_hand_written_loop(name):
    cfg = KINDS[name]
    ref = _hand_stack(cfg)
    np.testing.assert_allclose(S.stack_forward(cfg), ref, rtol=1e-12, atol=1e-12)
    rows = np.array([4, 0, 2])
    np.testing.assert_allclose(S.stack_forward(cfg, rows=rows), ref[rows], rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("name", sorted(KINDS))
def test_segments_and_layers_are_distinct(name):
    """The pin above only bites if the segments differ: their tensors (and the MoE layers'
    logits) are distinct draws, and every segment changes the activations."""
    cfg = KINDS[name]
    a, b = synth.draw_segment(cfg, 0, threads=1), synth.draw_segment(cfg, 1, threads=1)
    assert not np.array_equal(a[0], b[0])
    if cfg.kind == synth.KIND_MOE_SWIGLU_BF16:
        assert not np.array_equal(_logits(cfg, 0), _logits(cfg, 1))
    y1 = S.stack_forward(cfg, n_segments=1)
    y2 = S.stack_forward(cfg, n_segments=2)
    assert np.max(np.abs(y2 - y1)) > 1e-3


# ------------------------------------------------------------------ planted mistakes
def _synth_proxy(**over):
    """A stand-in for the synth module inside oracle.stack with some draws replaced."""
    ns = types.SimpleNamespace(**{k: getattr(synth, k) for k in dir(synth) if not k.startswith("__")})
    for k, v in over.items():
        setattr(ns, k, v)
    return ns


def _every_segment_is_zero(cfg, segment, *a, **k):
    return synth.draw_segment(cfg, 0, *a, **k)


def _every_expert_from_layer_zero(cfg, layer, expert):
    return synth.draw_expert(cfg, 0, expert)


def _every_layer_logits_zero(cfg, layer, tokens=None):
    return synth.draw_logits(cfg, 0, tokens)


def _reversed_stack(cfg, rows=None, x=None, n_segments=None, logits=None):
    xa = synth.draw_x(cfg)
    x = F.as_f64(xa if rows is None else xa[rows], cfg.dtype)
    shared = S.shared_f64(cfg)[0] if cfg.kind == synth.KIND_FFN_GELU_SHARED_BF16 else None
    for s in reversed(range(cfg.n_segments)):
        x = S.apply_segment(cfg, s, x, rows=rows, shared=shared)
    return x


def _skips_last_segment(cfg, rows=None, x=None, n_segments=None, logits=None):
    return _ORIG_STACK(cfg, rows=rows, x=x, n_segments=cfg.n_segments - 1, logits=logits)


_ORIG_STACK = S.stack_forward

PLANTED = {
    "segment_zero_tensors_everywhere": ("synth", dict(draw_segment=_every_segment_is_zero,
                                                      draw_expert=_every_expert_from_layer_zero)),
    "layer_zero_logits_everywhere": ("synth", dict(draw_logits=_every_layer_logits_zero)),
    "segments_in_reverse": ("stack_forward", _reversed_stack),
    "last_segment_skipped": ("stack_forward", _skips_last_segment),
}


@pytest.mark.parametrize("mistake", sorted(PLANTED))
def test_planted_composition_mistake_is_caught(mistake, monkeypatch):
    what, repl = PLANTED[mistake]
    if what == "synth":
        monkeypatch.setattr(S, "synth", _synth_proxy(**repl))
    else:
        monkeypatch.setattr(S, what, repl)
    caught = []
    for name in sorted(KINDS):
        try:
            test_stack_equals_hand_written_loop(name)
        except AssertionError:
            caught.append(name)
    assert caught, f"no kind caught the planted mistake {mistake}"
    if mistake == "layer_zero_logits_everywhere":
        assert caught == ["moe"]
    elif mistake != "segments_in_reverse":
        assert len(caught) == len(KINDS), caught
