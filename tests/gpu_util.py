"""Helpers shared by the GPU tests (marshalling only)."""
import numpy as np
import torch

import synth
from host_offloaded_weight_gb300 import lstream as L
from oracle import forward as F

BOUND = 1e-2  # max|gpu - ref| / max|ref| per stack output


def bf16_dev(bits: np.ndarray) -> torch.Tensor:
    """uint16 bf16 patterns -> bf16 CUDA tensor."""
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def rand_bf16(shape, seed, scale=1.0):
    r = np.random.default_rng(seed)
    bits = synth.f32_to_bf16_bits(r.standard_normal(shape).astype(np.float32) * np.float32(scale))
    return bits, F.bf16_bits_to_f64(bits)


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def rel_err(got, ref) -> float:
    return float(np.max(np.abs(got - ref)) / max(np.max(np.abs(ref)), 1e-30))


def x_dev(cfg, tokens=None):
    x = synth.draw_x(cfg, tokens)
    if cfg.dtype == "f32":
        return torch.from_numpy(x).cuda()
    return bf16_dev(x)


def make_ctx(cfg, hs, **over):
    kw = dict(prefetch_depth=cfg.prefetch_depth, resident_layers=cfg.resident_layers,
              max_vram_bytes=cfg.max_vram_bytes, use_pool=cfg.use_pool, wait_limit_ms=5000)
    kw.update(over)
    ctx = L.ls_ctx_create(L.ls_params_init(**kw))
    try:
        st = L.ls_register_segments(ctx, hs.segments, hs.shared_map)
    except Exception:
        L.ls_ctx_destroy(ctx)
        raise
    return ctx, st


def logits_dev(cfg, tokens=None, n_layers=None):
    n = cfg.n_segments if n_layers is None else n_layers
    lg = np.stack([synth.draw_logits(cfg, l, tokens) for l in range(n)])
    return torch.from_numpy(lg).cuda(), lg
