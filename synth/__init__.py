"""Seeded synthetic layer stacks for layer-streamed execution.

This module only draws random numbers and lays them out; it holds none of the
arithmetic of the method (no activation, no matmul, no routing, no policy).
Both the CUDA path (through the tests and ``bench.py``) and the CPU oracle take
their inputs from here, so they see exactly the same bytes.

Recipe (one stream per tensor):
  * generator: ``numpy.random.default_rng(SeedSequence([seed, segment, index]))``
    drawing ``standard_normal`` in float32, in row-major order;
  * weights and biases are multiplied (in float32) by ``1/sqrt(fan_in)`` of the
    linear they belong to, so they are N(0, std = 1/sqrt(fan_in)); the down
    projection D of the gate/up/down kinds (dense and per expert) also carries a
    depth factor ``1/sqrt(n_segments)``: with plain 1/sqrt(fan_in) the residual
    stream of a SwiGLU stack grows quadratically per layer and overflows float
    range within a dozen layers (the product of two N(0, v) projections has
    variance ~ v^2);
  * activations ``x`` are N(0, 1) from ``SeedSequence([seed, 2_000_000, 0])``;
  * MoE router logits for layer ``l`` are N(0, 1) float32 from
    ``SeedSequence([seed, 1_000_000 + l])``, shape ``[tokens, experts]``;
  * bf16 tensors are the float32 draws rounded to nearest-even bf16 and stored
    as their 16-bit patterns (``numpy.uint16``);
  * the tensor order inside a segment is W1, b1, W2, b2 (FFN kinds), W, b
    (fp32 linear), G, U, D (SwiGLU) and expert-major G_e, U_e, D_e (MoE);
  * the shared projection of the shared-projection stack is drawn as segment
    ``SHARED_SEGMENT_ID``, index 0.

Weights are row-major ``[out, in]`` (PyTorch's linear layout); activations are
``[tokens, hidden]`` row-major.
"""
from __future__ import annotations

import math
import mmap
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field, replace

import numpy as np

SHARED_SEGMENT_ID = 10_000
X_STREAM = 2_000_000
LOGIT_STREAM = 1_000_000
GIB = 1 << 30

# Segment kinds (the numeric values are part of the C ABI, see include/ls_api.h).
KIND_LINEAR_GELU_F32 = 0
KIND_FFN_GELU_BF16 = 1
KIND_FFN_GELU_SHARED_BF16 = 2
KIND_SWIGLU_BF16 = 3
KIND_MOE_SWIGLU_BF16 = 4

_CHUNK = 1 << 22  # values per draw call; chunked draws reproduce the one-shot stream


@dataclass(frozen=True)
class TensorSpec:
    name: str
    shape: tuple
    dtype: str          # "f32" or "bf16"
    fan_in: int
    index: int          # stream index inside the segment
    gain: float = 1.0   # extra factor on top of 1/sqrt(fan_in)

    @property
    def numel(self) -> int:
        return int(np.prod(self.shape))

    @property
    def nbytes(self) -> int:
        return self.numel * (4 if self.dtype == "f32" else 2)


@dataclass(frozen=True)
class StackConfig:
    """One synthetic layer stack plus the streaming parameters it is run with."""
    name: str
    kind: int
    n_segments: int
    tokens: int
    hidden: int
    ffn: int
    dtype: str                      # activation / weight dtype: "f32" or "bf16"
    prefetch_depth: int = 1
    resident_layers: int = 0
    max_vram_bytes: int = 0
    use_pool: int = 1
    n_experts: int = 0
    top_k: int = 0
    seed: int = 0
    shared_proj: bool = False
    notes: str = ""

    def with_(self, **kw) -> "StackConfig":
        return replace(self, **kw)


def segment_tensors(cfg: StackConfig) -> list:
    """Private tensors of one segment, in registration order."""
    h, f = cfg.hidden, cfg.ffn
    k = cfg.kind
    if k == KIND_LINEAR_GELU_F32:
        return [TensorSpec("W", (f, h), "f32", h, 0), TensorSpec("b", (f,), "f32", h, 1)]
    if k in (KIND_FFN_GELU_BF16, KIND_FFN_GELU_SHARED_BF16):
        return [TensorSpec("W1", (f, h), "bf16", h, 0), TensorSpec("b1", (f,), "bf16", h, 1),
                TensorSpec("W2", (h, f), "bf16", f, 2), TensorSpec("b2", (h,), "bf16", f, 3)]
    depth_gain = 1.0 / math.sqrt(cfg.n_segments)
    if k == KIND_SWIGLU_BF16:
        return [TensorSpec("G", (f, h), "bf16", h, 0), TensorSpec("U", (f, h), "bf16", h, 1),
                TensorSpec("D", (h, f), "bf16", f, 2, depth_gain)]
    if k == KIND_MOE_SWIGLU_BF16:
        out = []
        for e in range(cfg.n_experts):
            out += [TensorSpec(f"G{e}", (f, h), "bf16", h, 3 * e),
                    TensorSpec(f"U{e}", (f, h), "bf16", h, 3 * e + 1),
                    TensorSpec(f"D{e}", (h, f), "bf16", f, 3 * e + 2, depth_gain)]
        return out
    raise ValueError(f"unknown kind {k}")


def shared_tensors(cfg: StackConfig) -> list:
    if cfg.kind == KIND_FFN_GELU_SHARED_BF16:
        return [TensorSpec("P", (cfg.hidden, cfg.hidden), "bf16", cfg.hidden, 0)]
    return []


def align256(n: int) -> int:
    return (n + 255) // 256 * 256


def segment_slot_bytes(cfg: StackConfig) -> int:
    """Footprint of one segment's private tensors packed at 256-byte offsets."""
    return sum(align256(t.nbytes) for t in segment_tensors(cfg))


def stack_bytes(cfg: StackConfig) -> int:
    """Bytes of a HostStack's buffer: every segment's footprint, then the shared tensors."""
    return cfg.n_segments * segment_slot_bytes(cfg) + sum(align256(t.nbytes) for t in shared_tensors(cfg))


# ---------------------------------------------------------------- the stacks
def _tiny() -> StackConfig:
    s = 256 * 256 * 4 + 256 * 4
    return StackConfig("tiny_f32_4x256", KIND_LINEAR_GELU_F32, 4, 8, 256, 256, "f32",
                       prefetch_depth=1, resident_layers=0, max_vram_bytes=2 * s, use_pool=1,
                       notes="4 x fp32 linear 256x256 + bias + GELU, 8 tokens")


def _dit() -> StackConfig:
    c = StackConfig("dit_ffn_12x1024x4096", KIND_FFN_GELU_BF16, 12, 4096, 1024, 4096, "bf16",
                    prefetch_depth=1, resident_layers=0, use_pool=1,
                    notes="12 x bf16 FFN 1024->4096->1024 + GELU + residual, 4096 tokens")
    return c.with_(max_vram_bytes=2 * segment_slot_bytes(c))


def _shared() -> StackConfig:
    return StackConfig("shared_proj_24x3072x12288", KIND_FFN_GELU_SHARED_BF16, 24, 2048, 3072,
                       12288, "bf16", prefetch_depth=1, resident_layers=-1,
                       max_vram_bytes=2 * GIB, use_pool=1, shared_proj=True,
                       notes="24 x bf16 FFN 3072->12288->3072, one shared 3072x3072 "
                             "projection, 2048 tokens")


def _large() -> StackConfig:
    return StackConfig("swiglu_48x5120x13824", KIND_SWIGLU_BF16, 48, 512, 5120, 13824, "bf16",
                       prefetch_depth=2, resident_layers=4, max_vram_bytes=4 * GIB, use_pool=1,
                       notes="48 x bf16 SwiGLU gate/up/down 5120x13824, 512 tokens")


def _moe() -> StackConfig:
    c = StackConfig("moe_48x128x2048x768", KIND_MOE_SWIGLU_BF16, 48, 2048, 2048, 768, "bf16",
                    prefetch_depth=1, resident_layers=0, use_pool=1, n_experts=128, top_k=8,
                    notes="48 MoE layers, 128 experts 2048->768->2048 SwiGLU, top-8, "
                          "2048 tokens")
    return c.with_(max_vram_bytes=2 * segment_slot_bytes(c))


STACKS = {c.name: c for c in (_tiny(), _dit(), _shared(), _large(), _moe())}
TINY, DIT, SHARED, LARGE, MOE = (STACKS[n] for n in STACKS)


# ---------------------------------------------------------------- drawing
def _draw_f32_into(out_f32: np.ndarray, seq: list, scale: float) -> None:
    rng = np.random.default_rng(np.random.SeedSequence(seq))
    flat = out_f32.reshape(-1)
    sc = np.float32(scale)
    for i in range(0, flat.size, _CHUNK):
        v = flat[i:i + _CHUNK]
        rng.standard_normal(out=v, dtype=np.float32)
        if scale != 1.0:
            np.multiply(v, sc, out=v)


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 to the nearest bf16 (ties to even); returns the bit patterns."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def _draw_bf16_into(out_u16: np.ndarray, seq: list, scale: float) -> None:
    rng = np.random.default_rng(np.random.SeedSequence(seq))
    flat = out_u16.reshape(-1)
    tmp = np.empty(min(_CHUNK, flat.size), np.float32)
    sc = np.float32(scale)
    for i in range(0, flat.size, _CHUNK):
        n = min(_CHUNK, flat.size - i)
        v = tmp[:n]
        rng.standard_normal(out=v, dtype=np.float32)
        if scale != 1.0:
            np.multiply(v, sc, out=v)
        flat[i:i + n] = f32_to_bf16_bits(v)


def tensor_seq(cfg: StackConfig, segment: int, spec: TensorSpec) -> list:
    return [cfg.seed, segment, spec.index]


def draw_tensor(cfg: StackConfig, segment: int, spec: TensorSpec, out: np.ndarray | None = None):
    """Draw one tensor. fp32 tensors come back as float32, bf16 as uint16 bit patterns."""
    scale = spec.gain / math.sqrt(spec.fan_in)
    if spec.dtype == "f32":
        if out is None:
            out = np.empty(spec.shape, np.float32)
        _draw_f32_into(out, tensor_seq(cfg, segment, spec), scale)
    else:
        if out is None:
            out = np.empty(spec.shape, np.uint16)
        _draw_bf16_into(out, tensor_seq(cfg, segment, spec), scale)
    return out


def draw_segment(cfg: StackConfig, segment: int, outs: list | None = None, threads: int = 0):
    """Draw every private tensor of one segment (optionally into given buffers)."""
    specs = segment_tensors(cfg)
    if outs is None:
        outs = [None] * len(specs)
    threads = threads or min(len(specs), os.cpu_count() or 1)
    if threads <= 1 or len(specs) == 1:
        return [draw_tensor(cfg, segment, s, o) for s, o in zip(specs, outs)]
    with ThreadPoolExecutor(threads) as ex:
        return list(ex.map(lambda so: draw_tensor(cfg, segment, so[0], so[1]), zip(specs, outs)))


def draw_shared(cfg: StackConfig, outs: list | None = None):
    specs = shared_tensors(cfg)
    outs = outs or [None] * len(specs)
    return [draw_tensor(cfg, SHARED_SEGMENT_ID, s, o) for s, o in zip(specs, outs)]


def draw_x(cfg: StackConfig, tokens: int | None = None):
    """Input activations [tokens, hidden]: float32 for fp32 stacks, bf16 bits otherwise."""
    t = cfg.tokens if tokens is None else tokens
    spec = TensorSpec("x", (t, cfg.hidden), cfg.dtype, 1, 0)
    out = np.empty(spec.shape, np.float32 if cfg.dtype == "f32" else np.uint16)
    seq = [cfg.seed, X_STREAM, 0]
    if cfg.dtype == "f32":
        _draw_f32_into(out, seq, 1.0)
    else:
        _draw_bf16_into(out, seq, 1.0)
    return out


def draw_logits(cfg: StackConfig, layer: int, tokens: int | None = None) -> np.ndarray:
    """Router logits of one MoE layer, float32 [tokens, experts]."""
    t = cfg.tokens if tokens is None else tokens
    out = np.empty((t, cfg.n_experts), np.float32)
    _draw_f32_into(out, [cfg.seed, LOGIT_STREAM + layer], 1.0)
    return out


def draw_expert(cfg: StackConfig, layer: int, expert: int):
    """The three tensors (G, U, D) of one expert of one MoE layer."""
    specs = segment_tensors(cfg)[3 * expert:3 * expert + 3]
    return [draw_tensor(cfg, layer, s) for s in specs]


# ---------------------------------------------------------------- host layout
class HostStack:
    """A whole stack drawn into one page-aligned host buffer.

    Each segment's private tensors sit at 256-byte aligned offsets in the
    segment's region, in registration order (the same packing as a device
    slot); the shared tensors follow the last segment. ``segments`` is a list of
    (kind, [numpy views]) and ``shared_map`` a list of
    (segment, tensor_index, shared_id), the shapes the C ABI registers.
    bf16 tensors are uint16 views holding the bit patterns."""

    def __init__(self, cfg: StackConfig, n_segments: int | None = None, threads: int = 0, alloc=None,
                 draw: bool = True):
        """``alloc(nbytes) -> (address, release)``, optional: where the buffer lives (for example
        pinned memory from a driver allocator, or memory another process shares); ``release()``
        is called by ``close()``. Default: anonymous pages of the process. ``draw=False`` lays
        the views over a buffer that already holds the stack (drawn by another process)."""
        self.cfg = cfg
        n = cfg.n_segments if n_segments is None else n_segments
        specs = segment_tensors(cfg)
        sh = shared_tensors(cfg)
        seg_bytes = segment_slot_bytes(cfg)
        sh_bytes = sum(align256(t.nbytes) for t in sh)
        total = n * seg_bytes + sh_bytes
        self._release = None
        self._map = None
        if alloc is not None:
            import ctypes
            addr, self._release = alloc(max(total, 1))
            self.buffer = np.ctypeslib.as_array((ctypes.c_uint8 * max(total, 1)).from_address(addr))[:total]
        else:
            # anonymous pages of its own: nothing else lives in the buffer's pages. Large
            # pages where the kernel offers them on request: fewer translations for the
            # device's reads of pinned host memory (a hint; ignored where unsupported)
            self._map = mmap.mmap(-1, max(total, 1))
            if hasattr(mmap, "MADV_HUGEPAGE") and total >= (64 << 20):
                try:
                    self._map.madvise(mmap.MADV_HUGEPAGE)
                except OSError:
                    pass
            self.buffer = np.frombuffer(self._map, dtype=np.uint8, count=total)
        self.shared_views = []
        o = n * seg_bytes
        for t in sh:
            self.shared_views.append(self._view(o, t))
            o += align256(t.nbytes)
        self.seg_views = []
        jobs = []
        for s in range(n):
            o = s * seg_bytes
            views = []
            for t in specs:
                v = self._view(o, t)
                views.append(v)
                jobs.append((s, t, v))
                o += align256(t.nbytes)
            self.seg_views.append(views)
        jobs += [(SHARED_SEGMENT_ID, t, v) for t, v in zip(sh, self.shared_views)]
        threads = threads or (os.cpu_count() or 1)
        if draw:
            with ThreadPoolExecutor(threads) as ex:
                list(ex.map(lambda j: draw_tensor(cfg, j[0], j[1], j[2]), jobs))
        self.segments = []
        self.shared_map = []
        for s in range(n):
            tensors = list(self.seg_views[s])
            if sh:
                tensors = list(self.shared_views) + tensors
                for i in range(len(sh)):
                    self.shared_map.append((s, i, i))
            self.segments.append((cfg.kind, tensors))

    def close(self) -> None:
        """Give the buffer back now (views into it must no longer be used)."""
        self.seg_views, self.shared_views, self.segments = [], [], []
        self.buffer = None
        if self._release is not None:
            self._release()
            self._release = None
        if self._map is not None:
            try:
                self._map.close()
            except BufferError:   # a view is still alive; the mapping goes with the last one
                pass
            self._map = None

    def _view(self, off: int, t: TensorSpec) -> np.ndarray:
        dt = np.float32 if t.dtype == "f32" else np.uint16
        return self.buffer[off:off + t.nbytes].view(dt).reshape(t.shape)
