#!/usr/bin/env python
"""Layer-streamed execution benchmark (one JSON line on stdout, rank 0).

Workload (default): the 48-layer MoE prefill stack - per layer 128 experts, each
a bf16 SwiGLU 2048->768->2048 (9.4 MB), top-8 routing of 2048 tokens from N(0,1)
router logits - with its 58 GB of experts in pinned host memory, prefetch depth 1,
no residents, a two-slot pool of 1.2 GB slots. One step = one streamed pass over
all 48 layers: each layer's routed experts cross the host link again, tokens are
grouped by expert and run through the grouped GEMMs. The other stacks run with
--workload. Inputs are synthetic (seeded N(0,1) activations, N(0, 1/sqrt(fan_in))
weights).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

N > 1 runs N independent replicas (one process per GPU under torchrun): the
path has no exchange step, so the ranks share nothing but the barrier and the
max-over-ranks timing (and, when N copies of the host stack would not fit the
host's memory, one read-only host stack per node). --impl reference times the CPU
fp64 oracle instead.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "streamed tokens/s; overlap eff. vs max(H2D,compute); host-link GB/s"
UNIT = "tokens/s"
FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS = 6800.0, 1900.0
L2_FLUSH_BYTES = 256 << 20
L2_BYTES = 129 << 20          # GB300 L2, when the device properties do not report it


def seg_flops(cfg, tokens) -> float:
    """Multiply-add FLOPs of one segment (the GEMMs)."""
    T, H, F = tokens, cfg.hidden, cfg.ffn
    if cfg.kind == synth.KIND_LINEAR_GELU_F32:
        return 2.0 * T * H * F
    if cfg.kind == synth.KIND_FFN_GELU_BF16:
        return 4.0 * T * H * F
    if cfg.kind == synth.KIND_FFN_GELU_SHARED_BF16:
        return 4.0 * T * H * F + 2.0 * T * H * H
    if cfg.kind == synth.KIND_SWIGLU_BF16:
        return 6.0 * T * H * F
    return 6.0 * T * cfg.top_k * H * F


def kernel_flops(cfg, tokens) -> dict:
    T, H, F = tokens, cfg.hidden, cfg.ffn
    if cfg.kind == synth.KIND_SWIGLU_BF16:
        return {"gemm_up": 4.0 * T * H * F, "gemm_down": 2.0 * T * H * F}
    if cfg.kind == synth.KIND_MOE_SWIGLU_BF16:
        return {"gemm_up": 4.0 * T * cfg.top_k * H * F, "gemm_down": 2.0 * T * cfg.top_k * H * F}
    return {"gemm_up": 2.0 * T * H * F, "gemm_down": 2.0 * T * H * F, "gemm_proj": 2.0 * T * H * H}


def kernel_bytes(cfg, tokens, routed=None) -> dict:
    """Algorithmic bytes one launch reads and writes: operands, bias, residual and outputs
    once each (bf16 = 2 B, fp32 = 4 B). routed = experts a MoE layer moves (default all)."""
    T, H, F = tokens, cfg.hidden, cfg.ffn
    if cfg.kind == synth.KIND_MOE_SWIGLU_BF16:
        e = cfg.n_experts if routed is None else routed
        rows = T * cfg.top_k
        return {"gemm_up": 2 * (rows * H + e * 2 * F * H + rows * F),
                "gemm_down": 2 * (rows * F + e * H * F) + 4 * rows * H}
    up_b = 2 * F * H * (2 if cfg.kind == synth.KIND_SWIGLU_BF16 else 1)
    out = {"gemm_up": 2 * T * H + up_b + 2 * F + 2 * T * F,
           "gemm_down": 2 * T * F + 2 * H * F + 2 * H + 4 * T * H + 2 * T * H + 4 * T * H}
    if cfg.kind != synth.KIND_SWIGLU_BF16:
        out["gemm_proj"] = 2 * T * H + 2 * H * H + 2 * T * H
    return out


def measured_peaks() -> tuple:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", 0)) or None, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, None, "fallback"


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.path = tempfile.mktemp(suffix=".csv")
        self.f = open(self.path, "w")
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", gpu_id, f"--query-gpu={self.FIELDS}",
                                       "--format=csv,noheader,nounits", "-lms", "200"],
                                      stdout=self.f, stderr=subprocess.DEVNULL)
        except FileNotFoundError:
            self.p = None

    def stop(self) -> dict:
        if self.p is not None:
            self.p.terminate()
            try:
                self.p.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.p.kill()
        self.f.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        os.remove(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- distributed glue
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def aggregate(step_seconds: float, units: float, world: int, device=None) -> tuple:
    """(max step time over ranks, total units over ranks): whole-job throughput
    is total units / max time. Works on gloo (CPU) and nccl."""
    if world == 1:
        return step_seconds, units
    import torch
    import torch.distributed as dist
    t = torch.tensor([step_seconds], dtype=torch.float64, device=device)
    u = torch.tensor([units], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


# ---------------------------------------------------------------- oracle (CPU) timing
# Bounded samples of each workload for the CPU oracle: (token rows, leading segments).
# Rows are independent in every kind and all segments of a stack have the same shapes,
# so the time of a sample scales to the whole stack by n_segments / segments sampled.
CPU_SAMPLE = {"tiny_f32_4x256": (8, None), "dit_ffn_12x1024x4096": (1024, None),
              "shared_proj_24x3072x12288": (256, 4), "swiglu_48x5120x13824": (512, 2),
              "moe_48x128x2048x768": (256, 1)}
E2E_BLOCK = 5   # steps per block of the alternating device-buffer / host-buffer measurement
REF_SAMPLE = {"tiny_f32_4x256": (8, None), "dit_ffn_12x1024x4096": (256, None),
              "shared_proj_24x3072x12288": (64, 2), "swiglu_48x5120x13824": (128, 1),
              "moe_48x128x2048x768": (128, 1)}


class OracleRun:
    """The fp64 oracle forward of the first `tokens` rows through the first `layers`
    segments of the stack.

    Only the oracle's arithmetic is timed: drawing the weights (or taking them from
    `hs`, the host stack the GPU streams from) and widening them to fp64 happen per
    segment before its timer starts, and the widened segments are kept between passes
    while they fit in CACHE_BYTES. For the MoE kind only the experts routed by the
    sampled rows are widened."""
    CACHE_BYTES = 8 << 30

    def __init__(self, cfg, tokens: int, layers=None, hs=None):
        from oracle import forward as F
        from oracle import stack as ostack
        self.cfg, self.F, self.ostack, self.hs = cfg, F, ostack, hs
        self.layers = cfg.n_segments if layers is None else min(layers, cfg.n_segments)
        self.rows = np.arange(tokens)
        self.x0 = F.as_f64(synth.draw_x(cfg, tokens), cfg.dtype)
        self.shared = ostack.shared_f64(cfg)[0] if cfg.kind == synth.KIND_FFN_GELU_SHARED_BF16 else None
        per_seg = sum(t.numel for t in synth.segment_tensors(cfg)) * 8
        self.cache = {} if per_seg * self.layers <= self.CACHE_BYTES else None
        self.moe = {}
        if cfg.kind == synth.KIND_MOE_SWIGLU_BF16:
            for s in range(self.layers):
                logits = synth.draw_logits(cfg, s)[self.rows]
                sel, _ = F.route_topk(logits, cfg.top_k)
                self.moe[s] = (logits, [int(e) for e in np.unique(sel)])

    @property
    def scale(self) -> float:
        """Whole-stack time over sample time (segments of one stack share their shapes)."""
        return self.cfg.n_segments / self.layers

    def _prepare(self, s):
        if self.cache is not None and s in self.cache:
            return self.cache[s]
        cfg = self.cfg
        if cfg.kind == synth.KIND_MOE_SWIGLU_BF16:
            logits, routed = self.moe[s]
            experts = {}
            for e in routed:
                bits = self.hs.seg_views[s][3 * e:3 * e + 3] if self.hs is not None else synth.draw_expert(cfg, s, e)
                experts[e] = [self.F.as_f64(np.asarray(b), "bf16") for b in bits]
            out = (logits, experts)
        elif self.hs is not None:
            out = [self.F.as_f64(np.asarray(a), sp.dtype)
                   for a, sp in zip(self.hs.seg_views[s], synth.segment_tensors(cfg))]
        else:
            out = self.ostack.segment_f64(cfg, s)
        if self.cache is not None:
            self.cache[s] = out
        return out

    def time_pass(self) -> float:
        """Seconds of the oracle's arithmetic over the sample."""
        cfg, F, x, total = self.cfg, self.F, self.x0, 0.0
        for s in range(self.layers):
            prep = self._prepare(s)
            t0 = time.perf_counter()
            if cfg.kind == synth.KIND_MOE_SWIGLU_BF16:
                logits, experts = prep
                x = F.moe_swiglu(x, logits, experts.__getitem__, cfg.top_k)
            else:
                x = self.ostack.apply_segment(cfg, s, x, rows=self.rows, tensors=prep, shared=self.shared)
            total += time.perf_counter() - t0
        return total

    def describe(self) -> str:
        what = f"{len(self.rows)} of {self.cfg.tokens} tokens through "
        if self.layers == self.cfg.n_segments:
            what += f"all {self.cfg.n_segments} segments"
        else:
            what += (f"the first {self.layers} of {self.cfg.n_segments} segments (same shapes), "
                     f"time scaled by {self.scale:g}")
        what += ", fp64; weight drawing and widening not timed"
        if self.cfg.kind == synth.KIND_MOE_SWIGLU_BF16:
            what += " (only the routed experts of the sampled rows are widened)"
        return what


def run_reference(args, cfg, world, rank):
    if rank != 0:
        return 0
    tokens, layers = REF_SAMPLE.get(cfg.name, (256, None))
    tokens = args.ref_tokens or tokens
    run = OracleRun(cfg, tokens, layers)
    for _ in range(args.warmup):
        run.time_pass()
    secs = [run.time_pass() * run.scale for _ in range(args.steps)]
    cores = len(os.sched_getaffinity(0))
    mean = statistics.mean(secs)
    value = tokens / mean
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": mean * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": cfg.name, "tokens": cfg.tokens, "segments": cfg.n_segments},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": run.describe()},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- GPU arm
def ce_link_peak(torch, nbytes=1 << 30, reps=10) -> float:
    """Pinned host -> device copy-engine bandwidth (best of reps), GB/s."""
    h = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    h.fill_(1)
    d = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    best = 1e30
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(s):
            e0.record()
            d.copy_(h, non_blocking=True)
            e1.record()
        e1.synchronize()
        best = min(best, e0.elapsed_time(e1))
    del h, d
    return nbytes / (best * 1e-3) / 1e9


def write_timeline(path, L, ctx, x, y, T, s, logits, cfg):
    """Two back-to-back passes with events around every copy and around each segment's
    compute kernels after its hand-off wait (launches keep programmatic dependent
    launch); the second pass per segment, in ms from its first event, with how busy the
    copy stream and the compute stream were."""
    L.ls_set_kernel_timing(ctx, 3)
    for _ in range(2):
        L.ls_run_async(ctx, x, y, T, s, logits=logits, top_k=cfg.top_k)
    L.ls_sync(ctx)
    trace = L.ls_get_trace(ctx)
    L.ls_set_kernel_timing(ctx, 0)
    L.ls_get_kernel_times(ctx, reset=True)
    second = trace[len(trace) // 2:]      # both passes record the same spans, in order
    t0 = min(e[3] for e in second)
    by_seg = {}
    for name, stream, seg, a, b in second:
        by_seg.setdefault(seg, []).append((name, stream, a - t0, b - t0))
    span = max(e[4] for e in second) - t0
    busy = {0: 0.0, 1: 0.0}
    for name, stream, seg, a, b in second:
        busy[stream] += b - a
    with open(path, "w") as f:
        f.write(f"# {cfg.name}: one pass (ms from its first event)\n")
        f.write(f"# span {span:.3f} ms; copy stream busy {busy[1]:.3f} ms ({100 * busy[1] / span:.1f} %), "
                f"compute kernels busy {busy[0]:.3f} ms ({100 * busy[0] / span:.1f} %)\n")
        f.write("segment | span | stream | start | end | ms\n")
        for seg in sorted(by_seg):
            for name, stream, a, b in sorted(by_seg[seg], key=lambda e: e[2]):
                f.write(f"{seg} | {name} | {'copy' if stream else 'compute'} | {a:.3f} | {b:.3f} | {b - a:.3f}\n")


def mem_available() -> int:
    """MemAvailable of the host in bytes (0 when unknown)."""
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) * 1024
    except OSError:
        pass
    return 0


def shared_host_stack(cfg, local_rank: int, barrier, local_world: int = 2):
    """One host stack for all ranks of a node: local rank 0 draws it into a memfd and hands
    the descriptor to the other local ranks over a Unix socket; they map the same pages.
    Each process registers its own mapping with the library."""
    import ctypes
    import mmap as _mmap
    import socket
    total = synth.stack_bytes(cfg)
    path = os.path.join(tempfile.gettempdir(), f"ls_bench_{cfg.name}_{os.environ.get('MASTER_PORT', '0')}.sock")
    if local_rank == 0:
        fd = os.memfd_create(f"ls_{cfg.name}")
        os.ftruncate(fd, total)
        if os.path.exists(path):
            os.remove(path)
        srv = socket.socket(socket.AF_UNIX, socket.SOCK_STREAM)
        srv.bind(path)
        srv.listen(local_world)
        barrier()                   # the socket is listening
        for _ in range(local_world - 1):
            conn, _ = srv.accept()
            socket.send_fds(conn, [b"fd"], [fd])
            conn.close()
        srv.close()
        os.remove(path)
    else:
        barrier()
        cli = socket.socket(socket.AF_UNIX, socket.SOCK_STREAM)
        cli.connect(path)
        _, fds, _, _ = socket.recv_fds(cli, 16, 1)
        cli.close()
        fd = fds[0]
    m = _mmap.mmap(fd, total, _mmap.MAP_SHARED, _mmap.PROT_READ | _mmap.PROT_WRITE)
    os.close(fd)
    addr = ctypes.addressof(ctypes.c_char.from_buffer(m))

    def alloc(n):
        return addr, m.close

    hs = synth.HostStack(cfg, alloc=alloc, draw=local_rank == 0)
    barrier()                       # drawn before the other ranks read it
    return hs


def time_alone(torch, L, cfg, hs, x, logits, reps=20) -> dict:
    """{kernel class: average ms per launch} of a stack's GEMMs timed alone, at the workload's
    shapes: back-to-back launches on one stream between one pair of CUDA events, operands
    rotated over enough sets (more than twice the L2 together) that every launch reads its
    inputs from DRAM. MoE: two layers' experts copied from the host stack and routed by their
    own logits; dense kinds: random bf16 operands of the segment's shapes."""
    dev = x.device
    T, H, F = cfg.tokens, cfg.hidden, cfg.ffn
    l2 = 2 * L2_BYTES
    bf = torch.bfloat16
    launches = {}
    if cfg.kind == synth.KIND_MOE_SWIGLU_BF16:
        E, k = cfg.n_experts, cfg.top_k
        seg = synth.segment_slot_bytes(cfg)
        n = 2
        rows = T * k
        W = [torch.from_numpy(hs.buffer[l * seg:(l + 1) * seg]).to(dev) for l in range(n)]
        sel = torch.empty(n, rows, dtype=torch.int32, device=dev)
        w = torch.empty(n, rows, dtype=torch.float32, device=dev)
        table = torch.empty(n, rows, dtype=torch.int32, device=dev)
        bounds = torch.empty(n, E + 1, dtype=torch.int32, device=dev)
        L.lsk_moe_route(logits[:n].contiguous(), n, T, E, k, sel, w)
        L.lsk_moe_group(sel, n, T, E, k, table, bounds)
        xs = [torch.empty(rows, H, dtype=bf, device=dev) for _ in range(n)]
        hsd = [torch.empty(rows, F, dtype=bf, device=dev) for _ in range(n)]
        y = [torch.empty(rows, H, dtype=torch.float32, device=dev) for _ in range(n)]
        for l in range(n):
            L.lsk_moe_gather(x, table[l], rows, k, H, xs[l])
        eb = seg // E
        launches["gemm_up"] = lambda i: L.lsk_gemm_grouped_bf16(
            L.LSK_EPI_SWIGLU, xs[i % n], W[i % n], seg // (2 * H), 0, eb // (2 * H), F, bounds[i % n], E,
            hsd[i % n], rows, F, H)
        launches["gemm_down"] = lambda i: L.lsk_gemm_grouped_bf16(
            L.LSK_EPI_SCALE_F32, hsd[i % n], W[i % n], seg // (2 * F), 2 * H, eb // (2 * F), 0, bounds[i % n], E,
            y[i % n], rows, H, F, row_table=table[i % n], row_weight=w[i % n])
    elif cfg.kind != synth.KIND_LINEAR_GELU_F32:
        g = torch.Generator(device=dev).manual_seed(0)

        def rnd(*shape, dtype=bf):
            return torch.randn(*shape, device=dev, generator=g).to(dtype)
        swiglu = cfg.kind == synth.KIND_SWIGLU_BF16
        up_bytes = 2 * (T * H + (2 if swiglu else 1) * F * H + T * F)
        dn_bytes = 2 * (T * F + H * F) + 12 * T * H
        nu, nd = -(-l2 // up_bytes), -(-l2 // dn_bytes)
        ups = [(rnd(T, H), rnd((2 if swiglu else 1) * F, H), rnd(F), torch.empty(T, F, dtype=bf, device=dev))
               for _ in range(nu)]
        dns = [(rnd(T, F), rnd(H, F), rnd(H), rnd(T, H, dtype=torch.float32), torch.empty(T, H, dtype=bf, device=dev),
                torch.empty(T, H, dtype=torch.float32, device=dev)) for _ in range(nd)]
        if swiglu:
            launches["gemm_up"] = lambda i: L.lsk_gemm_bf16(L.LSK_EPI_SWIGLU, ups[i % nu][0], ups[i % nu][1],
                                                            ups[i % nu][3], T, F, H, b_rows=2 * F, b2_row_off=F)
            launches["gemm_down"] = lambda i: L.lsk_gemm_bf16(L.LSK_EPI_RESID, dns[i % nd][0], dns[i % nd][1],
                                                              dns[i % nd][4], T, H, F, resid=dns[i % nd][3],
                                                              C32=dns[i % nd][5])
        else:
            launches["gemm_up"] = lambda i: L.lsk_gemm_bf16(L.LSK_EPI_BIAS_GELU, ups[i % nu][0], ups[i % nu][1],
                                                            ups[i % nu][3], T, F, H, bias=ups[i % nu][2])
            launches["gemm_down"] = lambda i: L.lsk_gemm_bf16(L.LSK_EPI_BIAS_RESID, dns[i % nd][0], dns[i % nd][1],
                                                              dns[i % nd][4], T, H, F, bias=dns[i % nd][2],
                                                              resid=dns[i % nd][3], C32=dns[i % nd][5])
    out = {}
    s = torch.cuda.current_stream()
    for name, fn in launches.items():
        for i in range(3):
            fn(i)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(s)
        for i in range(reps):
            fn(i)
        e1.record(s)
        e1.synchronize()
        out[name] = e0.elapsed_time(e1) / reps
    return out


def run_ours(args, cfg, world, rank, local):
    import torch
    from host_offloaded_weight_gb300 import lstream as L
    from host_offloaded_weight_gb300.profiling import traffic

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    hbm_peak, tc_peak, tc_sustained, peak_src = measured_peaks()
    link_peak = ce_link_peak(torch)

    def pinned(nbytes):   # the stack's host memory: pinned and mapped by the driver (ls_host_alloc)
        ptr = L.ls_host_alloc(nbytes)
        return ptr, (lambda: L.ls_host_free(ptr))
    local_world = int(os.environ.get("LOCAL_WORLD_SIZE", "1"))
    barrier = (lambda: torch.distributed.barrier()) if world > 1 else (lambda: None)
    host_memory = "ls_host_alloc (pinned and mapped by the driver)"
    if local_world > 1 and mem_available() < local_world * synth.stack_bytes(cfg) * 1.1:
        # N replicas of the stack do not fit the host: the ranks of this node share one
        hs = shared_host_stack(cfg, local, barrier, local_world)
        host_memory = f"one stack shared by the node's {local_world} ranks (memfd), registered by each"
    else:
        hs = synth.HostStack(cfg, alloc=pinned)
    p = L.ls_params_init(prefetch_depth=cfg.prefetch_depth, resident_layers=cfg.resident_layers,
                         max_vram_bytes=cfg.max_vram_bytes, use_pool=cfg.use_pool,
                         copy_path={"auto": 0, "kernel": 1, "engine": 2}[args.copy_path],
                         copy_ctas=args.copy_ctas, reserve_sms=args.reserve_sms, kernel_timing=0,
                         cross_run_prefetch=int(args.cross_run),
                         expert_cache_bytes=int(args.expert_cache_gb * 2**30),
                         debug_checks=int(args.debug_checks))
    ctx = L.ls_ctx_create(p)
    L.ls_register_segments(ctx, hs.segments, hs.shared_map)
    T = cfg.tokens
    xb = synth.draw_x(cfg)
    x = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).to(dev) if cfg.dtype == "bf16" \
        else torch.from_numpy(xb).to(dev)
    y = torch.empty_like(x)
    logits = None
    if cfg.kind == synth.KIND_MOE_SWIGLU_BF16:
        logits = torch.from_numpy(np.stack([synth.draw_logits(cfg, l) for l in range(cfg.n_segments)])).to(dev)
    s = torch.cuda.current_stream()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    # A pass that streams more bytes than L2 holds leaves none of its inputs in L2 for the
    # next one: passes then run back to back and K of them make one contiguous timed region.
    # Smaller stacks get a 256 MB write before every pass instead (outside the pass's events).
    l2_bytes = int(getattr(torch.cuda.get_device_properties(local), "L2_cache_size", 0)) or L2_BYTES
    st0 = L.ls_get_stats(ctx)
    streamed_per_pass = (cfg.n_segments - st0["residents"]) * synth.segment_slot_bytes(cfg)
    flush_between = streamed_per_pass <= l2_bytes
    gpu_id = "GPU-" + str(torch.cuda.get_device_properties(local).uuid)
    sampler = ClockSampler(gpu_id)   # started early: its start-up must not overlap the timed region
    time.sleep(1.5)
    # warm-up passes are issued like the timed ones (asynchronously, flush in between), so
    # the first timed pass starts from the same state as the others
    for _ in range(args.warmup):   # with --graph the warm-up also captures the pass
        if flush_between:
            flush.zero_()
        if args.graph:
            L.ls_run_graph(ctx, x, y, T, s)
        else:
            L.ls_run_async(ctx, x, y, T, s, logits=logits, top_k=cfg.top_k)
    L.ls_sync(ctx)

    def timed_passes(graph=False, n=None):
        n = args.steps if n is None else n
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(n)]
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        for i in range(n):
            if flush_between:
                flush.zero_()                # write 256 MB (> 129 MB L2) between timed passes
            ev[i][0].record(s)
            if graph:
                L.ls_run_graph(ctx, x, y, T, s)
            else:
                L.ls_run_async(ctx, x, y, T, s, logits=logits, top_k=cfg.top_k)
            ev[i][1].record(s)
        L.ls_sync(ctx)
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        return [a.elapsed_time(b) for a, b in ev]

    # throughput (device buffers, passes as a user queues them, no per-launch events in the
    # stream) and end to end (host buffers: every step copies its input in from pinned host memory
    # and its output back out, queued with ls_run_host_async as a serving loop would queue them,
    # one ls_sync closing each block) in alternating blocks of E2E_BLOCK steps: both then see the
    # same state of the host, whose DMA reads of the stack slow down over a process's life
    xh = x.cpu().pin_memory()
    yh = torch.empty_like(xh).pin_memory()
    lh = logits.cpu().pin_memory() if logits is not None else None
    for _ in range(2):
        L.ls_run_host(ctx, xh, yh, T, lh, cfg.top_k)
    L.ls_sync(ctx)
    step_ms, sched, e2e_total = [], [], 0.0
    for b0 in range(0, args.steps, E2E_BLOCK):
        nb = min(E2E_BLOCK, args.steps - b0)
        n_before = len(L.ls_get_schedule(ctx))
        step_ms += timed_passes(graph=args.graph, n=nb)
        sched += L.ls_get_schedule(ctx)[n_before:]
        if world > 1:
            torch.distributed.barrier()
        t0 = time.perf_counter()
        for _ in range(nb):
            L.ls_run_host_async(ctx, xh, yh, T, lh, cfg.top_k)
        L.ls_sync(ctx)
        e2e_total += time.perf_counter() - t0
    e2e_s = e2e_total / args.steps
    # kernel times: the same K passes again with every launch bracketed by events
    L.ls_set_kernel_timing(ctx, 1)
    L.ls_get_kernel_times(ctx, reset=True)
    step_ms_kt = timed_passes()
    ktimes = L.ls_get_kernel_times(ctx, reset=True)
    # segment compute spans: the same K passes with events only around each segment's
    # compute kernels (after the hand-off wait) and the copies; launches keep programmatic
    # dependent launch, so a span shows the kernels as the throughput passes run them
    spans = {}
    if cfg.kind in (synth.KIND_FFN_GELU_BF16, synth.KIND_SWIGLU_BF16):
        L.ls_set_kernel_timing(ctx, 3)
        timed_passes()
        spans = L.ls_get_kernel_times(ctx, reset=True)
    L.ls_set_kernel_timing(ctx, 0)
    if args.timeline and rank == 0:
        write_timeline(args.timeline, L, ctx, x, y, T, s, logits, cfg)
    clocks = sampler.stop()
    mean_s = statistics.mean(step_ms) / 1e3
    stats = L.ls_get_stats(ctx)
    link_bytes = sum(e[5] for e in sched if e[2] in (L.LS_EV_PREFETCH, L.LS_EV_LOAD_SYNC)) / args.steps
    flops = seg_flops(cfg, T) * cfg.n_segments
    max_s, total_tokens = aggregate(mean_s, float(T), world, dev if world > 1 else None)
    value = total_tokens / max_s
    e2e_max, e2e_tokens = aggregate(e2e_s, float(T), world, dev if world > 1 else None)
    h2d = xh.numel() * xh.element_size() + (lh.numel() * 4 if lh is not None else 0)
    d2h = yh.numel() * yh.element_size()
    L.ls_get_kernel_times(ctx, reset=True)
    alone = time_alone(torch, L, cfg, hs, x, logits) if not args.no_alone else {}
    # --- kernels: live averages over the timed region
    kt = {k: {"launches": n, "avg_ms": ms / max(n, 1), "total_ms": ms} for k, (n, ms) in ktimes.items()}
    # kernels of this library launched in the timed region (a copy-engine load raises its
    # ready word with a stream memory operation, not a kernel)
    launches = sum(v["launches"] for k, v in kt.items() if k != "copy_engine")
    # the copy engine is not a kernel, and the hand-off wait does no work of its own
    kernels_only = [k for k in kt if k not in ("copy_engine", "wait_ready")]
    dominant = max(kernels_only, key=lambda k: kt[k]["total_ms"]) if kernels_only else None
    kf = kernel_flops(cfg, T)
    per_load = link_bytes / max(1, sum(1 for e in sched if e[2] in (L.LS_EV_PREFETCH, L.LS_EV_LOAD_SYNC)) / args.steps)
    routed = None
    if cfg.kind == synth.KIND_MOE_SWIGLU_BF16:   # experts a streamed layer moves, on average
        routed = per_load / (sum(t.nbytes for t in synth.segment_tensors(cfg)) / cfg.n_experts)
    kb = kernel_bytes(cfg, T, routed)
    def roof(name, avg_ms=None):
        avg_ms = kt[name]["avg_ms"] if avg_ms is None else avg_ms
        if name in ("copy_h2slot", "copy_engine"):
            ach = per_load / (avg_ms * 1e-3) / 1e9
            return {"kernel": name, "bound": "host_link", "achieved": ach, "peak": link_peak, "unit": "GB/s",
                    "frac": ach / link_peak, "traffic": traffic(cfg.name, name),
                    "peak_source": "pinned copy-engine H2D, 1 GiB, best of 10, measured in this run"}
        if name == "linear_gelu_f32":   # CUDA-core FMA: 152 SMs x 128 lanes x 2 FLOP x max clock
            peak = 152 * 128 * 2 * 2.07e9 / 1e12
            ach = seg_flops(cfg, T) / (avg_ms * 1e-3) / 1e12
            return {"kernel": name, "bound": "alu", "achieved": ach, "peak": peak, "unit": "TFLOP/s",
                    "frac": ach / peak, "traffic": traffic(cfg.name, name),
                    "peak_source": "fp32 FMA lanes x clock (152 x 128 x 2 x 2.07 GHz)"}
        if name in kf:
            # below the ridge (FLOP per byte under peak FLOP/s over peak bytes/s) a launch is
            # bound by HBM: the MoE layers' expert GEMMs, ~128 rows per expert
            sec = avg_ms * 1e-3
            if kf[name] / kb[name] < tc_peak * 1e12 / (hbm_peak * 1e9):
                ach = kb[name] / sec / 1e9
                return {"kernel": name, "bound": "hbm", "achieved": ach, "peak": hbm_peak, "unit": "GB/s",
                        "frac": ach / hbm_peak, "traffic": traffic(cfg.name, name),
                        "algorithmic_bytes": kb[name], "peak_source": f"hbm_gbs ({peak_src})"}
            ach = kf[name] / sec / 1e12
            return {"kernel": name, "bound": "tensor", "achieved": ach, "peak": tc_peak, "unit": "TFLOP/s",
                    "frac": ach / tc_peak, "traffic": traffic(cfg.name, name),
                    "peak_source": f"bf16_tflops ({peak_src})"}
        return None
    roofline = roof(dominant) if dominant else None
    # the same kernels timed alone (back to back, inputs from DRAM): no launch delay or
    # copy-engine traffic in the event brackets
    roofline_alone = None
    if alone:
        roofline_alone = {k: dict(roof(k, ms), avg_ms=ms) for k, ms in alone.items()}
        for v in roofline_alone.values():
            v["measured"] = ("kernel alone: 20 launches back to back between one pair of CUDA events, operands "
                             "rotated over sets larger than twice the L2")
    # the dense stacks' segment compute as the throughput passes run it (GEMMs back to back
    # with programmatic dependent launch, the next segment's copy running meanwhile)
    segment_compute = None
    if cfg.kind in (synth.KIND_FFN_GELU_BF16, synth.KIND_SWIGLU_BF16) and spans.get("compute", (0, 0))[0]:
        n_sp, ms_sp = spans["compute"]
        ach = seg_flops(cfg, T) / (ms_sp / n_sp * 1e-3) / 1e12
        segment_compute = {"spans": n_sp, "avg_ms": ms_sp / n_sp, "achieved": ach, "peak": tc_peak,
                           "unit": "TFLOP/s", "frac": ach / tc_peak,
                           "what": "both GEMMs of a segment, CUDA events from the end of its hand-off "
                                   "wait to its last kernel, launches with programmatic dependent launch"}
    gemm_name = "gemm_down" if "gemm_down" in kt else None
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": max_s * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if cfg.dtype == "bf16" else "f32", "data": "synthetic",
        "config": {"workload": cfg.name, "tokens": T, "segments": cfg.n_segments, "hidden": cfg.hidden,
                   "ffn": cfg.ffn, "prefetch_depth": cfg.prefetch_depth, "resident_layers": cfg.resident_layers,
                   "max_vram_bytes": cfg.max_vram_bytes, "pool": cfg.use_pool,
                   "copy_path": ["per segment", "kernel", "engine"][stats["copy_path"]],
                   "kernel_copy_segments": stats["kernel_copy_segments"],
                   "plan": {"residents": stats["residents"], "depth": stats["depth"],
                            "pool_slots": stats["pool_slots"], "slot_bytes": stats["slot_bytes"],
                            "warnings": stats["warnings"]},
                   "parallelism": f"replicas{world}" if world > 1 else "single",
                   "cross_run_prefetch": bool(args.cross_run),
                   "host_memory": host_memory,
                   "cuda_graph": bool(args.graph), "debug_checks": bool(args.debug_checks),
                   "expert_cache_bytes": int(args.expert_cache_gb * 2**30),
                   "l2": ("flushed between timed passes (256 MB write)" if flush_between else
                          f"inputs larger than L2: each pass streams {streamed_per_pass / 1e6:.0f} MB of "
                          f"weights through HBM (L2 {l2_bytes / 1e6:.0f} MB); passes back to back")},
        "overlap_eff": max(link_bytes / (link_peak * 1e9), flops / (tc_peak * 1e12)) / mean_s,
        "link_gbs": link_bytes / mean_s / 1e9, "link_peak_gbs": link_peak,
        "link_frac": link_bytes / mean_s / 1e9 / link_peak,
        "bytes_per_step": link_bytes, "flops_per_step": flops,
        # the dominant kernel timed alone (burst peak) when it is one of the GEMMs timed alone;
        # otherwise its per-launch figure in the kernel-timed passes
        "roofline": (dict(roofline_alone[dominant], **{"dominant_by": "total time in the kernel-timed passes"})
                     if roofline_alone and dominant in roofline_alone else roofline),
        "roofline_in_pipeline": dict(roofline, measured="per-launch CUDA events in the kernel-timed passes "
                                                        "(includes launch delay while the copy engine works)")
        if roofline else None,
        "roofline_alone": roofline_alone,
        "roofline_gemm": roof(gemm_name) if gemm_name else None,
        "segment_compute": segment_compute,
        "kernels": kt,
        "gpu_launches": launches,
        "step_ms": {"min": min(step_ms), "median": statistics.median(step_ms), "max": max(step_ms),
                    "all": [round(v, 4) for v in step_ms]},
        "kernel_times_from": "a second set of the same K passes with per-launch CUDA events and no "
                             "programmatic dependent launch "
                             f"(mean {statistics.mean(step_ms_kt):.4f} ms per pass with the events)",
        "clocks": {k: clocks[k] for k in ("sm_mhz", "sm_max_mhz", "reasons")},
        "e2e": {"value": e2e_tokens / e2e_max, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "copy_paths_gbs": {"kernel": stats["copy_kernel_gbs"], "engine": stats["copy_engine_gbs"]},
        "expert_cache": {"hits": stats["expert_cache_hits"], "host_loads": stats["expert_host_loads"]}
        if cfg.kind == synth.KIND_MOE_SWIGLU_BF16 else None,
    }
    L.ls_ctx_destroy(ctx)
    if rank == 0 and not args.no_cpu_baseline:
        ntok, nlay = CPU_SAMPLE.get(cfg.name, (1024, None))
        ntok = min(args.cpu_tokens or ntok, T)
        run = OracleRun(cfg, ntok, nlay, hs=hs)
        secs = run.time_pass() * run.scale
        line["cpu_baseline"] = {"value": ntok / secs, "unit": UNIT, "cores": len(os.sched_getaffinity(0)),
                                "kind": "oracle", "sample": run.describe()}
        del run
    hs.close()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def main() -> int:
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=synth.MOE.name, choices=sorted(synth.STACKS))
    ap.add_argument("--copy-path", default="auto", choices=["auto", "kernel", "engine"])
    ap.add_argument("--copy-ctas", type=int, default=0)
    ap.add_argument("--reserve-sms", type=int, default=-1)
    ap.add_argument("--cpu-tokens", type=int, default=0, help="token rows of the CPU oracle sample (0: per workload)")
    ap.add_argument("--ref-tokens", type=int, default=0, help="token rows of the reference arm's sample (0: per workload)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-alone", action="store_true", help="skip timing the GEMMs alone after the passes")
    ap.add_argument("--debug-checks", action="store_true",
                    help="run with params.debug_checks (canaries after every slot, MoE table checks): their cost")
    ap.add_argument("--prefetch-depth", type=int, default=None,
                    help="override the workload's prefetch depth (the planner re-derives residents)")
    ap.add_argument("--expert-cache-gb", type=float, default=0.0,
                    help="MoE: device memory (GiB) for hot experts of streamed layers, beyond the budget")
    ap.add_argument("--graph", action="store_true",
                    help="issue the timed passes as replays of a captured CUDA graph (ls_run_graph)")
    ap.add_argument("--cross-run", action="store_true",
                    help="let the prefetch window cross the pass boundary (off by default, as in the pages)")
    ap.add_argument("--segments", type=int, default=None,
                    help="run only the first N segments of the workload (same per-segment shapes; e.g. a "
                         "profiler capture of the per-segment kernels on a smaller stack)")
    ap.add_argument("--tokens", type=int, default=None, help="override the workload's token count")
    ap.add_argument("--max-vram-bytes", type=int, default=None,
                    help="override the workload's parameter budget (e.g. a one-slot run)")
    ap.add_argument("--timeline", default=None, metavar="FILE",
                    help="after the measurement, trace two more passes (events around every copy and "
                         "around each segment's compute kernels) and write the second one's timeline to FILE")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    world, rank, local = dist_env()
    cfg = synth.STACKS[args.workload]
    if args.prefetch_depth is not None:
        cfg = cfg.with_(prefetch_depth=args.prefetch_depth)
    if args.max_vram_bytes is not None:
        cfg = cfg.with_(max_vram_bytes=args.max_vram_bytes)
    if args.segments is not None:
        cfg = cfg.with_(n_segments=max(1, min(args.segments, cfg.n_segments)))
    if args.tokens is not None:
        cfg = cfg.with_(tokens=max(1, args.tokens))
    if args.graph and (cfg.kind == synth.KIND_MOE_SWIGLU_BF16 or args.cross_run):
        ap.error("--graph needs a kind without per-pass routing and no --cross-run")
    if args.impl == "reference":
        return run_reference(args, cfg, world, rank)
    return run_ours(args, cfg, world, rank, local)


if __name__ == "__main__":
    sys.exit(main())
