"""Whole streamed stacks through ls_run against the fp64 oracle, with the executed
schedule against the policy simulator and bit-identity across depth, residency
and pool settings ("feat: pool VRAM for streamed layer", Verification: zero
differing channels with and without the pool; "feat: prefetch streamed layers
during compute", Verification: matching output hashes)."""
import os

import numpy as np
import pytest
import torch

import synth
from host_offloaded_weight_gb300 import lstream as L
from oracle import policy
from oracle import stack as ostack

from gpu_util import BOUND, make_ctx, rel_err, to_f64, x_dev, logits_dev

pytestmark = pytest.mark.gpu


def _sim_events(cfg, hs, depth, resident, budget, pool, runs, load=None, **kw):
    seg = [synth.segment_slot_bytes(cfg)] * len(hs.segments)
    shared = [(i, v.nbytes) for i, v in enumerate(hs.shared_views)]
    if load is None:  # a load moves the segment's exact private bytes
        exact = sum(t.nbytes for t in synth.segment_tensors(cfg))
        load = [[exact] * len(hs.segments) for _ in range(runs)]
    sim, st = policy.simulate(seg, shared, depth, resident, budget, use_pool=pool, runs=runs,
                              load_bytes=load, **kw)
    return sim, st


def _run(cfg, hs, runs=2, logits=None, **over):
    ctx, st = make_ctx(cfg, hs, **over)
    try:
        x = x_dev(cfg)
        y = torch.empty_like(x)
        sts = [L.ls_run(ctx, x, y, cfg.tokens, logits=logits, top_k=cfg.top_k) for _ in range(runs)]
        torch.cuda.synchronize()
        return y.clone(), L.ls_get_schedule(ctx), L.ls_get_stats(ctx), st, sts
    finally:
        L.ls_ctx_destroy(ctx)


def _bits(t):
    return t.view(torch.int16 if t.dtype == torch.bfloat16 else torch.int32).cpu().numpy()


# ------------------------------------------------------------------ tiny fp32 stack (full size)
def test_tiny_fp32_stack_full():
    cfg = synth.TINY
    hs = synth.HostStack(cfg)
    y, ev, stats, st, sts = _run(cfg, hs, runs=3)
    ref = ostack.stack_forward(cfg)
    assert rel_err(to_f64(y), ref) <= 1e-5
    sim, sst = _sim_events(cfg, hs, 1, 0, cfg.max_vram_bytes, 1, 3)
    assert ev == [tuple(e) for e in sim.events]
    assert stats["pool_slots"] == 2 and [e[4] for e in ev if e[2] == L.LS_EV_ACTIVATE][:4] == [0, 1, 0, 1]
    y0, ev0, *_ = _run(cfg, hs, runs=2, prefetch_depth=0)
    assert np.array_equal(_bits(y0), _bits(y)), "depth 0 and depth 1 must give the same bits"


# ------------------------------------------------------------------ small bf16 stacks (full oracle)
SMALL = {
    "ffn": synth.DIT.with_(n_segments=5, tokens=300, hidden=256, ffn=520),
    "proj": synth.SHARED.with_(n_segments=6, tokens=200, hidden=256, ffn=1032),
    "swiglu": synth.LARGE.with_(n_segments=6, tokens=130, hidden=264, ffn=512),
}


@pytest.mark.parametrize("name", sorted(SMALL))
def test_small_stacks_all_settings(name):
    cfg = SMALL[name]
    hs = synth.HostStack(cfg)
    S = synth.segment_slot_bytes(cfg)
    shared_b = sum(synth.align256(v.nbytes) for v in hs.shared_views)
    ref = ostack.stack_forward(cfg)
    base = None
    cases = [(d, r, b, p) for d in (0, 1, 2, 3) for (r, b) in ((0, shared_b + 2 * S), (-1, shared_b + 4 * S), (2, 0))
             for p in (1, 0)]
    for depth, resident, budget, pool in cases:
        y, ev, stats, st, sts = _run(cfg, hs, runs=2, prefetch_depth=depth, resident_layers=resident,
                                     max_vram_bytes=budget, use_pool=pool)
        sim, sst = _sim_events(cfg, hs, depth, resident, budget, pool, 2)
        assert ev == [tuple(e) for e in sim.events], (name, depth, resident, budget, pool)
        assert sts == sst
        if base is None:
            base = _bits(y)
            assert rel_err(to_f64(y), ref) <= BOUND, rel_err(to_f64(y), ref)
        else:
            assert np.array_equal(_bits(y), base), ("bits differ", name, depth, resident, budget, pool)


@pytest.mark.parametrize("path", [L.LS_COPY_KERNEL, L.LS_COPY_ENGINE])
def test_copy_paths_agree(path):
    cfg = SMALL["ffn"]
    hs = synth.HostStack(cfg)
    y, ev, stats, *_ = _run(cfg, hs, copy_path=path,
                            max_vram_bytes=2 * synth.segment_slot_bytes(cfg), prefetch_depth=1,
                            resident_layers=0)
    assert stats["copy_path"] == path
    y2, *_ = _run(cfg, hs, copy_path=L.LS_COPY_KERNEL if path == L.LS_COPY_ENGINE else L.LS_COPY_ENGINE,
                  max_vram_bytes=2 * synth.segment_slot_bytes(cfg), prefetch_depth=1, resident_layers=0)
    assert np.array_equal(_bits(y), _bits(y2))


@pytest.mark.parametrize("name,depth,pool,stride,graph", [("ffn", 1, 1, 2, False), ("ffn", 2, 0, 3, False),
                                                          ("proj", 1, 1, 2, True), ("swiglu", 2, 1, 2, False),
                                                          ("swiglu", 0, 1, 2, False)])
def test_mixed_copy_paths_keep_bits_and_schedule(name, depth, pool, stride, graph):
    """Segments whose loads take different copy paths (every stride-th segment on the copy
    kernel, the others on the copy engine, as the per-segment timing may choose): the bits of
    every load on the copy engine, and the simulator's schedule."""
    cfg = SMALL[name]
    hs = synth.HostStack(cfg)
    S = synth.segment_slot_bytes(cfg)
    shared_b = sum(synth.align256(v.nbytes) for v in hs.shared_views)
    kw = dict(prefetch_depth=depth, resident_layers=0, max_vram_bytes=shared_b + (depth + 1) * S, use_pool=pool)
    ref, ev_ref, *_ = _run(cfg, hs, runs=3, copy_path=L.LS_COPY_ENGINE, **kw)
    ctx, _ = make_ctx(cfg, hs, copy_path=L.LS_COPY_AUTO, test_kernel_copy_stride=stride, **kw)
    try:
        st = L.ls_get_stats(ctx)
        n_kernel = len(range(0, cfg.n_segments, stride))
        assert st["kernel_copy_segments"] == n_kernel and st["copy_path"] == L.LS_COPY_AUTO
        x = x_dev(cfg)
        y = torch.empty_like(x)
        for _ in range(3):
            if graph:
                L.ls_run_graph(ctx, x, y, cfg.tokens)
                L.ls_sync(ctx)
            else:
                L.ls_run(ctx, x, y, cfg.tokens)
            torch.cuda.synchronize()
            assert np.array_equal(_bits(y), _bits(ref))
        assert L.ls_get_schedule(ctx) == ev_ref
    finally:
        L.ls_ctx_destroy(ctx)


def test_auto_copy_path_is_chosen_per_segment():
    """AUTO times both paths on every segment's own load: the summary agrees with the
    per-segment count, both rates are measured, and the bits are those of either forced path."""
    cfg = SMALL["swiglu"]
    hs = synth.HostStack(cfg)
    S = synth.segment_slot_bytes(cfg)
    kw = dict(prefetch_depth=1, resident_layers=0, max_vram_bytes=2 * S, use_pool=1)
    y, _, st, *_ = _run(cfg, hs, runs=2, copy_path=L.LS_COPY_AUTO, **kw)
    k = st["kernel_copy_segments"]
    assert 0 <= k <= cfg.n_segments
    assert st["copy_path"] == (L.LS_COPY_ENGINE if k == 0 else L.LS_COPY_KERNEL if k == cfg.n_segments
                               else L.LS_COPY_AUTO)
    assert st["copy_kernel_gbs"] > 0 and st["copy_engine_gbs"] > 0
    for path in (L.LS_COPY_KERNEL, L.LS_COPY_ENGINE):
        y2, _, st2, *_ = _run(cfg, hs, runs=2, copy_path=path, **kw)
        assert st2["kernel_copy_segments"] == (cfg.n_segments if path == L.LS_COPY_KERNEL else 0)
        assert np.array_equal(_bits(y), _bits(y2))


def test_moe_mixed_copy_paths_keep_bits():
    """The MoE stack with every second layer's routed experts moved by the copy kernel and the
    rest by the copy engine: the bits of the all-engine run and its schedule (bytes of the
    routed experts only)."""
    cfg = _moe_cfg(4, 200, experts=16, hidden=128, ffn=64, k=4)
    hs = synth.HostStack(cfg)
    lg_dev, _ = logits_dev(cfg)
    ref, ev_ref, *_ = _run(cfg, hs, logits=lg_dev, runs=2, copy_path=L.LS_COPY_ENGINE)
    y, ev, st, *_ = _run(cfg, hs, logits=lg_dev, runs=2, copy_path=L.LS_COPY_AUTO, test_kernel_copy_stride=2)
    assert st["kernel_copy_segments"] == 2
    assert np.array_equal(_bits(y), _bits(ref)) and ev == ev_ref


# ------------------------------------------------------------------ full-size stacks, sampled rows
def _rows(cfg, n=48):
    return np.sort(np.random.default_rng(1).choice(cfg.tokens, n, replace=False))


def test_dit_stack_full_size():
    cfg = synth.DIT
    hs = synth.HostStack(cfg)
    y1, ev1, st1, *_ = _run(cfg, hs, runs=2)
    rows = _rows(cfg)
    ref = ostack.stack_forward(cfg, rows=rows)
    assert rel_err(to_f64(y1)[rows], ref) <= BOUND
    sim, _ = _sim_events(cfg, hs, 1, 0, cfg.max_vram_bytes, 1, 2)
    assert ev1 == [tuple(e) for e in sim.events]
    y0, *_ = _run(cfg, hs, runs=1, prefetch_depth=0)
    assert np.array_equal(_bits(y0), _bits(y1))


@pytest.mark.parametrize("copy_path,graph", [(1, False), (1, True), (2, True)])
def test_dit_stack_full_size_other_issue_paths(copy_path, graph):
    """The full DiT stack, whose GEMMs fill every SM, with the copy kernel and with graph
    passes (where the ready word is raised by a publish kernel). The GEMM behind a hand-off
    wait must not be placed early there: its CTAs would leave the copy or publish kernel no
    SM and the wait would run out. Same bits as the copy engine's ordinary passes."""
    cfg = synth.DIT
    hs = synth.HostStack(cfg)
    ref, *_ = _run(cfg, hs, runs=1, copy_path=2)
    ctx, _ = make_ctx(cfg, hs, copy_path=copy_path)
    try:
        x = x_dev(cfg)
        y = torch.empty_like(x)
        for _ in range(4):
            if graph:
                L.ls_run_graph(ctx, x, y, cfg.tokens)
            else:
                L.ls_run_async(ctx, x, y, cfg.tokens)
        L.ls_sync(ctx)
        assert np.array_equal(_bits(y), _bits(ref))
        if graph:
            assert L.ls_get_stats(ctx)["graph_replays"] == 3
    finally:
        L.ls_ctx_destroy(ctx)


def test_shared_projection_stack_full_size():
    cfg = synth.SHARED
    hs = synth.HostStack(cfg)
    rows = _rows(cfg, 32)
    ref = ostack.stack_forward(cfg, rows=rows)
    base = None
    for depth in (0, 1, 2, 3):
        for pool in (1, 0):
            y, ev, stats, st, sts = _run(cfg, hs, runs=2, prefetch_depth=depth, use_pool=pool)
            sim, _ = _sim_events(cfg, hs, depth, -1, cfg.max_vram_bytes, pool, 2)
            assert ev == [tuple(e) for e in sim.events], (depth, pool)
            assert stats["residents"] == 13 - depth and stats["pool_slots"] == 14
            if base is None:
                base = _bits(y)
                assert rel_err(to_f64(y)[rows], ref) <= BOUND
            else:
                assert np.array_equal(_bits(y), base), (depth, pool)


def _oracle_from_host(cfg, hs, rows):
    """fp64 oracle on sampled rows, widening the host stack's own tensors
    (the same bytes the GPU streams) instead of drawing them again."""
    from oracle import forward as F
    x = F.as_f64(synth.draw_x(cfg)[rows], cfg.dtype)
    specs = synth.segment_tensors(cfg)
    for s in range(len(hs.segments)):
        if cfg.kind == synth.KIND_MOE_SWIGLU_BF16:
            views = hs.seg_views[s]
            experts = lambda e, v=views: [F.as_f64(t, "bf16") for t in v[3 * e:3 * e + 3]]
            x = F.moe_swiglu(x, synth.draw_logits(cfg, s)[rows], experts, cfg.top_k)
        else:
            t = [F.as_f64(v, sp.dtype) for v, sp in zip(hs.seg_views[s], specs)]
            x = ostack.apply_segment(cfg, s, x, rows=rows, tensors=t)
    return x


def test_large_swiglu_stack_full_size():
    """48 x 425 MB segments (20 GB in host memory), 4 GiB budget, resident cap
    4, depth 2; then the one-slot budget that takes the mandatory-slot path."""
    cfg = synth.LARGE
    hs = synth.HostStack(cfg)
    y, ev, stats, st, sts = _run(cfg, hs, runs=2)
    assert (stats["residents"], stats["depth"], stats["pool_slots"]) == (4, 2, 7)
    sim, _ = _sim_events(cfg, hs, 2, 4, cfg.max_vram_bytes, 1, 2)
    assert ev == [tuple(e) for e in sim.events]
    rows = _rows(cfg, 16)
    ref = _oracle_from_host(cfg, hs, rows)
    assert rel_err(to_f64(y)[rows], ref) <= BOUND
    one = int(0.1 * 2**30)
    y1, ev1, stats1, st1, _ = _run(cfg, hs, runs=1, max_vram_bytes=one)
    assert st1 == L.LS_WARN_MANDATORY_SLOT and stats1["pool_slots"] == 1 and stats1["depth"] == 0
    assert np.array_equal(_bits(y1), _bits(y))


def test_moe_stack_full_size_with_and_without_expert_cache():
    """The 48-layer MoE stack at full size (58 GB of host experts): one pass matches the
    oracle on sampled rows. Then 40 GiB of expert cache: the third pass reads ~4,500 hot
    experts in place (cache rows far past 2^24) and keeps the bits of the uncached pass."""
    cfg = synth.MOE
    hs = synth.HostStack(cfg)
    lg_dev, _ = logits_dev(cfg)
    # the uncached pass runs with the debug checks on (canaries after both 1.2 GB slots, the
    # routing tables of all 48 layers validated): they find nothing and change no bit
    y0, ev0, stats0, st0, _ = _run(cfg, hs, logits=lg_dev, runs=1, debug_checks=1)
    assert st0 == L.LS_OK and stats0["pool_slots"] == 2 and stats0["depth"] == 1
    assert stats0["debug_violations"] == 0
    # the executed schedule is the simulator's, each load moving its layer's routed experts
    from oracle import forward as F
    eb = synth.segment_slot_bytes(cfg) // cfg.n_experts
    lg = lg_dev.cpu().numpy()
    load = [[len(np.unique(F.route_topk(lg[l], cfg.top_k)[0])) * eb for l in range(cfg.n_segments)]]
    sim, _ = _sim_events(cfg, hs, 1, 0, cfg.max_vram_bytes, 1, 1, load=load)
    assert ev0 == [tuple(e) for e in sim.events]
    rows = _rows(cfg, 8)
    ref = _oracle_from_host(cfg, hs, rows)
    assert rel_err(to_f64(y0)[rows], ref) <= BOUND
    y, ev, stats, st, sts = _run(cfg, hs, logits=lg_dev, runs=3, expert_cache_bytes=40 << 30)
    assert stats["expert_cache_hits"] > 4000
    assert np.array_equal(_bits(y), _bits(y0))


def test_driver_pinned_host_memory_gives_the_same_bits():
    """The stack's tensors in memory from ls_host_alloc (already pinned and mapped, so the
    library registers nothing) stream and compute exactly as from registered pages."""
    cfg = SMALL["ffn"]
    hs = synth.HostStack(cfg)
    y0, ev0, *_ = _run(cfg, hs, runs=2)

    def pinned(n):
        ptr = L.ls_host_alloc(n)
        return ptr, (lambda: L.ls_host_free(ptr))
    hp = synth.HostStack(cfg, alloc=pinned)
    try:
        y1, ev1, *_ = _run(cfg, hp, runs=2)
    finally:
        hp.close()
    assert ev1 == ev0
    assert np.array_equal(_bits(y1), _bits(y0))


# ------------------------------------------------------------------ faults (host-made, bounded)
def test_dropped_handoff_times_out_then_recovers():
    """"layer split: overlap the stages' hand-off", Changes since #936: with the
    drop hook the Nth publish leaves its flag down; the bounded wait sets the
    error word, the run fails with a clear error, and the next run is clean."""
    cfg = SMALL["ffn"].with_(max_vram_bytes=2 * synth.segment_slot_bytes(SMALL["ffn"]))
    hs = synth.HostStack(cfg)
    ctx, _ = make_ctx(cfg, hs, test_drop_publish=3, wait_limit_ms=200, copy_path=L.LS_COPY_KERNEL)
    try:
        x = x_dev(cfg)
        y = torch.empty_like(x)
        with pytest.raises(L.LsError) as e:
            L.ls_run(ctx, x, y, cfg.tokens)
        assert e.value.status == L.LS_ERR_HANDOFF_TIMEOUT
        assert "slot" in L.ls_last_error(ctx)
        L.ls_run(ctx, x, y, cfg.tokens)
        torch.cuda.synchronize()
        assert rel_err(to_f64(y), ostack.stack_forward(cfg)) <= BOUND
    finally:
        L.ls_ctx_destroy(ctx)


def test_pool_degradation_under_allocator_cap():
    cfg = SMALL["ffn"]
    hs = synth.HostStack(cfg)
    S = synth.segment_slot_bytes(cfg)
    y_ref, *_ = _run(cfg, hs, max_vram_bytes=0, prefetch_depth=0)
    y, ev, stats, st, sts = _run(cfg, hs, max_vram_bytes=6 * S, prefetch_depth=1, resident_layers=-1,
                                 test_alloc_cap_bytes=3 * S)
    assert stats["pool_slots"] == 3 and stats["pool_degradations"] >= 1 and stats["slot_bytes"] == S
    sim, _ = _sim_events(cfg, hs, 1, -1, 6 * S, 1, 2, alloc_cap=3 * S)
    assert ev == [tuple(e) for e in sim.events]
    assert np.array_equal(_bits(y), _bits(y_ref))
    with pytest.raises(L.LsError) as e:
        _run(cfg, hs, max_vram_bytes=6 * S, prefetch_depth=1, test_alloc_cap_bytes=S // 2)
    assert e.value.status == L.LS_ERR_OOM
    # the failed registration released its host registration: the same memory registers again
    y2, *_ = _run(cfg, hs, max_vram_bytes=0, prefetch_depth=0)
    assert np.array_equal(_bits(y2), _bits(y_ref))


def test_async_failure_falls_back_synchronously():
    cfg = SMALL["ffn"]
    hs = synth.HostStack(cfg)
    S = synth.segment_slot_bytes(cfg)
    y_ref, *_ = _run(cfg, hs, max_vram_bytes=0, prefetch_depth=0)
    y, ev, stats, st, sts = _run(cfg, hs, max_vram_bytes=2 * S, prefetch_depth=1, resident_layers=0,
                                 test_fail_async=1)
    assert sts[0] == L.LS_WARN_SYNC_FALLBACK and stats["sync_fallbacks"] == 1
    assert all(e[2] != L.LS_EV_PREFETCH for e in ev)
    assert np.array_equal(_bits(y), _bits(y_ref))


def test_pool_off_eviction_under_pressure():
    cfg = SMALL["ffn"].with_(n_segments=6)
    hs = synth.HostStack(cfg)
    S = synth.segment_slot_bytes(cfg)
    y_ref, *_ = _run(cfg, hs, max_vram_bytes=0, prefetch_depth=0)
    y, ev, stats, st, sts = _run(cfg, hs, runs=3, max_vram_bytes=10 * S, prefetch_depth=1, resident_layers=3,
                                 use_pool=0, test_alloc_cap_bytes=4 * S)
    sim, _ = _sim_events(cfg, hs, 1, 3, 10 * S, 0, 3, alloc_cap=4 * S)
    assert ev == [tuple(e) for e in sim.events]
    assert stats["evictions"] >= 1
    assert np.array_equal(_bits(y), _bits(y_ref))


def test_mandatory_slot_warning():
    cfg = SMALL["ffn"]
    hs = synth.HostStack(cfg)
    ctx, st = make_ctx(cfg, hs, max_vram_bytes=synth.segment_slot_bytes(cfg) // 3, prefetch_depth=1)
    try:
        assert st == L.LS_WARN_MANDATORY_SLOT
        s = L.ls_get_stats(ctx)
        assert (s["pool_slots"], s["depth"], s["residents"]) == (1, 0, 0)
    finally:
        L.ls_ctx_destroy(ctx)


@pytest.mark.parametrize("name", ["ffn", "swiglu"])
def test_token_count_changes_between_runs(name):
    """One context runs passes of 1 to 300 tokens in turn: single-CTA tiles below 129
    rows, pair tiles above, the workspaces regrown for the longest; rows are independent,
    so each pass matches the oracle's first T rows. A pass of no tokens is refused."""
    cfg = SMALL[name]
    hs = synth.HostStack(cfg)
    ref = ostack.stack_forward(cfg)
    ctx, _ = make_ctx(cfg, hs)
    try:
        x = x_dev(cfg)
        for T in [t for t in (1, 129, 64, cfg.tokens, 257, 2) if t <= cfg.tokens]:
            y = torch.empty_like(x[:T])
            L.ls_run(ctx, x[:T].contiguous(), y, T)
            torch.cuda.synchronize()
            assert rel_err(to_f64(y), ref[:T]) <= BOUND, (name, T)
        with pytest.raises(L.LsError) as e:
            L.ls_run(ctx, x, torch.empty_like(x), 0)
        assert e.value.status == L.LS_ERR_INVALID_ARG
    finally:
        L.ls_ctx_destroy(ctx)


def test_two_contexts_interleaved():
    """Two contexts with different stacks, their passes interleaved on one stream: each
    gives the bits it gives alone (the GEMMs' descriptor and attribute caches are shared
    by all contexts of the process)."""
    cfgs = [SMALL["ffn"], SMALL["swiglu"]]
    hss = [synth.HostStack(c) for c in cfgs]
    alone = [_bits(_run(c, h, runs=1)[0]) for c, h in zip(cfgs, hss)]
    ctxs = [make_ctx(c, h)[0] for c, h in zip(cfgs, hss)]
    try:
        xs = [x_dev(c) for c in cfgs]
        for _ in range(2):
            ys = [torch.empty_like(x) for x in xs]
            for i in (0, 1):
                L.ls_run_async(ctxs[i], xs[i], ys[i], cfgs[i].tokens)
            for i in (0, 1):
                L.ls_sync(ctxs[i])
            torch.cuda.synchronize()
            for i in (0, 1):
                assert np.array_equal(_bits(ys[i]), alone[i]), i
    finally:
        for c in ctxs:
            L.ls_ctx_destroy(c)


@pytest.mark.parametrize("name", sorted(SMALL))
def test_each_segment_against_the_oracle_on_the_gpus_own_input(name):
    """Diagnostic parity per segment: prefix stacks of 1..N segments give the GPU's bf16
    activation after each segment; the oracle applies segment k to the GPU's own output of
    segment k-1, which isolates that one segment's error (a bf16 rounding of its output and
    of the residual it reads, plus fp32 accumulation)."""
    cfg = SMALL[name]
    outs = [to_f64(x_dev(cfg))]
    for k in range(1, cfg.n_segments + 1):
        hs = synth.HostStack(cfg, n_segments=k)
        y, _, _, _, _ = _run(cfg.with_(n_segments=k), hs, runs=1)
        outs.append(to_f64(y))
    for k in range(1, cfg.n_segments + 1):
        ref = ostack.apply_segment(cfg, k - 1, outs[k - 1])
        assert rel_err(outs[k], ref) <= 6e-3, (name, k, rel_err(outs[k], ref))


def test_run_host_matches_run():
    cfg = SMALL["proj"]
    hs = synth.HostStack(cfg)
    ctx, _ = make_ctx(cfg, hs, max_vram_bytes=0)
    try:
        x = x_dev(cfg)
        y = torch.empty_like(x)
        L.ls_run(ctx, x, y, cfg.tokens)
        xh = x.cpu().pin_memory()
        yh = torch.empty_like(xh).pin_memory()
        L.ls_run_host(ctx, xh, yh, cfg.tokens)
        assert torch.equal(yh.view(torch.int16), y.cpu().view(torch.int16))
    finally:
        L.ls_ctx_destroy(ctx)


@pytest.mark.parametrize("kind", ["proj", "moe"])
def test_run_host_async_pipelines_distinct_inputs(kind):
    """Passes queued from host buffers (ls_run_host_async), each with its own input, logits and
    output buffer, then one ls_sync: every output has the bits of an ls_run of its input."""
    if kind == "moe":
        cfg = _moe_cfg(3, 200, experts=16, hidden=128, ffn=64, k=4)
    else:
        cfg = SMALL["proj"]
    hs = synth.HostStack(cfg)
    ctx, _ = make_ctx(cfg, hs, max_vram_bytes=0 if kind == "proj" else cfg.max_vram_bytes)
    try:
        g = torch.Generator().manual_seed(5)
        xs = [(torch.randn(cfg.tokens, cfg.hidden, generator=g) * (i + 1)).to(torch.bfloat16) for i in range(3)]
        lgs = [torch.randn(cfg.n_segments, cfg.tokens, cfg.n_experts, generator=g) * 2 if kind == "moe" else None
               for _ in range(3)]
        refs = []
        for x, lg in zip(xs, lgs):
            y = torch.empty(cfg.tokens, cfg.hidden, dtype=torch.bfloat16, device="cuda")
            L.ls_run(ctx, x.cuda(), y, cfg.tokens, logits=lg.cuda() if lg is not None else None, top_k=cfg.top_k)
            refs.append(y.cpu())
        xh = [x.pin_memory() for x in xs]
        lh = [lg.pin_memory() if lg is not None else None for lg in lgs]
        yh = [torch.full((cfg.tokens, cfg.hidden), float("nan"), dtype=torch.bfloat16).pin_memory() for _ in range(3)]
        for i in range(3):
            L.ls_run_host_async(ctx, xh[i], yh[i], cfg.tokens, lh[i], cfg.top_k)
        L.ls_sync(ctx)
        for i in range(3):
            assert torch.equal(yh[i].view(torch.int16), refs[i].view(torch.int16)), i
    finally:
        L.ls_ctx_destroy(ctx)


def test_readme_example():
    """The usage shown in the README: torch bf16 CPU tensors registered as FFN segments, one
    pass on device tensors, against the fp64 oracle layer by layer."""
    from oracle import forward as F
    g = torch.Generator().manual_seed(9)
    T, H, Fw, n = 300, 256, 512, 5
    layers = []
    for _ in range(n):
        w1 = (torch.randn(Fw, H, generator=g) / H ** 0.5).to(torch.bfloat16)
        b1 = (torch.randn(Fw, generator=g) * 0.1).to(torch.bfloat16)
        w2 = (torch.randn(H, Fw, generator=g) / Fw ** 0.5 / n ** 0.5).to(torch.bfloat16)
        b2 = (torch.randn(H, generator=g) * 0.1).to(torch.bfloat16)
        layers.append((w1, b1, w2, b2))
    x = torch.randn(T, H, generator=g).to(torch.bfloat16).cuda()
    segs = [(L.LS_KIND_FFN_GELU_BF16, [w1, b1, w2, b2]) for (w1, b1, w2, b2) in layers]
    ctx = L.ls_ctx_create(L.ls_params_init(prefetch_depth=1, resident_layers=-1,
                                           max_vram_bytes=2 * sum(t.nbytes for t in layers[0]), use_pool=1))
    try:
        L.ls_register_segments(ctx, segs)
        y = torch.empty_like(x)
        L.ls_run(ctx, x, y, x.shape[0])
        torch.cuda.synchronize()
        assert L.ls_get_stats(ctx)["depth"] == 1 and len(L.ls_get_schedule(ctx)) > 0
    finally:
        L.ls_ctx_destroy(ctx)
    f64 = lambda t: t.float().numpy().astype(np.float64)
    ref = f64(x.cpu())
    for (w1, b1, w2, b2) in layers:
        ref = F.ffn_gelu(ref, f64(w1), f64(b1), f64(w2), f64(b2))
    assert rel_err(to_f64(y), ref) <= BOUND


def test_kernel_timing_switch():
    """Per-launch timing switched on between passes: refused while a pass is
    queued, and the results do not depend on it (timed and untimed passes
    produce the same bits)."""
    cfg = SMALL["ffn"]
    hs = synth.HostStack(cfg)
    ctx, _ = make_ctx(cfg, hs, kernel_timing=0)
    try:
        x = x_dev(cfg)
        y0, y1 = torch.empty_like(x), torch.empty_like(x)
        L.ls_run_async(ctx, x, y0, cfg.tokens)
        with pytest.raises(L.LsError) as e:
            L.ls_set_kernel_timing(ctx, 1)
        assert e.value.status == L.LS_ERR_STATE
        L.ls_sync(ctx)
        assert L.ls_get_kernel_times(ctx) == {}
        L.ls_set_kernel_timing(ctx, 1)
        L.ls_run(ctx, x, y1, cfg.tokens)
        kt = L.ls_get_kernel_times(ctx, reset=True)
        assert kt["gemm_up"][0] == cfg.n_segments and kt["gemm_down"][0] == cfg.n_segments
        assert all(ms > 0 for _, ms in kt.values())
        assert torch.equal(y0.view(torch.int16), y1.view(torch.int16))
        # segment spans: the copies and one compute span per segment, the same bits again
        y2 = torch.empty_like(x)
        L.ls_set_kernel_timing(ctx, 3)
        L.ls_run(ctx, x, y2, cfg.tokens)
        tr = L.ls_get_trace(ctx)
        kt = {k: v for k, v in L.ls_get_kernel_times(ctx, reset=True).items() if v[0] > 0}
        assert kt["compute"][0] == cfg.n_segments and set(kt) <= {"compute", "copy_engine", "copy_h2slot"}
        spans = [e for e in tr if e[0] == "compute"]
        assert [e[2] for e in spans] == list(range(cfg.n_segments)) and all(e[1] == 0 for e in spans)
        assert all(e[4] >= e[3] for e in tr)
        assert torch.equal(y0.view(torch.int16), y2.view(torch.int16))
        with pytest.raises(L.LsError):
            L.ls_set_kernel_timing(ctx, 4)
    finally:
        L.ls_ctx_destroy(ctx)


# ------------------------------------------------------------------ plan changes, cross-run window
def _sched_script(cfg, hs, depth, resident, budget, pool, script, cross=False):
    seg = [synth.segment_slot_bytes(cfg)] * len(hs.segments)
    shared = [(i, v.nbytes) for i, v in enumerate(hs.shared_views)]
    exact = sum(t.nbytes for t in synth.segment_tensors(cfg))
    sim, st = policy.simulate_script(seg, shared, depth, resident, budget, use_pool=pool, script=script,
                                     cross_run=cross)
    # a load moves the segment's exact private bytes, not its aligned footprint
    ev = [(r, k, kind, sg, sl, exact if kind in (policy.PREFETCH, policy.LOAD_SYNC, policy.LOAD_RESIDENT) else b)
          for (r, k, kind, sg, sl, b) in sim.events]
    return ev, st


@pytest.mark.parametrize("pool", [1, 0])
def test_replan_between_runs_keeps_the_bits(pool):
    """Budget shrinks and grows between runs ("releases stale residents and prefetches when
    the graph plan changes"; "evicts residents from the end of the resident prefix"): every
    run's output equals the all-resident output bit for bit, and the executed schedule is the
    simulator's."""
    cfg = SMALL["ffn"]
    hs = synth.HostStack(cfg)
    S = synth.segment_slot_bytes(cfg)
    ref, _, _, _, _ = _run(cfg, hs, runs=1, max_vram_bytes=0)
    steps = [("run",), ("replan", 1, -1, 4 * S), ("run",), ("replan", 1, -1, 2 * S), ("run",),
             ("replan", 2, 1, 5 * S), ("run",), ("replan", 1, -1, 0), ("run",), ("replan", 1, -1, S // 2),
             ("run",)]
    ctx, _ = make_ctx(cfg, hs, prefetch_depth=1, resident_layers=-1, max_vram_bytes=3 * S, use_pool=pool)
    try:
        x = x_dev(cfg)
        got = []
        for st in steps:
            if st[0] == "run":
                y = torch.empty_like(x)
                L.ls_run(ctx, x, y, cfg.tokens)
                got.append(y)
            else:
                L.ls_replan(ctx, *st[1:])
        torch.cuda.synchronize()
        for y in got:
            assert torch.equal(y.view(torch.int16), ref.view(torch.int16))
        ev, sst = _sched_script(cfg, hs, 1, -1, 3 * S, pool, steps)
        assert L.ls_get_schedule(ctx) == ev
        assert L.ls_get_stats(ctx)["residents"] == 0
    finally:
        L.ls_ctx_destroy(ctx)


@pytest.mark.parametrize("seed,name,pool,cross", [(1, "ffn", 1, False), (2, "ffn", 0, False), (3, "ffn", 1, True),
                                                   (4, "ffn", 0, True), (7, "proj", 1, False), (8, "proj", 0, True)])
def test_random_sequences_of_passes_and_replans(seed, name, pool, cross):
    """Seeded random sequences on one context: passes of random token counts through ls_run,
    ls_run_async (synchronised before the next plan change) and ls_run_host, and plan changes
    of depth, residency and budget in between. Every output matches the oracle's first T rows,
    full-length passes keep the all-resident bits, and the executed schedule is the
    simulator's for the same script. The shared-projection stack adds its deduplicated shared
    parameter, loaded once and kept across plan changes."""
    cfg = SMALL[name]
    hs = synth.HostStack(cfg)
    S = synth.segment_slot_bytes(cfg)
    ref_bits, _, _, _, _ = _run(cfg, hs, runs=1, max_vram_bytes=0)
    ref = ostack.stack_forward(cfg)
    rng = np.random.default_rng(seed)
    n = cfg.n_segments
    script, outs = [], []
    ctx, _ = make_ctx(cfg, hs, prefetch_depth=1, resident_layers=-1, max_vram_bytes=3 * S, use_pool=pool,
                      cross_run_prefetch=int(cross))
    try:
        x = x_dev(cfg)
        for _ in range(24):
            op = rng.choice(["run", "async", "host", "replan"], p=[0.35, 0.25, 0.15, 0.25])
            if op == "replan":
                L.ls_sync(ctx)
                step = ("replan", int(rng.integers(0, 4)), int(rng.choice([-1, 0, 1, 3])),
                        int(rng.choice([0, S // 2, 2 * S, 3 * S, 5 * S, (n + 3) * S])))
                L.ls_replan(ctx, *step[1:])
                script.append(step)
                continue
            T = int(rng.choice([1, 2, 64, 129, 200, cfg.tokens]))
            T = min(T, cfg.tokens)
            xin = x[:T].contiguous()
            if op == "host":
                yh = torch.empty(T, cfg.hidden, dtype=torch.bfloat16).pin_memory()
                L.ls_run_host(ctx, xin.cpu().pin_memory(), yh, T)
                outs.append((T, yh))
            else:
                y = torch.empty_like(xin)
                (L.ls_run if op == "run" else L.ls_run_async)(ctx, xin, y, T)
                outs.append((T, y))
            script.append(("run",))
        L.ls_sync(ctx)
        torch.cuda.synchronize()
        for T, y in outs:
            assert rel_err(to_f64(y), ref[:T]) <= BOUND, T
            if T == cfg.tokens:
                assert torch.equal(y.cpu().view(torch.int16), ref_bits.cpu().view(torch.int16))
        ev, sst = _sched_script(cfg, hs, 1, -1, 3 * S, pool, script, cross=cross)
        assert all(v >= 0 for v in sst)
        assert L.ls_get_schedule(ctx) == ev
    finally:
        L.ls_ctx_destroy(ctx)


@pytest.mark.parametrize("pool", [1, 0])
def test_cross_run_window_matches_simulator_and_bits(pool):
    """The opt-in cross-run window queues the next run's first streamed segment during the
    last step; outputs stay identical, the schedule is the simulator's, and a plan change
    releases the queued prefetch."""
    cfg = SMALL["ffn"]
    hs = synth.HostStack(cfg)
    S = synth.segment_slot_bytes(cfg)
    ref, _, _, _, _ = _run(cfg, hs, runs=1, max_vram_bytes=0)
    ctx, _ = make_ctx(cfg, hs, prefetch_depth=1, resident_layers=0, max_vram_bytes=2 * S, use_pool=pool,
                      cross_run_prefetch=1)
    try:
        x = x_dev(cfg)
        ys = [torch.empty_like(x) for _ in range(3)]
        for y in ys:
            L.ls_run_async(ctx, x, y, cfg.tokens)
        L.ls_sync(ctx)
        L.ls_replan(ctx, 1, 0, 3 * S)
        y4 = torch.empty_like(x)
        L.ls_run(ctx, x, y4, cfg.tokens)
        torch.cuda.synchronize()
        for y in ys + [y4]:
            assert torch.equal(y.view(torch.int16), ref.view(torch.int16))
        steps = [("run",)] * 3 + [("replan", 1, 0, 3 * S), ("run",)]
        ev, _ = _sched_script(cfg, hs, 1, 0, 2 * S, pool, steps, cross=True)
        assert L.ls_get_schedule(ctx) == ev
        kinds = [e[2] for e in ev if e[0] == 3 and e[1] == -1]
        assert kinds[0] == policy.EVICT                         # the stale cross-run prefetch
        assert L.ls_get_stats(ctx)["sync_loads"] == 0
    finally:
        L.ls_ctx_destroy(ctx)


def test_replan_refused_while_passes_are_queued():
    cfg = SMALL["ffn"]
    hs = synth.HostStack(cfg)
    S = synth.segment_slot_bytes(cfg)
    ctx, _ = make_ctx(cfg, hs, prefetch_depth=1, max_vram_bytes=3 * S, use_pool=1)
    try:
        x = x_dev(cfg)
        y = torch.empty_like(x)
        L.ls_run_async(ctx, x, y, cfg.tokens)
        with pytest.raises(L.LsError) as e:
            L.ls_replan(ctx, 1, -1, 2 * S)
        assert e.value.status == L.LS_ERR_STATE
        L.ls_sync(ctx)
        with pytest.raises(L.LsError) as e:
            L.ls_replan(ctx, -1, -1, 2 * S)
        assert e.value.status == L.LS_ERR_INVALID_ARG
        assert L.ls_replan(ctx, 1, -1, 2 * S) == L.LS_OK
    finally:
        L.ls_ctx_destroy(ctx)


# ------------------------------------------------------------------ CUDA-graph passes (NEXT-3)
GRAPH_CASES = {"tiny": synth.TINY, "ffn": SMALL["ffn"], "proj": SMALL["proj"], "swiglu": SMALL["swiglu"]}


@pytest.mark.parametrize("name", sorted(GRAPH_CASES))
@pytest.mark.parametrize("copy_path", [2, 1])
def test_graph_passes_keep_bits_and_schedule(name, copy_path):
    """Passes issued through ls_run_graph: the first steady pass is captured, the rest are
    replays; every output equals an ordinary pass's bit for bit and the schedule log is the
    simulator's, run for run."""
    cfg = GRAPH_CASES[name]
    hs = synth.HostStack(cfg)
    ref, _, _, _, _ = _run(cfg, hs, runs=1)
    runs = 6
    ctx, _ = make_ctx(cfg, hs, copy_path=copy_path)
    try:
        x = x_dev(cfg)
        ys = [torch.empty_like(x) for _ in range(runs)]
        y = torch.empty_like(x)
        for i in range(runs):
            L.ls_run_graph(ctx, x, y, cfg.tokens)
            ys[i].copy_(y)
        L.ls_sync(ctx)
        for yi in ys:
            assert torch.equal(_bits_t(yi), _bits_t(ref))
        sim, _ = _sim_events(cfg, hs, cfg.prefetch_depth, cfg.resident_layers, cfg.max_vram_bytes,
                             cfg.use_pool, runs)
        assert L.ls_get_schedule(ctx) == [tuple(e) for e in sim.events]
        st = L.ls_get_stats(ctx)
        first = 1 if (hs.shared_views or sim.plan.R > 0) else 0   # run 0 loads shared/residents
        assert st["graph_captures"] == 1 and st["graph_replays"] == runs - first - 1
    finally:
        L.ls_ctx_destroy(ctx)


def _bits_t(t):
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)


def test_graph_recaptured_after_changes():
    cfg = SMALL["ffn"]
    hs = synth.HostStack(cfg)
    S = synth.segment_slot_bytes(cfg)
    ref, _, _, _, _ = _run(cfg, hs, runs=1)
    ctx, _ = make_ctx(cfg, hs)
    try:
        x = x_dev(cfg)
        y1, y2 = torch.empty_like(x), torch.empty_like(x)
        for y in (y1, y1, y2, y2):          # a new output buffer: captured again
            L.ls_run_graph(ctx, x, y, cfg.tokens)
        L.ls_sync(ctx)
        assert L.ls_get_stats(ctx)["graph_captures"] == 2
        L.ls_replan(ctx, 1, -1, 3 * S)      # the plan changes: the graph is dropped
        for _ in range(3):
            L.ls_run_graph(ctx, x, y1, cfg.tokens)
        L.ls_sync(ctx)
        st = L.ls_get_stats(ctx)
        assert st["graph_captures"] == 3
        assert torch.equal(_bits_t(y1), _bits_t(ref)) and torch.equal(_bits_t(y2), _bits_t(ref))
        L.ls_run(ctx, x, y2, cfg.tokens)    # an ordinary pass after replays
        assert torch.equal(_bits_t(y2), _bits_t(ref))
    finally:
        L.ls_ctx_destroy(ctx)


def test_graph_refused_for_moe():
    cfg = _moe_cfg(2, 64, experts=8, hidden=256, ffn=128, k=2)
    hs = synth.HostStack(cfg)
    ctx, _ = make_ctx(cfg, hs)
    try:
        x = x_dev(cfg)
        with pytest.raises(L.LsError) as e:
            L.ls_run_graph(ctx, x, torch.empty_like(x), cfg.tokens)
        assert e.value.status == L.LS_ERR_UNSUPPORTED
    finally:
        L.ls_ctx_destroy(ctx)


# ------------------------------------------------------------------ MoE
def _moe_cfg(layers, tokens, experts=128, hidden=2048, ffn=768, k=8):
    c = synth.MOE.with_(n_segments=layers, tokens=tokens, n_experts=experts, hidden=hidden, ffn=ffn, top_k=k)
    return c.with_(max_vram_bytes=2 * synth.segment_slot_bytes(c))


def test_moe_small_all_rows():
    cfg = _moe_cfg(3, 200, experts=16, hidden=128, ffn=64, k=4)
    hs = synth.HostStack(cfg)
    lg_dev, lg = logits_dev(cfg)
    y, ev, stats, st, sts = _run(cfg, hs, logits=lg_dev)
    ref = ostack.stack_forward(cfg)
    assert rel_err(to_f64(y), ref) <= BOUND
    eb = synth.segment_slot_bytes(cfg) // cfg.n_experts
    load = []
    for _ in range(2):
        from oracle import forward as F
        row = []
        for l in range(cfg.n_segments):
            sel, _w = F.route_topk(lg[l], cfg.top_k)
            row.append(len(np.unique(sel)) * eb)
        load.append(row)
    sim, _ = _sim_events(cfg, hs, 1, 0, cfg.max_vram_bytes, 1, 2, load=load)
    assert ev == [tuple(e) for e in sim.events]
    y0, *_ = _run(cfg, hs, logits=lg_dev, prefetch_depth=0, runs=1)
    assert np.array_equal(_bits(y0), _bits(y))


def test_moe_token_counts_change_between_runs():
    """One MoE context runs passes of 1, 7, 200 and 33 tokens in turn (most experts empty at one
    token: 4 of 16 routed); rows are independent given their logits, so each pass matches the
    oracle's first T rows."""
    cfg = _moe_cfg(3, 200, experts=16, hidden=128, ffn=64, k=4)
    hs = synth.HostStack(cfg)
    lg_dev, _ = logits_dev(cfg)
    ref = ostack.stack_forward(cfg)
    ctx, _ = make_ctx(cfg, hs)
    try:
        x = x_dev(cfg)
        for T in (1, 7, 200, 33):
            y = torch.empty_like(x[:T])
            L.ls_run(ctx, x[:T].contiguous(), y, T, logits=lg_dev[:, :T].contiguous(), top_k=cfg.top_k)
            torch.cuda.synchronize()
            assert rel_err(to_f64(y), ref[:T]) <= BOUND, T
    finally:
        L.ls_ctx_destroy(ctx)


def test_moe_residents_follow_routing_changes():
    """Resident MoE layers hold every expert: a later pass that routes to other experts
    still matches the oracle (a resident loaded with only the first pass's routed experts
    would not), and streamed layers move only their routed experts in each pass."""
    cfg = _moe_cfg(4, 64, experts=8, hidden=256, ffn=128, k=2)
    S = synth.segment_slot_bytes(cfg)
    cfg = cfg.with_(max_vram_bytes=4 * S, resident_layers=2)
    hs = synth.HostStack(cfg)
    lg_a_dev, lg_a = logits_dev(cfg)
    lg_b = -lg_a                          # a different top-k in every row
    lg_b_dev = torch.from_numpy(lg_b).cuda()
    ctx, _ = make_ctx(cfg, hs)
    try:
        x = x_dev(cfg)
        ya, yb = torch.empty_like(x), torch.empty_like(x)
        L.ls_run(ctx, x, ya, cfg.tokens, logits=lg_a_dev, top_k=cfg.top_k)
        L.ls_run(ctx, x, yb, cfg.tokens, logits=lg_b_dev, top_k=cfg.top_k)
        torch.cuda.synchronize()
        assert L.ls_get_stats(ctx)["residents"] == 2
        assert rel_err(to_f64(ya), ostack.stack_forward(cfg, logits=list(lg_a))) <= BOUND
        assert rel_err(to_f64(yb), ostack.stack_forward(cfg, logits=list(lg_b))) <= BOUND
        from oracle import forward as F
        eb = S // cfg.n_experts
        exact = sum(t.nbytes for t in synth.segment_tensors(cfg))
        load = []
        for lg in (lg_a, lg_b):
            row = [exact if l < 2 else len(np.unique(F.route_topk(lg[l], cfg.top_k)[0])) * eb
                   for l in range(cfg.n_segments)]
            load.append(row)
        sim, _ = _sim_events(cfg, hs, cfg.prefetch_depth, 2, cfg.max_vram_bytes, 1, 2, load=load)
        assert L.ls_get_schedule(ctx) == [tuple(e) for e in sim.events]
    finally:
        L.ls_ctx_destroy(ctx)


@pytest.mark.parametrize("seed", [5, 6])
def test_moe_random_sequences_of_routings_and_token_counts(seed):
    """Seeded random MoE passes on one context (one resident layer, three streamed): each pass
    draws its own logits (sometimes skewed towards few experts) and token count, and runs
    through ls_run, ls_run_async or ls_run_host. Every output matches the oracle with those
    logits, and each streamed load moves exactly the experts its pass's tokens route to."""
    from oracle import forward as F
    cfg = _moe_cfg(4, 96, experts=8, hidden=256, ffn=128, k=2)
    S = synth.segment_slot_bytes(cfg)
    cfg = cfg.with_(max_vram_bytes=3 * S, resident_layers=1)
    hs = synth.HostStack(cfg)
    rng = np.random.default_rng(seed)
    eb = S // cfg.n_experts
    exact = sum(t.nbytes for t in synth.segment_tensors(cfg))
    ctx, _ = make_ctx(cfg, hs)
    outs, load = [], []
    try:
        x = x_dev(cfg)
        for _ in range(10):
            lg = rng.standard_normal((cfg.n_segments, cfg.tokens, cfg.n_experts)).astype(np.float32)
            if rng.random() < 0.4:
                lg[..., :3] += 4.0                      # most tokens pick the same few experts
            T = int(rng.choice([1, 5, 50, cfg.tokens]))
            lg_t = torch.from_numpy(np.ascontiguousarray(lg[:, :T]))
            xin = x[:T].contiguous()
            op = rng.choice(["run", "async", "host"])
            if op == "host":
                y = torch.empty(T, cfg.hidden, dtype=torch.bfloat16).pin_memory()
                L.ls_run_host(ctx, xin.cpu().pin_memory(), y, T, lg_t.pin_memory(), cfg.top_k)
            else:
                y = torch.empty_like(xin)
                (L.ls_run if op == "run" else L.ls_run_async)(ctx, xin, y, T, logits=lg_t.cuda(), top_k=cfg.top_k)
            outs.append((T, y, lg))
            load.append([exact if l < 1 else len(np.unique(F.route_topk(lg[l, :T], cfg.top_k)[0])) * eb
                         for l in range(cfg.n_segments)])
        L.ls_sync(ctx)
        torch.cuda.synchronize()
        for T, y, lg in outs:
            ref = ostack.stack_forward(cfg, logits=list(lg))
            assert rel_err(to_f64(y), ref[:T]) <= BOUND, T
        sim, _ = _sim_events(cfg, hs, cfg.prefetch_depth, 1, cfg.max_vram_bytes, 1, len(outs), load=load)
        assert L.ls_get_schedule(ctx) == [tuple(e) for e in sim.events]
    finally:
        L.ls_ctx_destroy(ctx)


@pytest.mark.parametrize("copy_path", [2, 1, "mixed"])
@pytest.mark.parametrize("skewed", [True, False])
def test_moe_expert_cache_matches_oracle_policy(copy_path, skewed):
    """Expert cache of the streamed layers: hot experts come from device memory, the
    schedule's load bytes are the oracle policy's host copies, and the bits equal a run
    without the cache. Uniform routing makes most counts tie, which the tie rule decides.
    "mixed": every second layer's host copies go through the copy kernel, the rest through
    the copy engine."""
    from oracle import expert_cache, forward as F
    cfg = _moe_cfg(4, 64, experts=8, hidden=256, ffn=128, k=2)
    S = synth.segment_slot_bytes(cfg)
    eb = S // cfg.n_experts
    K = 6
    hs = synth.HostStack(cfg)
    rng = np.random.default_rng(9)
    bias = np.array([3.0, 2.0, 1.5, 0.5, 0, 0, 0, 0] if skewed else [0] * 8, np.float32)   # data-dependent routing
    passes = [(rng.standard_normal((cfg.n_segments, cfg.tokens, cfg.n_experts)).astype(np.float32) + bias)
              for _ in range(5)]
    outs = {}
    for cache in (0, K * eb):
        path = dict(copy_path=L.LS_COPY_AUTO, test_kernel_copy_stride=2) if copy_path == "mixed" \
            else dict(copy_path=copy_path)
        ctx, _ = make_ctx(cfg, hs, expert_cache_bytes=cache, **path)
        try:
            x = x_dev(cfg)
            ys = []
            for lg in passes:
                y = torch.empty_like(x)
                L.ls_run(ctx, x, y, cfg.tokens, logits=torch.from_numpy(lg).cuda(), top_k=cfg.top_k)
                ys.append(y)
            torch.cuda.synchronize()
            outs[cache] = (ys, L.ls_get_schedule(ctx), L.ls_get_stats(ctx))
        finally:
            L.ls_ctx_destroy(ctx)
    ys, sched, st = outs[K * eb]
    for y, y0 in zip(ys, outs[0][0]):
        assert torch.equal(y.view(torch.int16), y0.view(torch.int16))
    assert rel_err(to_f64(ys[-1]), ostack.stack_forward(cfg, logits=list(passes[-1]))) <= BOUND
    used = []
    for lg in passes:
        u = np.zeros((cfg.n_segments, cfg.n_experts), bool)
        for l in range(cfg.n_segments):
            u[l, np.unique(F.route_topk(lg[l], cfg.top_k)[0])] = True
        used.append(u)
    plan = expert_cache.cache_passes(used, K, 0)
    load = [[int(host[l].sum()) * eb for l in range(cfg.n_segments)] for host, *_ in plan]
    sim, _ = _sim_events(cfg, hs, 1, 0, cfg.max_vram_bytes, 1, len(passes), load=load)
    assert sched == [tuple(e) for e in sim.events]
    hits = sum(int(h.sum()) for _, h, _, _ in plan)
    assert hits > 0 and st["expert_cache_hits"] == hits
    assert st["expert_host_loads"] == sum(int(h.sum()) for h, *_ in plan)


def test_moe_full_expert_shapes_sampled_rows():
    cfg = _moe_cfg(4, 2048)
    hs = synth.HostStack(cfg)
    lg_dev, _ = logits_dev(cfg)
    y, ev, stats, st, sts = _run(cfg, hs, logits=lg_dev, runs=1)
    rows = _rows(cfg, 24)
    ref = ostack.stack_forward(cfg, rows=rows)
    assert rel_err(to_f64(y)[rows], ref) <= BOUND
