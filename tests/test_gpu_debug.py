"""The debug-checks mode (params.debug_checks), which stands in for a memory sanitizer:
canaries after every pool slot, the shared region and per-load buffers, and a device-side
validation of the MoE row table and group bounds.

On valid runs the mode finds nothing and changes no bit of the output or the schedule.
A canary overwritten by the host (the test hook, an in-bounds write of the canary itself)
and routing tables made invalid on the host are reported; the checks only read, so no
invalid index is ever used to address memory.
"""
import numpy as np
import pytest
import torch

import synth
from host_offloaded_weight_gb300 import lstream as L
from gpu_util import logits_dev

import test_gpu_stacks as TS

pytestmark = pytest.mark.gpu


def _moe_small():
    return TS._moe_cfg(3, 200, experts=16, hidden=128, ffn=64, k=4)


CASES = [("ffn", dict(use_pool=1)), ("ffn", dict(use_pool=0)), ("proj", dict(use_pool=1)),
         ("swiglu", dict(use_pool=1, prefetch_depth=2)), ("moe", dict(use_pool=1)), ("moe", dict(use_pool=0))]


@pytest.mark.parametrize("name,over", CASES, ids=[f"{n}-pool{o['use_pool']}" for n, o in CASES])
def test_debug_checks_find_nothing_and_keep_the_bits(name, over):
    cfg = _moe_small() if name == "moe" else TS.SMALL[name]
    hs = synth.HostStack(cfg)
    lg = logits_dev(cfg)[0] if name == "moe" else None
    y0, ev0, st0, s0, r0 = TS._run(cfg, hs, logits=lg, runs=3, **over)
    y1, ev1, st1, s1, r1 = TS._run(cfg, hs, logits=lg, runs=3, debug_checks=1, **over)
    assert s1 == s0 and r1 == r0 and all(r >= 0 for r in r1)
    assert st1["debug_violations"] == 0
    assert ev1 == ev0, "the checks change the schedule"
    assert np.array_equal(TS._bits(y1), TS._bits(y0)), "the checks change the output bits"


def test_overwritten_slot_canary_fails_the_run():
    cfg = TS.SMALL["ffn"]
    hs = synth.HostStack(cfg)
    ctx, _ = TS.make_ctx(cfg, hs, debug_checks=1, test_corrupt_canary=2)
    try:
        x = TS.x_dev(cfg)
        y = torch.empty_like(x)
        with pytest.raises(L.LsError) as e:
            L.ls_run(ctx, x, y, cfg.tokens)
        assert e.value.status == L.LS_ERR_BOUNDS
        assert "pool slot 1" in str(e.value)
        assert L.ls_get_stats(ctx)["debug_violations"] == 1
    finally:
        L.ls_ctx_destroy(ctx)


def _routing(T=96, E=12, k=3, layers=2, seed=4):
    lg = torch.from_numpy(np.random.default_rng(seed).standard_normal((layers, T, E)).astype(np.float32)).cuda()
    sel = torch.empty(layers, T * k, dtype=torch.int32, device="cuda")
    w = torch.empty(layers, T * k, dtype=torch.float32, device="cuda")
    table = torch.empty(layers, T * k, dtype=torch.int32, device="cuda")
    bounds = torch.empty(layers, E + 1, dtype=torch.int32, device="cuda")
    L.lsk_moe_route(lg, layers, T, E, k, sel, w)
    L.lsk_moe_group(sel, layers, T, E, k, table, bounds)
    torch.cuda.synchronize()
    return sel, table, bounds, (T, E, k, layers)


def _check(sel, table, bounds, dims):
    T, E, k, layers = dims
    err = torch.zeros(1, dtype=torch.int32).pin_memory()
    L.lsk_moe_check(sel, table, bounds, layers, T, k, E, err)
    torch.cuda.synchronize()
    return int(err.item()) & 0xFFFFFFFF


def test_moe_check_accepts_the_grouping_kernels_output():
    sel, table, bounds, dims = _routing()
    assert _check(sel, table, bounds, dims) == 0


def _bad(kind, sel, table, bounds, dims):
    T, E, k, layers = dims
    t, b = table.cpu().numpy().copy(), bounds.cpu().numpy().copy()
    lay = 1
    if kind == "rows_swapped_across_groups":        # a row filed under another expert
        lo = b[lay, 1]
        t[lay, 0], t[lay, lo] = t[lay, lo], t[lay, 0]
    elif kind == "row_twice":
        t[lay, 1] = t[lay, 0]
    elif kind == "row_out_of_range":
        t[lay, 2] = T * k
    elif kind == "bounds_decrease":
        b[lay, 3], b[lay, 4] = b[lay, 4], b[lay, 3] - 1
    elif kind == "bounds_short":
        b[lay, E] -= 1
    elif kind == "group_out_of_order":
        lo, hi = b[lay, 0], b[lay, 1]
        assert hi - lo >= 2
        t[lay, lo], t[lay, lo + 1] = t[lay, lo + 1], t[lay, lo]
    return torch.from_numpy(t).cuda(), torch.from_numpy(b).cuda()


@pytest.mark.parametrize("kind", ["rows_swapped_across_groups", "row_twice", "row_out_of_range",
                                  "bounds_decrease", "bounds_short", "group_out_of_order"])
def test_moe_check_flags_invalid_tables(kind):
    sel, table, bounds, dims = _routing()
    t, b = _bad(kind, sel, table, bounds, dims)
    code = _check(sel, t, b, dims)
    assert code & 0xFF == 4 and code >> 8 == 0x20000 + 1, hex(code)     # DERR_BOUNDS, layer 1
