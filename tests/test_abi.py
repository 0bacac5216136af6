"""The C ABI without a GPU: the library loads, exports every declared entry
point, validates its versioned parameters, and its scheduler produces the same
events as the independent policy simulator."""
import ctypes
import itertools
import os
import random
import re
import subprocess

import pytest

from host_offloaded_weight_gb300 import lstream as L
from oracle import policy as pol

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")


def _declared():
    names = set()
    for h in os.listdir(INCLUDE):
        if not h.endswith(".h"):
            continue
        text = open(os.path.join(INCLUDE, h)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"\b((?:ls|lsk)_[a-z0-9_]+)\s*\(", text):
            names.add(m.group(1))
    return names


def test_every_declared_symbol_is_exported():
    declared = _declared()
    assert {"ls_ctx_create", "ls_register_segments", "ls_run", "ls_get_schedule"} <= declared
    out = subprocess.run(["nm", "-D", "--defined-only", L.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    missing = declared - exported
    assert not missing, missing
    assert declared <= set(L.EXPORTED)


def test_params_defaults_and_validation():
    p = L.ls_params_init()
    assert p.struct_size == ctypes.sizeof(L.ls_params) and p.version == 1
    assert (p.prefetch_depth, p.resident_layers, p.max_vram_bytes, p.use_pool) == (0, -1, 0, 0)
    assert p.wait_limit_ms == 30000
    ctx = L.ls_ctx_create(p)
    L.ls_ctx_destroy(ctx)
    for bad in ({"prefetch_depth": -1}, {"resident_layers": -2}, {"max_vram_bytes": -5},
                {"use_pool": 2}, {"wait_limit_ms": 0}, {"wait_limit_ms": 600001}):
        with pytest.raises(L.LsError) as e:
            L.ls_ctx_create(L.ls_params_init(**bad))
        assert e.value.status == L.LS_ERR_INVALID_ARG
    with pytest.raises(L.LsError) as e:
        L.ls_ctx_create(L.ls_params_init(version=2))
    assert e.value.status == L.LS_ERR_VERSION
    assert L.ls_status_string(L.LS_ERR_HANDOFF_TIMEOUT).startswith("hand-off")


def test_caller_built_against_the_shorter_struct():
    exe = os.path.join(ROOT, "tests", "abi", "_old_caller")
    src = os.path.join(ROOT, "tests", "abi", "old_caller.c")
    subprocess.run(["gcc", "-O1", "-o", exe, src, L.LIB_PATH, "-Wl,-rpath," + os.path.dirname(L.LIB_PATH)],
                   check=True)
    try:
        r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
        assert r.returncode == 0 and r.stdout.strip() == "ok", (r.returncode, r.stdout, r.stderr)
    finally:
        os.remove(exe)


STRUCTS = ("ls_params", "ls_tensor_desc", "ls_segment_desc", "ls_shared_ref", "ls_moe_routing",
           "ls_kernel_time", "ls_trace_event", "ls_sched_event", "ls_stats")


def test_binding_structs_match_the_header_layout(tmp_path):
    """Every struct the binding declares has the header's size and field offsets, as a C
    compiler lays them out (a field added to one side only shows up here)."""
    lines = ["#include <stdio.h>", "#include <stddef.h>", '#include "ls_api.h"', "int main(void) {"]
    for name in STRUCTS:
        cls = getattr(L, name)
        lines.append(f'    printf("{name} size %zu\\n", sizeof({name}));')
        for field, _ in cls._fields_:
            lines.append(f'    printf("{name} {field} %zu\\n", offsetof({name}, {field}));')
    lines += ["    return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-O0", "-I", INCLUDE, "-o", str(exe), str(src)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True, timeout=60).stdout
    c_layout = {tuple(ln.split()[:2]): int(ln.split()[2]) for ln in out.splitlines()}
    for name in STRUCTS:
        cls = getattr(L, name)
        assert c_layout[(name, "size")] == ctypes.sizeof(cls), name
        for field, _ in cls._fields_:
            assert c_layout[(name, field)] == getattr(cls, field).offset, (name, field)


def _native(seg, shared, depth, resident, budget, pool, runs, cap=None, fail_async=False, load=None):
    p = L.ls_params_init(prefetch_depth=depth, resident_layers=resident, max_vram_bytes=budget,
                         use_pool=pool, test_alloc_cap_bytes=cap or 0,
                         test_fail_async=int(fail_async))
    return L.ls_simulate(p, seg, shared, runs, load)


def _compare(seg, shared, depth, resident, budget, pool, runs, cap=None, fail_async=False, load=None):
    st, ev, stats, rs = _native(seg, shared, depth, resident, budget, pool, runs, cap, fail_async, load)
    sim, sst = pol.simulate(seg, shared, depth, resident, budget, use_pool=pool, runs=runs,
                            alloc_cap=cap, fail_async=fail_async, load_bytes=load)
    if sst and sst[0] < 0 and sim.plan is None:
        assert st == sst[0]
        return
    assert st == sim.status, (seg, depth, resident, budget, pool, cap, st, sim.status)
    assert ev == [tuple(e) for e in sim.events], (seg, depth, resident, budget, pool, cap)
    assert rs == sst
    p = sim.plan
    assert (stats["pool_slots"], stats["slot_bytes"], stats["residents"]) == (p.P, p.S, sim.R)
    assert stats["prefetch_queued"] == sim.stats.prefetch_queued
    assert stats["prefetch_activated"] == sim.stats.prefetch_activated
    assert stats["evictions"] == sim.stats.evictions
    assert stats["pool_degradations"] == sim.stats.pool_degradations
    assert stats["bytes_loaded"] == sim.stats.bytes_loaded


def test_native_scheduler_matches_simulator_grid():
    sizes = ([100] * 5, [100, 60, 100, 40], [80, 100, 100, 100, 20, 100], [100], [256] * 9)
    n = 0
    for seg, depth, resident, budget, pool in itertools.product(
            sizes, range(0, 5), range(-1, 6), (0, 50, 100, 150, 200, 300, 450, 700, 2400), (0, 1)):
        for shared in ([], [(7, 30), (2, 300)]):
            _compare(seg, shared, depth, resident, budget, pool, runs=3)
            n += 1
    assert n > 2000


def test_native_scheduler_matches_simulator_failures():
    n = 0
    for seg, depth, resident, budget, pool, cap, fa in itertools.product(
            ([100] * 6, [100, 50, 100, 100, 70]), (0, 1, 2), (-1, 0, 3), (0, 350, 1000),
            (0, 1), (None, 50, 150, 250, 300, 400, 520), (False, True)):
        _compare(seg, [], depth, resident, budget, pool, runs=3, cap=cap, fail_async=fa)
        n += 1
    assert n > 500


def test_native_scheduler_per_run_load_bytes():
    load = [[10, 20, 30, 40], [11, 21, 31, 41]]
    _compare([100] * 4, [], 1, 1, 1000, 1, runs=2, load=load)


def _compare_script(seg, shared, depth, resident, budget, pool, script, cap=None, fail_async=False,
                    cross=False):
    """The library's scheduler and the policy simulator follow the same script of runs and
    plan changes: same events, same per-step statuses, same counters."""
    p = L.ls_params_init(prefetch_depth=depth, resident_layers=resident, max_vram_bytes=budget,
                         use_pool=pool, test_alloc_cap_bytes=cap or 0, test_fail_async=int(fail_async),
                         cross_run_prefetch=int(cross))
    st, ev, stats, steps = L.ls_simulate_script(p, seg, script, shared)
    sim, ref = pol.simulate_script(seg, shared, depth, resident, budget, use_pool=pool, script=script,
                                      alloc_cap=cap, fail_async=fail_async, cross_run=cross)
    ctx = (seg, shared, depth, resident, budget, pool, script, cap, fail_async, cross)
    if sim.plan is None and not ref:
        assert st == sim.status, ctx
        return
    assert steps == ref, ctx
    assert ev == sim.events, ctx
    if sim.plan is not None:
        assert stats["evictions"] == sim.stats.evictions, ctx
        assert stats["prefetch_queued"] == sim.stats.prefetch_queued, ctx
        assert stats["prefetch_activated"] == sim.stats.prefetch_activated, ctx
        assert stats["resident_loads"] == sim.stats.resident_loads, ctx
        assert stats["pool_degradations"] == sim.stats.pool_degradations, ctx


def test_native_scheduler_matches_simulator_plan_changes():
    rng = random.Random(11)
    n = 0
    for _ in range(1500):
        N = rng.randint(1, 7)
        seg = [rng.choice([64, 100, 128]) for _ in range(N)]
        S = max(seg)
        shared = [] if rng.random() < 0.7 else [(3, rng.choice([40, 200]))]
        sh = sum((b + 255) // 256 * 256 for _, b in shared)

        def controls():
            return (rng.randint(0, N), rng.randint(-1, N),
                    rng.choice([0, sh + rng.randint(1, N + 2) * S, rng.randint(0, sh + (N + 2) * S)]))
        d0, r0, b0 = controls()
        script = [("run",) if rng.random() < 0.6 else ("replan",) + controls() for _ in range(rng.randint(1, 6))]
        script.append(("run",))
        cap = None if rng.random() < 0.6 else sh + rng.randint(1, N + 2) * S
        _compare_script(seg, shared, d0, r0, b0, rng.randint(0, 1), script, cap=cap,
                        fail_async=rng.random() < 0.15, cross=rng.random() < 0.5)
        n += 1
    assert n == 1500
