"""The copy entry point that allocates no device memory.

Some callers cannot allocate device memory: their device memory is all held by
another allocator, or they run in a loop where cudaMalloc/cudaFree must not be
called because they can synchronise the device. For them the library offers
lsk_copy_h2slot_static, which keeps its scratch (range table and ticket word) in
a fixed array inside the library. Its bytes and its ready word must equal those
of the regular entry point, call after call, as the array is reused.
"""
import numpy as np
import pytest
import torch

from host_offloaded_weight_gb300 import lstream as L

pytestmark = pytest.mark.gpu

SIZES = [1_000_003, 16, 4_101, 65_536, 7]


def _sources(seed):
    g = torch.Generator().manual_seed(seed)
    return [torch.randint(0, 256, (n,), dtype=torch.uint8, generator=g).pin_memory() for n in SIZES]


def _offsets():
    offs, o = [], 0
    for n in SIZES:
        offs.append(o)
        o += (n + 255) // 256 * 256 + 256       # 16-byte aligned, with gaps that stay untouched
    return offs, o


def test_static_copy_matches_regular_entry_point_twice():
    offs, total = _offsets()
    for call, seed in enumerate((11, 12)):       # two calls in a row reuse the scratch array
        srcs = _sources(seed)
        ref = torch.zeros(total, dtype=torch.uint8, device="cuda")
        ready_ref = torch.zeros(len(SIZES), dtype=torch.int32, device="cuda")
        tickets = torch.zeros(len(SIZES), dtype=torch.int32, device="cuda")
        for i, (src, off) in enumerate(zip(srcs, offs)):
            L.lsk_copy_h2slot(ref[off:], src, src.numel(), 0, ready_ref[i:], tickets[i:], 100 + call)
        out = torch.zeros(total, dtype=torch.uint8, device="cuda")
        ready = torch.zeros(1, dtype=torch.int32, device="cuda")
        L.lsk_copy_h2slot_static(out, srcs, [s.numel() for s in srcs], offs, 0, ready, 100 + call)
        torch.cuda.synchronize()
        assert torch.equal(out, ref), f"call {call}: bytes differ from the regular entry point"
        assert int(ready) == 100 + call and all(int(r) == 100 + call for r in ready_ref)


def test_static_copy_rejects_more_ranges_than_its_table():
    n = L.LSK_STATIC_MAX_RANGES + 1
    src = torch.zeros(16, dtype=torch.uint8).pin_memory()
    out = torch.zeros(16, dtype=torch.uint8, device="cuda")
    ready = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(L.LsError) as e:
        L.lsk_copy_h2slot_static(out, [src] * n, [16] * n, [0] * n, 0, ready, 1)
    assert e.value.status == L.LS_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert int(ready) == 0, "a rejected call must queue no work"
