"""The copy entry point that allocates no device memory.

Some callers cannot allocate device memory: their device memory is all held by
another allocator, or they run in a loop where cudaMalloc/cudaFree must not be
called because they can synchronise the device. For them the library offers
lsk_copy_h2slot_static, which keeps its scratch (range table and ticket word) in
a fixed array inside the library. Its bytes and its ready word must equal those
of the regular entry point and the source bytes themselves, call after call, as
the array is reused.
"""
import numpy as np
import pytest
import torch

from host_offloaded_weight_gb300 import lstream as L

pytestmark = pytest.mark.gpu

SIZES = [1_000_003, 16, 4_101, 65_536, 7]


def _sources(sizes, seed):
    g = torch.Generator().manual_seed(seed)
    return [torch.randint(0, 256, (max(n, 1),), dtype=torch.uint8, generator=g)[:n].pin_memory()
            if n else torch.zeros(16, dtype=torch.uint8).pin_memory() for n in sizes]


def _offsets(sizes):
    offs, o = [], 0
    for n in sizes:
        offs.append(o)
        o += (n + 255) // 256 * 256 + 256       # 16-byte aligned, with gaps that stay untouched
    return offs, o


def _expected(srcs, sizes, offs, total):
    """The destination as the copies must leave it: each source at its offset, zeros elsewhere."""
    want = torch.zeros(total, dtype=torch.uint8)
    for src, n, off in zip(srcs, sizes, offs):
        want[off:off + n] = src[:n]
    return want


def _regular(srcs, sizes, offs, total, epoch):
    """The same ranges through the regular entry point, one call per range."""
    ref = torch.zeros(total, dtype=torch.uint8, device="cuda")
    ready = torch.zeros(len(sizes), dtype=torch.int32, device="cuda")
    tickets = torch.zeros(len(sizes), dtype=torch.int32, device="cuda")
    for i, (src, n, off) in enumerate(zip(srcs, sizes, offs)):
        L.lsk_copy_h2slot(ref[off:], src, n, 0, ready[i:], tickets[i:], epoch)
    return ref, ready


def test_static_copy_matches_regular_entry_point_twice():
    offs, total = _offsets(SIZES)
    for call, seed in enumerate((11, 12)):       # two calls in a row reuse the scratch array
        srcs = _sources(SIZES, seed)
        ref, ready_ref = _regular(srcs, SIZES, offs, total, 100 + call)
        out = torch.zeros(total, dtype=torch.uint8, device="cuda")
        ready = torch.zeros(1, dtype=torch.int32, device="cuda")
        L.lsk_copy_h2slot_static(out, srcs, SIZES, offs, 0, ready, 100 + call)
        torch.cuda.synchronize()
        assert torch.equal(out, ref), f"call {call}: bytes differ from the regular entry point"
        assert torch.equal(out.cpu(), _expected(srcs, SIZES, offs, total)), f"call {call}: bytes differ from the sources"
        assert int(ready) == 100 + call and all(int(r) == 100 + call for r in ready_ref)


def test_static_copy_full_table_with_an_empty_range_on_two_ctas():
    """All 64 table entries, one of them empty, on two CTAs: each CTA walks many chunks
    and the chunk-to-range search runs over the whole table."""
    rng = np.random.default_rng(5)
    sizes = [1_000_003, 0] + [int(v) for v in rng.integers(1, 150_000, L.LSK_STATIC_MAX_RANGES - 2)]
    assert len(sizes) == L.LSK_STATIC_MAX_RANGES
    offs, total = _offsets(sizes)
    for call, seed in enumerate((21, 22)):
        srcs = _sources(sizes, seed)
        ref, ready_ref = _regular(srcs, sizes, offs, total, 7 + call)
        out = torch.zeros(total, dtype=torch.uint8, device="cuda")
        ready = torch.zeros(1, dtype=torch.int32, device="cuda")
        L.lsk_copy_h2slot_static(out, srcs, sizes, offs, 2, ready, 7 + call)
        torch.cuda.synchronize()
        assert torch.equal(out.cpu(), _expected(srcs, sizes, offs, total)), f"call {call}: bytes differ from the sources"
        assert torch.equal(out, ref), f"call {call}: bytes differ from the regular entry point"
        assert int(ready) == 7 + call and all(int(r) == 7 + call for r in ready_ref)


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


def test_static_copy_refuses_a_capturing_stream():
    """The range table is staged from the call's stack frame, which a graph replay would
    read again: a call on a stream under capture is refused and queues nothing. The
    capture is ended without launching the graph."""
    src = torch.arange(64, dtype=torch.uint8).pin_memory()
    out = torch.zeros(64, dtype=torch.uint8, device="cuda")
    ready = torch.zeros(1, dtype=torch.int32, device="cuda")
    keep = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    status = None
    with torch.cuda.stream(s):
        g.capture_begin()
        try:
            L.lsk_copy_h2slot_static(out, [src], [64], [0], 0, ready, 3, stream=s)
        except L.LsError as e:
            status = e.status
        finally:
            keep.add_(1)                # the captured graph is not empty
            g.capture_end()
    del g
    torch.cuda.synchronize()
    assert status == L.LS_ERR_INVALID_ARG
    assert int(ready) == 0 and int(out.sum()) == 0 and int(keep) == 0
    # the same call outside the capture runs
    L.lsk_copy_h2slot_static(out, [src], [64], [0], 0, ready, 3)
    torch.cuda.synchronize()
    assert int(ready) == 3 and torch.equal(out.cpu(), src)
