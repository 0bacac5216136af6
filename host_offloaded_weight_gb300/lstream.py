"""ctypes binding of liblstream.so: the C ABI of include/ls_api.h and include/ls_kernels.h
under the same names. It only marshals arguments (torch tensors and numpy
arrays to pointers, Python lists to C arrays); all work happens in the library.

Negative status codes raise ``LsError`` carrying the context's ``ls_last_error``;
warnings (positive codes) are returned.
"""
from __future__ import annotations

import ctypes as C
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "liblstream.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()' "
        "or python host_offloaded_weight_gb300/build.py). There is no fallback path.")
_lib = C.CDLL(LIB_PATH)

# ------------------------------------------------------------------ constants
LS_PARAMS_VERSION = 1
LS_OK, LS_WARN_MANDATORY_SLOT, LS_WARN_SYNC_FALLBACK = 0, 1, 2
LS_ERR_INVALID_ARG, LS_ERR_VERSION, LS_ERR_OOM = -1, -2, -3
LS_ERR_HANDOFF_TIMEOUT, LS_ERR_CUDA, LS_ERR_STATE, LS_ERR_UNSUPPORTED, LS_ERR_BOUNDS = -4, -5, -6, -7, -8
LS_KIND_LINEAR_GELU_F32, LS_KIND_FFN_GELU_BF16, LS_KIND_FFN_GELU_SHARED_BF16 = 0, 1, 2
LS_KIND_SWIGLU_BF16, LS_KIND_MOE_SWIGLU_BF16 = 3, 4
LS_DTYPE_F32, LS_DTYPE_BF16 = 0, 1
LS_EV_SHARED_LOAD, LS_EV_LOAD_RESIDENT, LS_EV_LOAD_SYNC, LS_EV_PREFETCH, LS_EV_ACTIVATE, LS_EV_EVICT = range(6)
LS_COPY_AUTO, LS_COPY_KERNEL, LS_COPY_ENGINE = 0, 1, 2
LSK_EPI_STORE, LSK_EPI_BIAS_GELU, LSK_EPI_BIAS_RESID, LSK_EPI_SWIGLU, LSK_EPI_RESID, LSK_EPI_SCALE_F32 = range(6)

ALLOC_FN = C.CFUNCTYPE(C.c_void_p, C.c_void_p, C.c_size_t, C.c_void_p)
FREE_FN = C.CFUNCTYPE(None, C.c_void_p, C.c_void_p, C.c_size_t, C.c_void_p)


class ls_params(C.Structure):
    _fields_ = [("struct_size", C.c_uint32), ("version", C.c_uint32),
                ("prefetch_depth", C.c_int32), ("resident_layers", C.c_int32),
                ("max_vram_bytes", C.c_int64), ("use_pool", C.c_int32),
                ("wait_limit_ms", C.c_int32), ("copy_path", C.c_int32), ("copy_ctas", C.c_int32),
                ("reserve_sms", C.c_int32), ("device", C.c_int32),
                ("alloc_fn", ALLOC_FN), ("free_fn", FREE_FN), ("alloc_user", C.c_void_p),
                ("test_alloc_cap_bytes", C.c_int64), ("test_fail_async", C.c_int32),
                ("test_drop_publish", C.c_int32), ("kernel_timing", C.c_int32),
                ("cross_run_prefetch", C.c_int32), ("expert_cache_bytes", C.c_int64),
                ("debug_checks", C.c_int32), ("test_corrupt_canary", C.c_int32),
                ("test_kernel_copy_stride", C.c_int32)]


class ls_tensor_desc(C.Structure):
    _fields_ = [("host_ptr", C.c_void_p), ("bytes", C.c_uint64), ("dtype", C.c_int32),
                ("ndim", C.c_int32), ("shape", C.c_int64 * 2)]


class ls_segment_desc(C.Structure):
    _fields_ = [("kind", C.c_int32), ("n_tensors", C.c_int32),
                ("tensors", C.POINTER(ls_tensor_desc))]


class ls_shared_ref(C.Structure):
    _fields_ = [("segment", C.c_int32), ("tensor_index", C.c_int32), ("shared_id", C.c_int32)]


class ls_moe_routing(C.Structure):
    _fields_ = [("logits", C.c_void_p), ("top_k", C.c_int32)]


class ls_kernel_time(C.Structure):
    _fields_ = [("name", C.c_char * 32), ("launches", C.c_int64), ("total_ms", C.c_double)]


class ls_trace_event(C.Structure):
    _fields_ = [("name", C.c_char * 32), ("stream", C.c_int32), ("segment", C.c_int32),
                ("start_ms", C.c_double), ("end_ms", C.c_double)]


class ls_sched_event(C.Structure):
    _fields_ = [("run", C.c_int32), ("step", C.c_int32), ("kind", C.c_int32),
                ("segment", C.c_int32), ("slot", C.c_int32), ("reserved", C.c_int32),
                ("bytes", C.c_int64)]


class ls_stats(C.Structure):
    _fields_ = [("struct_size", C.c_uint32), ("n_segments", C.c_int32), ("residents", C.c_int32),
                ("depth", C.c_int32), ("ring_slots", C.c_int32), ("pool_slots", C.c_int32),
                ("warnings", C.c_int32), ("copy_path", C.c_int32), ("slot_bytes", C.c_int64),
                ("shared_bytes", C.c_int64), ("pool_bytes", C.c_int64), ("runs", C.c_int64),
                ("prefetch_queued", C.c_int64), ("prefetch_activated", C.c_int64),
                ("sync_loads", C.c_int64), ("resident_loads", C.c_int64),
                ("shared_loads", C.c_int64), ("evictions", C.c_int64),
                ("sync_fallbacks", C.c_int64), ("pool_degradations", C.c_int64),
                ("bytes_loaded", C.c_int64), ("copy_kernel_gbs", C.c_double),
                ("copy_engine_gbs", C.c_double), ("graph_captures", C.c_int64),
                ("graph_replays", C.c_int64), ("expert_cache_hits", C.c_int64),
                ("expert_host_loads", C.c_int64), ("debug_violations", C.c_int64),
                ("kernel_copy_segments", C.c_int64)]


_P = C.c_void_p
_I32, _I64, _U32, _U64 = C.c_int32, C.c_int64, C.c_uint32, C.c_uint64
_sig = {
    "ls_params_init": (None, [C.POINTER(ls_params)]),
    "ls_ctx_create": (_I32, [C.POINTER(ls_params), C.POINTER(_P)]),
    "ls_register_segments": (_I32, [_P, C.POINTER(ls_segment_desc), _I32, C.POINTER(ls_shared_ref), _I32]),
    "ls_run": (_I32, [_P, _P, _P, _I64, _P, C.POINTER(ls_moe_routing)]),
    "ls_run_host": (_I32, [_P, _P, _P, _I64, C.POINTER(ls_moe_routing)]),
    "ls_run_host_async": (_I32, [_P, _P, _P, _I64, C.POINTER(ls_moe_routing)]),
    "ls_run_async": (_I32, [_P, _P, _P, _I64, _P, C.POINTER(ls_moe_routing)]),
    "ls_sync": (_I32, [_P]),
    "ls_get_schedule": (_I32, [_P, C.POINTER(ls_sched_event), _I64, C.POINTER(_I64)]),
    "ls_get_stats": (_I32, [_P, C.POINTER(ls_stats)]),
    "ls_set_kernel_timing": (_I32, [_P, _I32]),
    "ls_replan": (_I32, [_P, _I32, _I32, _I64]),
    "ls_run_graph": (_I32, [_P, _P, _P, _I64, _P]),
    "ls_simulate_script": (_I32, [C.POINTER(ls_params), C.POINTER(_I64), _I32, C.POINTER(_I64),
                                  C.POINTER(_I32), _I32, C.POINTER(_I64), _I32, C.POINTER(ls_sched_event),
                                  _I64, C.POINTER(_I64), C.POINTER(ls_stats), C.POINTER(_I32)]),
    "ls_get_kernel_times": (_I32, [_P, C.POINTER(ls_kernel_time), _I32, C.POINTER(_I32), _I32]),
    "ls_get_trace": (_I32, [_P, C.POINTER(ls_trace_event), _I64, C.POINTER(_I64)]),
    "ls_ctx_destroy": (None, [_P]),
    "ls_status_string": (C.c_char_p, [_I32]),
    "ls_last_error": (C.c_char_p, [_P]),
    "ls_simulate": (_I32, [C.POINTER(ls_params), C.POINTER(_I64), _I32, C.POINTER(_I64),
                           C.POINTER(_I32), _I32, _I32, C.POINTER(_I64), C.POINTER(ls_sched_event),
                           _I64, C.POINTER(_I64), C.POINTER(ls_stats), C.POINTER(_I32)]),
    "lsk_num_sms": (_I32, []),
    "lsk_gemm_tile_n": (_I32, [_I32, _I32, _I32]),
    "lsk_device_error": (_U32, []),
    "lsk_copy_h2slot": (_I32, [_P, _P, _U64, _I32, _P, _P, _U32, _P]),
    "lsk_wait_ready": (_I32, [_P, _U32, _I32, _P, _I32, _P]),
    "lsk_copy_h2slot_static": (_I32, [_P, C.POINTER(_P), C.POINTER(_U64), C.POINTER(_U64), _I32, _I32, _P,
                                      _U32, _P]),
    "lsk_gemm_bf16": (_I32, [_I32, _P, _P, _I64, _I32, _P, _P, _I32, _P, _P, _I32, _I32, _I32, _I32, _P]),
    "lsk_gemm_grouped_bf16": (_I32, [_I32, _P, _P, _I64, _I32, _I32, _I32, _P, _I32, _P, _P, _P,
                                     _I32, _I32, _I32, _I32, _P]),
    "lsk_linear_gelu_f32": (_I32, [_P, _P, _P, _P, _I32, _I32, _I32, _P]),
    "lsk_moe_route": (_I32, [_P, _I32, _I32, _I32, _I32, _P, _P, _P]),
    "lsk_moe_group": (_I32, [_P, _I32, _I32, _I32, _I32, _P, _P, _P, _P]),
    "lsk_moe_gather": (_I32, [_P, _P, _I32, _I32, _I32, _P, _P]),
    "lsk_moe_combine": (_I32, [_P, _I32, _P, _I32, _I32, _I32, _P, _P, _P]),
    "lsk_moe_check": (_I32, [_P, _P, _P, _I32, _I32, _I32, _I32, _P, _P]),
    "lsk_moe_group_masked": (_I32, [_P, _I32, _I32, _I32, _I32, _P, _P, _P, _P, _P]),
    "lsk_moe_rows_copy": (_I32, [_P, _P, _P, _P, _I32, _I32, _P, _P, _U32, _I32, _P]),
    "ls_helper_share": (C.c_double, [_I64]),
    "ls_host_alloc": (_I32, [_U64, C.POINTER(_P)]),
    "ls_host_free": (_I32, [_P]),
    "ls_helper_split": (_I32, [_P, _I32, C.c_double, _P]),
}
for _name, (_res, _args) in _sig.items():
    _f = getattr(_lib, _name)
    _f.restype = _res
    _f.argtypes = _args

EXPORTED = tuple(_sig)


class LsError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{ls_status_string(status)} ({status}): {msg}")
        self.status = status


def ls_status_string(s: int) -> str:
    return _lib.ls_status_string(int(s)).decode()


def _check(status: int, ctx=None) -> int:
    if status < 0:
        msg = _lib.ls_last_error(ctx.handle if isinstance(ctx, Ctx) else ctx).decode() if ctx else ""
        raise LsError(status, msg)
    return status


def _ptr(t) -> int:
    """Address of a torch tensor, numpy array or raw int pointer (None -> 0)."""
    if t is None:
        return 0
    if isinstance(t, int):
        return t
    if hasattr(t, "data_ptr"):
        return t.data_ptr()
    if hasattr(t, "ctypes"):
        return t.ctypes.data
    raise TypeError(f"cannot take the address of {type(t)}")


def _stream(stream) -> int:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


class Ctx:
    """A context handle plus references to the host buffers it reads."""

    def __init__(self, handle: int):
        self.handle = handle
        self.keep = []

    def __bool__(self):
        return bool(self.handle)


# ------------------------------------------------------------------ ls_api.h
def ls_params_init(**fields) -> ls_params:
    p = ls_params()
    _lib.ls_params_init(C.byref(p))
    for k, v in fields.items():
        setattr(p, k, v)
    return p


def ls_ctx_create(params: ls_params) -> Ctx:
    h = _P()
    _check(_lib.ls_ctx_create(C.byref(params), C.byref(h)))
    return Ctx(h.value)


def _dtype_code(t) -> int:
    name = str(getattr(t, "dtype", ""))
    if "float32" in name:
        return LS_DTYPE_F32
    if "bfloat16" in name or "uint16" in name:
        return LS_DTYPE_BF16
    raise TypeError(f"unsupported tensor dtype {name}")


def _nbytes(t) -> int:
    if hasattr(t, "nbytes"):
        return int(t.nbytes)
    return t.numel() * t.element_size()


def ls_register_segments(ctx: Ctx, segments, shared_map=()) -> int:
    """segments: list of (kind, [host tensors]) — torch CPU tensors (pinned or
    not) or numpy arrays; bf16 may be given as uint16 bit patterns.
    shared_map: list of (segment, tensor_index, shared_id)."""
    segs = (ls_segment_desc * len(segments))()
    for i, (kind, tensors) in enumerate(segments):
        arr = (ls_tensor_desc * len(tensors))()
        for j, t in enumerate(tensors):
            shape = tuple(t.shape)
            arr[j].host_ptr = _ptr(t)
            arr[j].bytes = _nbytes(t)
            arr[j].dtype = _dtype_code(t)
            arr[j].ndim = len(shape)
            for d, v in enumerate(shape[:2]):
                arr[j].shape[d] = v
            ctx.keep.append(t)
        ctx.keep.append(arr)
        segs[i].kind = kind
        segs[i].n_tensors = len(tensors)
        segs[i].tensors = arr
    sm = (ls_shared_ref * max(1, len(shared_map)))()
    for i, (s, ti, sid) in enumerate(shared_map):
        sm[i].segment, sm[i].tensor_index, sm[i].shared_id = s, ti, sid
    return _check(_lib.ls_register_segments(ctx.handle, segs, len(segments), sm, len(shared_map)), ctx)


def _routing(logits, top_k):
    if logits is None:
        return None
    r = ls_moe_routing()
    r.logits = _ptr(logits)
    r.top_k = top_k
    return r


def ls_run(ctx: Ctx, x, y, tokens: int, stream=None, logits=None, top_k: int = 0) -> int:
    """One streamed pass on device tensors (stream: torch stream, raw handle or None = current)."""
    r = _routing(logits, top_k)
    return _check(_lib.ls_run(ctx.handle, _ptr(x), _ptr(y), int(tokens), _stream(stream),
                              C.byref(r) if r is not None else None), ctx)


def ls_run_async(ctx: Ctx, x, y, tokens: int, stream=None, logits=None, top_k: int = 0) -> int:
    """Queue one pass without waiting for it; ls_sync reports device errors."""
    r = _routing(logits, top_k)
    return _check(_lib.ls_run_async(ctx.handle, _ptr(x), _ptr(y), int(tokens), _stream(stream),
                                    C.byref(r) if r is not None else None), ctx)


def ls_sync(ctx: Ctx) -> int:
    return _check(_lib.ls_sync(ctx.handle), ctx)


def ls_run_host(ctx: Ctx, x_host, y_host, tokens: int, logits_host=None, top_k: int = 0) -> int:
    r = _routing(logits_host, top_k)
    return _check(_lib.ls_run_host(ctx.handle, _ptr(x_host), _ptr(y_host), int(tokens),
                                   C.byref(r) if r is not None else None), ctx)


def ls_run_host_async(ctx: Ctx, x_host, y_host, tokens: int, logits_host=None, top_k: int = 0) -> int:
    """ls_run_host queued on the context's own stream; y_host is valid after ls_sync."""
    r = _routing(logits_host, top_k)
    return _check(_lib.ls_run_host_async(ctx.handle, _ptr(x_host), _ptr(y_host), int(tokens),
                                         C.byref(r) if r is not None else None), ctx)


def _events(buf, n):
    return [(e.run, e.step, e.kind, e.segment, e.slot, e.bytes) for e in buf[:n]]


def ls_get_schedule(ctx: Ctx) -> list:
    n = _I64()
    _check(_lib.ls_get_schedule(ctx.handle, None, 0, C.byref(n)), ctx)
    buf = (ls_sched_event * max(1, n.value))()
    _check(_lib.ls_get_schedule(ctx.handle, buf, n.value, C.byref(n)), ctx)
    return _events(buf, n.value)


def _stats_dict(s: ls_stats) -> dict:
    return {name: getattr(s, name) for name, _ in ls_stats._fields_}


def ls_get_stats(ctx: Ctx) -> dict:
    s = ls_stats()
    s.struct_size = C.sizeof(ls_stats)
    _check(_lib.ls_get_stats(ctx.handle, C.byref(s)), ctx)
    return _stats_dict(s)


def ls_run_graph(ctx: Ctx, x, y, tokens: int, stream=None) -> int:
    """One pass issued as a CUDA graph replay once the pass is steady (see include/ls_api.h)."""
    return _check(_lib.ls_run_graph(ctx.handle, _ptr(x), _ptr(y), tokens, _stream(stream)), ctx)


def ls_replan(ctx: Ctx, prefetch_depth: int, resident_layers: int, max_vram_bytes: int) -> int:
    """New streaming controls for the next run (see include/ls_api.h)."""
    return _check(_lib.ls_replan(ctx.handle, prefetch_depth, resident_layers, max_vram_bytes), ctx)


def ls_set_kernel_timing(ctx: Ctx, mode: int) -> int:
    return _check(_lib.ls_set_kernel_timing(ctx.handle, mode), ctx)


def ls_get_kernel_times(ctx: Ctx, reset: bool = False) -> dict:
    """{kernel class: (launches, total_ms)} accumulated while kernel_timing is on."""
    n = _I32()
    _check(_lib.ls_get_kernel_times(ctx.handle, None, 0, C.byref(n), 0), ctx)
    buf = (ls_kernel_time * max(1, n.value))()
    _check(_lib.ls_get_kernel_times(ctx.handle, buf, n.value, C.byref(n), int(reset)), ctx)
    return {buf[i].name.decode(): (buf[i].launches, buf[i].total_ms) for i in range(n.value)}


def ls_get_trace(ctx: Ctx) -> list:
    """[(name, stream, segment, start_ms, end_ms)] of the passes the last ls_sync completed."""
    n = _I64()
    _check(_lib.ls_get_trace(ctx.handle, None, 0, C.byref(n)), ctx)
    buf = (ls_trace_event * max(1, n.value))()
    _check(_lib.ls_get_trace(ctx.handle, buf, n.value, C.byref(n)), ctx)
    return [(b.name.decode(), b.stream, b.segment, b.start_ms, b.end_ms) for b in buf[:n.value]]


def ls_ctx_destroy(ctx: Ctx) -> None:
    if ctx and ctx.handle:
        _lib.ls_ctx_destroy(ctx.handle)
        ctx.handle = 0
        ctx.keep.clear()


def ls_last_error(ctx: Ctx) -> str:
    return _lib.ls_last_error(ctx.handle).decode()


def ls_simulate(params: ls_params, seg_slot_bytes, shared=(), runs: int = 1, load_bytes=None):
    """Returns (status, events, stats, run_status) from the library's scheduler
    run without a GPU. shared: [(shared_id, bytes)]; load_bytes: [runs][n] or None."""
    n = len(seg_slot_bytes)
    seg = (_I64 * n)(*seg_slot_bytes)
    sb = (_I64 * max(1, len(shared)))(*[b for _, b in shared])
    sid = (_I32 * max(1, len(shared)))(*[i for i, _ in shared])
    lb = None
    if load_bytes is not None:
        flat = [int(v) for row in load_bytes for v in row]
        lb = (_I64 * len(flat))(*flat)
    total = _I64()
    st = ls_stats()
    st.struct_size = C.sizeof(ls_stats)
    rs = (_I32 * max(1, runs))()
    status = _lib.ls_simulate(C.byref(params), seg, n, sb, sid, len(shared), runs, lb, None, 0,
                              C.byref(total), C.byref(st), rs)
    buf = (ls_sched_event * max(1, total.value))()
    status = _lib.ls_simulate(C.byref(params), seg, n, sb, sid, len(shared), runs, lb, buf,
                              total.value, C.byref(total), C.byref(st), rs)
    return status, _events(buf, total.value), _stats_dict(st), list(rs[:runs])


def ls_simulate_script(params: ls_params, seg_slot_bytes, script, shared=()):
    """ls_simulate along a script of ("run",) and ("replan", depth, resident, max_vram)
    steps. Returns (status, events, stats, step_status)."""
    n = len(seg_slot_bytes)
    seg = (_I64 * n)(*seg_slot_bytes)
    sb = (_I64 * max(1, len(shared)))(*[b for _, b in shared])
    sid = (_I32 * max(1, len(shared)))(*[i for i, _ in shared])
    flat = []
    for step in script:
        flat += [0, 0, 0, 0] if step[0] == "run" else [1, int(step[1]), int(step[2]), int(step[3])]
    sc = (_I64 * max(1, len(flat)))(*flat)
    total = _I64()
    st = ls_stats()
    st.struct_size = C.sizeof(ls_stats)
    ss = (_I32 * max(1, len(script)))(*([1 << 30] * max(1, len(script))))
    status = _lib.ls_simulate_script(C.byref(params), seg, n, sb, sid, len(shared), sc, len(script), None, 0,
                                     C.byref(total), C.byref(st), ss)
    buf = (ls_sched_event * max(1, total.value))()
    ss = (_I32 * max(1, len(script)))(*([1 << 30] * max(1, len(script))))
    status = _lib.ls_simulate_script(C.byref(params), seg, n, sb, sid, len(shared), sc, len(script), buf,
                                     total.value, C.byref(total), C.byref(st), ss)
    steps = [v for v in ss[:len(script)] if v != 1 << 30]
    return status, _events(buf, total.value), _stats_dict(st), steps


# ------------------------------------------------------------------ ls_kernels.h
def lsk_num_sms() -> int:
    return _lib.lsk_num_sms()


def lsk_gemm_tile_n(epilogue: int, M: int, N: int) -> int:
    """Output columns of one tile of lsk_gemm_bf16 for an M x N output on this device."""
    return _lib.lsk_gemm_tile_n(epilogue, M, N)


def lsk_device_error() -> int:
    return _lib.lsk_device_error()


def lsk_copy_h2slot(dst, src_host, nbytes: int, ctas: int, ready, ticket, epoch: int, stream=None) -> int:
    return _check(_lib.lsk_copy_h2slot(_ptr(dst), _ptr(src_host), int(nbytes), ctas, _ptr(ready),
                                       _ptr(ticket), epoch, _stream(stream)))


LSK_STATIC_MAX_RANGES = 64


def lsk_copy_h2slot_static(dst, srcs, sizes, dst_offsets, ctas: int, ready, epoch: int, stream=None) -> int:
    """The copy and publish of lsk_copy_h2slot for up to 64 pinned host ranges,
    without allocating device memory (its scratch is a fixed array in the library)."""
    n = len(srcs)
    src_arr = (_P * max(1, n))(*[_ptr(s) for s in srcs])
    sz = (_U64 * max(1, n))(*[int(b) for b in sizes])
    off = (_U64 * max(1, n))(*[int(o) for o in dst_offsets])
    return _check(_lib.lsk_copy_h2slot_static(_ptr(dst), src_arr, sz, off, n, ctas, _ptr(ready), epoch,
                                              _stream(stream)))


def lsk_wait_ready(ready, epoch: int, limit_ms: int, err_host, slot: int = 0, stream=None) -> int:
    return _check(_lib.lsk_wait_ready(_ptr(ready), epoch, limit_ms, _ptr(err_host), slot, _stream(stream)))


def lsk_gemm_bf16(epilogue: int, A, B, C_out, M: int, N: int, K: int, bias=None, resid=None,
                  b_rows: int | None = None, b2_row_off: int = 0, max_ctas: int = 0, stream=None,
                  C32=None) -> int:
    rows = b_rows if b_rows is not None else B.shape[0]
    rf32 = int(resid is not None and "float32" in str(getattr(resid, "dtype", "")))
    return _check(_lib.lsk_gemm_bf16(epilogue, _ptr(A), _ptr(B), rows, b2_row_off, _ptr(bias),
                                     _ptr(resid), rf32, _ptr(C_out), _ptr(C32), M, N, K, max_ctas,
                                     _stream(stream)))


def lsk_gemm_grouped_bf16(epilogue: int, A, B, b_rows: int, b_base_row: int, b_group_stride_rows: int,
                          b2_row_off: int, group_bounds, n_groups: int, C_out, M: int, N: int, K: int,
                          row_table=None, row_weight=None, max_ctas: int = 0, stream=None) -> int:
    return _check(_lib.lsk_gemm_grouped_bf16(
        epilogue, _ptr(A), _ptr(B), b_rows, b_base_row, b_group_stride_rows, b2_row_off,
        _ptr(group_bounds), n_groups, _ptr(row_table), _ptr(row_weight), _ptr(C_out), M, N, K,
        max_ctas, _stream(stream)))


def lsk_linear_gelu_f32(x, w, b, y, T: int, H: int, F: int, stream=None) -> int:
    return _check(_lib.lsk_linear_gelu_f32(_ptr(x), _ptr(w), _ptr(b), _ptr(y), T, H, F, _stream(stream)))


def lsk_moe_route(logits, n_layers, T, E, k, sel, weight, stream=None) -> int:
    return _check(_lib.lsk_moe_route(_ptr(logits), n_layers, T, E, k, _ptr(sel), _ptr(weight),
                                     _stream(stream)))


def lsk_moe_group(sel, n_layers, T, E, k, row_table, group_bounds, expert_used=None, stream=None) -> int:
    return _check(_lib.lsk_moe_group(_ptr(sel), n_layers, T, E, k, _ptr(row_table), _ptr(group_bounds),
                                     _ptr(expert_used), _stream(stream)))


def lsk_moe_gather(x, row_table, rows, k, H, x_sorted, stream=None) -> int:
    return _check(_lib.lsk_moe_gather(_ptr(x), _ptr(row_table), rows, k, H, _ptr(x_sorted), _stream(stream)))


def lsk_moe_check(sel, row_table, group_bounds, n_layers: int, T: int, k: int, E: int, err_host,
                  stream=None) -> int:
    return _check(_lib.lsk_moe_check(_ptr(sel), _ptr(row_table), _ptr(group_bounds), n_layers, T, k, E,
                                     _ptr(err_host), _stream(stream)))


def lsk_moe_group_masked(sel, n_layers, T, E, k, expert_mask, row_table, group_bounds, expert_used=None,
                         stream=None) -> int:
    return _check(_lib.lsk_moe_group_masked(_ptr(sel), n_layers, T, E, k, _ptr(expert_mask), _ptr(row_table),
                                            _ptr(group_bounds), _ptr(expert_used), _stream(stream)))


def lsk_moe_rows_copy(src, dst, rows: int, H: int, src_table=None, dst_table=None, ready=None, ticket=None,
                      epoch: int = 0, ctas: int = 0, stream=None) -> int:
    return _check(_lib.lsk_moe_rows_copy(_ptr(src), _ptr(src_table), _ptr(dst), _ptr(dst_table), rows, H,
                                         _ptr(ready), _ptr(ticket), epoch, ctas, _stream(stream)))


def ls_host_alloc(nbytes: int) -> int:
    """Pinned, device-mapped host memory of nbytes bytes (address as an int)."""
    p = _P()
    _check(_lib.ls_host_alloc(nbytes, C.byref(p)))
    return p.value


def ls_host_free(ptr: int) -> None:
    _check(_lib.ls_host_free(ptr))


def ls_helper_share(tokens: int) -> float:
    return float(_lib.ls_helper_share(tokens))


def ls_helper_split(routed, share: float):
    """routed: uint8 numpy array [E] (nonzero = routed) -> the helper's mask, uint8 [E]."""
    import numpy as np
    r = np.ascontiguousarray(routed, dtype=np.uint8)
    out = np.zeros_like(r)
    _check(_lib.ls_helper_split(_ptr(r), r.size, share, _ptr(out)))
    return out


def lsk_moe_combine(x, y, T, k, H, out, out32=None, stream=None) -> int:
    xf32 = int("float32" in str(getattr(x, "dtype", "")))
    return _check(_lib.lsk_moe_combine(_ptr(x), xf32, _ptr(y), T, k, H, _ptr(out), _ptr(out32), _stream(stream)))
