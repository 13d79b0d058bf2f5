"""ctypes binding of the moecache C ABI (include/moecache.h).

Argument marshalling only: every step of the layer runs in the CUDA library.
Functions keep the C names; torch tensors may be passed wherever the C API
takes a device pointer (their ``data_ptr()`` is used), and torch streams
wherever it takes a stream.  Importing this module raises if the compiled
library is missing: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

# MOECACHE_LIB selects another build of the library (the bounds-checked one)
_LIB_PATH = os.environ.get("MOECACHE_LIB") or os.path.join(os.path.dirname(os.path.abspath(__file__)), "_lib",
                                                           "libmoecache.so")

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_OOM, MOE_ERR_CAPACITY, MOE_ERR_BUSY, MOE_ERR_CUDA, MOE_ERR_TIMEOUT = range(7)
MOE_FP32, MOE_BF16, MOE_FP4 = 0, 1, 2
MOE_EV_HIT, MOE_EV_MISS, MOE_EV_RESIZE_EVICT, MOE_EV_PREFILL_EVICT = 0, 1, 2, 3
MOE_FILL_COPY, MOE_FILL_DEVICE = 0, 1
MOE_PREFILL_W4A16, MOE_PREFILL_W4A4 = 0, 1
STATUS_NAMES = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_OOM", 3: "MOE_ERR_CAPACITY",
                4: "MOE_ERR_BUSY", 5: "MOE_ERR_CUDA", 6: "MOE_ERR_TIMEOUT"}


class moe_model_desc(ctypes.Structure):
    _fields_ = [("L", ctypes.c_int32), ("E", ctypes.c_int32), ("k", ctypes.c_int32), ("H", ctypes.c_int32),
                ("I", ctypes.c_int32), ("wdtype", ctypes.c_int32), ("has_shared", ctypes.c_int32),
                ("max_tokens", ctypes.c_int32)]


class moe_stats(ctypes.Structure):
    _fields_ = [("calls", ctypes.c_int64), ("tokens", ctypes.c_int64), ("hits", ctypes.c_int64),
                ("misses", ctypes.c_int64), ("evictions", ctypes.c_int64), ("routed_pairs", ctypes.c_int64),
                ("routed_pair_hits", ctypes.c_int64), ("bytes_filled", ctypes.c_int64),
                ("layer_launches", ctypes.c_int64), ("records_streamed", ctypes.c_int64),
                ("layer_ms", ctypes.c_double), ("layer_timed", ctypes.c_int64), ("hit_only_ms", ctypes.c_double),
                ("hit_only_timed", ctypes.c_int64), ("hit_only_records", ctypes.c_int64),
                ("host_wait_us", ctypes.c_double), ("host_issue_us", ctypes.c_double),
                ("resize_calls", ctypes.c_int64), ("resize_moves", ctypes.c_int64),
                ("resize_evictions", ctypes.c_int64), ("prefill_layers", ctypes.c_int64),
                ("prefill_tokens", ctypes.c_int64), ("prefill_ms", ctypes.c_double),
                ("prefill_copy_ms", ctypes.c_double), ("prefill_compute_ms", ctypes.c_double),
                ("prefill_gemm_ms", ctypes.c_double), ("prefill_gemm_flop", ctypes.c_double),
                ("deferred_calls", ctypes.c_int64), ("finish_launches", ctypes.c_int64),
                ("pdl_launches", ctypes.c_int64), ("prefill_records_streamed", ctypes.c_int64),
                ("prefill_records_in_place", ctypes.c_int64), ("qstar_fills", ctypes.c_int64),
                ("summaries_lost", ctypes.c_int64)]

    def as_dict(self):
        return {name: getattr(self, name) for name, _ in self._fields_}


class moe_event(ctypes.Structure):
    _fields_ = [("call", ctypes.c_int64), ("layer", ctypes.c_int32), ("expert", ctypes.c_int32),
                ("kind", ctypes.c_int32), ("slot", ctypes.c_int32), ("evicted_key", ctypes.c_int32),
                ("pad", ctypes.c_int32)]


class moe_layer_aux(ctypes.Structure):
    _fields_ = [("ids", ctypes.c_void_p), ("weights", ctypes.c_void_p), ("slots", ctypes.c_void_p),
                ("perm", ctypes.c_void_p), ("offsets", ctypes.c_void_p), ("logits", ctypes.c_void_p),
                ("qstar", ctypes.c_void_p)]


class moe_prefill_aux(ctypes.Structure):
    _fields_ = [("ids", ctypes.c_void_p), ("weights", ctypes.c_void_p), ("perm", ctypes.c_void_p),
                ("offsets", ctypes.c_void_p), ("slots", ctypes.c_void_p)]


class moe_phase_times(ctypes.Structure):
    _fields_ = [("calls_hit_only", ctypes.c_int64), ("calls_with_fills", ctypes.c_int64),
                ("hit_only_us", ctypes.c_double * 20), ("with_fills_us", ctypes.c_double * 20)]

    def as_dict(self):
        return {"calls_hit_only": self.calls_hit_only, "calls_with_fills": self.calls_with_fills,
                "hit_only_us": list(self.hit_only_us), "with_fills_us": list(self.with_fills_us)}


_P = ctypes.c_void_p
_I32, _I64 = ctypes.c_int32, ctypes.c_int64

# name -> (restype, argtypes); the same list as include/moecache.h
SIGNATURES = {
    "moe_record_bytes": (ctypes.c_size_t, [ctypes.POINTER(moe_model_desc)]),
    "moe_cache_create": (_I32, [ctypes.POINTER(moe_model_desc), _P, _P, _I64, _I64, _P, ctypes.POINTER(_P)]),
    "moe_cache_resize": (_I32, [_P, _I64, _P]),
    "moe_layer_forward": (_I32, [_P, _I32, _P, _P, _P, _I32, _P, _P]),
    "moe_layer_forward_ex": (_I32, [_P, _I32, _P, _P, _P, _I32, _P, _P, ctypes.POINTER(moe_layer_aux)]),
    "moe_prefill_stream": (_I32, [_P, _I32, _I32, _P, _P, _I32, _P, _P]),
    "moe_prefill_stream_ex": (_I32, [_P, _I32, _I32, _P, _P, _I32, _P, _P, ctypes.POINTER(moe_prefill_aux)]),
    "moe_cache_stats": (_I32, [_P, ctypes.POINTER(moe_stats)]),
    "moe_cache_sync": (_I32, [_P, _P]),
    "moe_cache_set_wait_limit_ns": (_I32, [_P, _I64, _I64]),
    "moe_cache_set_split_bandwidths": (_I32, [_P, ctypes.c_double, ctypes.c_double]),
    "moe_cache_reset_stats": (_I32, [_P]),
    "moe_cache_set_profiling": (_I32, [_P, _I32]),
    "moe_cache_phase_times": (_I32, [_P, ctypes.POINTER(moe_phase_times)]),
    "moe_cache_set_trace": (_I32, [_P, _I32]),
    "moe_cache_trace": (_I32, [_P, ctypes.POINTER(moe_event), _I64, ctypes.POINTER(_I64)]),
    "moe_cache_state": (_I32, [_P, _P, _P, _I64, ctypes.POINTER(_I64), ctypes.POINTER(ctypes.c_uint64)]),
    "moe_cache_slot_ptr": (_P, [_P, _I64]),
    "moe_cache_set_fill_mode": (_I32, [_P, _I32]),
    "moe_cache_set_prefill_precision": (_I32, [_P, _I32]),
    "moe_cache_set_graph_mode": (_I32, [_P, _I32]),
    "moe_quantize_fp4": (_I32, [_P, _I32, _I64, _I32, _P, _P, _P]),
    "moe_cache_inject_fill_failure": (_I32, [_P, _I32]),
    "moe_layer_forward_resident_noalloc": (_I32, [ctypes.POINTER(moe_model_desc), _P, _P, _P, _P, _I32, _P, _P]),
    "moe_cache_destroy": (_I32, [_P]),
    "moe_debug_bounds_enabled": (_I32, []),
    "moe_debug_violations": (_I32, [ctypes.POINTER(_I64), ctypes.POINTER(_I32)]),
    "moe_measure_read_rate": (_I32, [_P, _I64, _I32, _I32, _P, ctypes.POINTER(ctypes.c_double)]),
    "moe_last_error": (ctypes.c_char_p, []),
    "moe_version": (_I32, []),
}


def load_library(path: str = _LIB_PATH) -> ctypes.CDLL:
    if not os.path.exists(path):
        raise ImportError(f"moecache CUDA library not built: {path} (run __graft_entry__.build())")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


lib = load_library()


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = lib.moe_last_error().decode(errors="replace")
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}: {msg}")


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if hasattr(t, "data_ptr"):
        return t.data_ptr()
    if hasattr(t, "ctypes"):
        return t.ctypes.data
    raise TypeError(f"cannot take the address of {type(t)}")


def _stream(s) -> int | None:
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream


def check(status: int, where: str) -> None:
    if status != MOE_OK:
        raise MoeError(status, where)


def moe_record_bytes(desc: moe_model_desc) -> int:
    return lib.moe_record_bytes(ctypes.byref(desc))


def moe_cache_create(desc: moe_model_desc, host_pool, shared_dev, n_slots: int, max_slots: int = 0,
                     copy_stream=None) -> int:
    out = _P()
    check(lib.moe_cache_create(ctypes.byref(desc), _ptr(host_pool), _ptr(shared_dev), n_slots, max_slots,
                               _stream(copy_stream), ctypes.byref(out)), "moe_cache_create")
    return out.value


def moe_cache_resize(cache: int, n_slots: int, stream=None) -> None:
    check(lib.moe_cache_resize(cache, n_slots, _stream(stream)), "moe_cache_resize")


def moe_layer_forward(cache: int, layer: int, x, logits, router_w, B: int, y, stream=None, aux=None) -> int:
    """Returns the status (MOE_OK or an error code) without raising for MOE_ERR_CAPACITY / MOE_ERR_CUDA."""
    if aux is None:
        return lib.moe_layer_forward(cache, layer, _ptr(x), _ptr(logits), _ptr(router_w), B, _ptr(y), _stream(stream))
    a = moe_layer_aux(*[_ptr(aux.get(f)) for f, _ in moe_layer_aux._fields_])
    return lib.moe_layer_forward_ex(cache, layer, _ptr(x), _ptr(logits), _ptr(router_w), B, _ptr(y),
                                    _stream(stream), ctypes.byref(a))


def moe_prefill_stream(cache: int, layer_begin: int, layer_end: int, x, logits, T: int, y, stream=None,
                       aux=None) -> int:
    if aux is None:
        return lib.moe_prefill_stream(cache, layer_begin, layer_end, _ptr(x), _ptr(logits), T, _ptr(y),
                                      _stream(stream))
    a = moe_prefill_aux(*[_ptr(aux.get(f)) for f, _ in moe_prefill_aux._fields_])
    return lib.moe_prefill_stream_ex(cache, layer_begin, layer_end, _ptr(x), _ptr(logits), T, _ptr(y),
                                     _stream(stream), ctypes.byref(a))


def moe_cache_stats(cache: int) -> dict:
    st = moe_stats()
    check(lib.moe_cache_stats(cache, ctypes.byref(st)), "moe_cache_stats")
    return st.as_dict()


def moe_cache_sync(cache: int, stream=None) -> int:
    """Waits for the cache's enqueued calls; returns the first error the GPU found after they returned."""
    return lib.moe_cache_sync(cache, _stream(stream))


def moe_cache_set_wait_limit_ns(cache: int, gate_up_ns: int, down_ns: int) -> None:
    check(lib.moe_cache_set_wait_limit_ns(cache, int(gate_up_ns), int(down_ns)), "moe_cache_set_wait_limit_ns")


def moe_cache_set_split_bandwidths(cache: int, b_p: float, b_h: float) -> None:
    check(lib.moe_cache_set_split_bandwidths(cache, float(b_p), float(b_h)), "moe_cache_set_split_bandwidths")


def moe_cache_reset_stats(cache: int) -> None:
    check(lib.moe_cache_reset_stats(cache), "moe_cache_reset_stats")


def moe_cache_set_profiling(cache: int, level: int) -> None:
    check(lib.moe_cache_set_profiling(cache, int(level)), "moe_cache_set_profiling")


def moe_cache_phase_times(cache: int) -> dict:
    pt = moe_phase_times()
    check(lib.moe_cache_phase_times(cache, ctypes.byref(pt)), "moe_cache_phase_times")
    return pt.as_dict()


def moe_cache_set_trace(cache: int, on: bool) -> None:
    check(lib.moe_cache_set_trace(cache, int(on)), "moe_cache_set_trace")


def moe_cache_trace(cache: int) -> list[tuple]:
    n = _I64()
    check(lib.moe_cache_trace(cache, None, 0, ctypes.byref(n)), "moe_cache_trace")
    buf = (moe_event * max(1, n.value))()
    check(lib.moe_cache_trace(cache, buf, n.value, ctypes.byref(n)), "moe_cache_trace")
    return [(e.call, e.layer, e.expert, e.kind, e.slot, e.evicted_key) for e in buf[:n.value]]


def moe_cache_state(cache: int, cap: int):
    import numpy as np

    owner = np.zeros(max(1, cap), dtype=np.int32)
    stamp = np.zeros(max(1, cap), dtype=np.uint64)
    n = _I64()
    g = ctypes.c_uint64()
    check(lib.moe_cache_state(cache, owner.ctypes.data, stamp.ctypes.data, cap, ctypes.byref(n), ctypes.byref(g)),
          "moe_cache_state")
    m = min(cap, n.value)
    return owner[:m].copy(), stamp[:m].copy(), n.value, g.value


def moe_cache_slot_ptr(cache: int, s: int) -> int | None:
    return lib.moe_cache_slot_ptr(cache, s)


def moe_cache_set_fill_mode(cache: int, mode: int) -> None:
    check(lib.moe_cache_set_fill_mode(cache, mode), "moe_cache_set_fill_mode")


def moe_debug_violations() -> tuple[int, int]:
    """(count, first site) of the bounds checks of a debug build (0, 0 otherwise)."""
    n, site = _I64(), _I32()
    check(lib.moe_debug_violations(ctypes.byref(n), ctypes.byref(site)), "moe_debug_violations")
    return n.value, site.value


def moe_measure_read_rate(bufs, nbytes: int, n_bufs: int, reps: int, stream=None) -> float:
    """GB/s of a kernel that only reads nbytes per launch, over n_bufs rotating buffers."""
    g = ctypes.c_double()
    check(lib.moe_measure_read_rate(_ptr(bufs), nbytes, n_bufs, reps, _stream(stream), ctypes.byref(g)),
          "moe_measure_read_rate")
    return g.value


def moe_cache_set_graph_mode(cache: int, on: int) -> None:
    check(lib.moe_cache_set_graph_mode(cache, on), "moe_cache_set_graph_mode")


def moe_cache_set_prefill_precision(cache: int, mode: int) -> None:
    check(lib.moe_cache_set_prefill_precision(cache, mode), "moe_cache_set_prefill_precision")


def moe_quantize_fp4(x, x_dtype: int, rows: int, K: int, codes, scales, stream=None) -> None:
    check(lib.moe_quantize_fp4(_ptr(x), x_dtype, rows, K, _ptr(codes), _ptr(scales), _stream(stream)),
          "moe_quantize_fp4")


def moe_cache_inject_fill_failure(cache: int, after: int) -> None:
    check(lib.moe_cache_inject_fill_failure(cache, after), "moe_cache_inject_fill_failure")


def moe_layer_forward_resident_noalloc(desc: moe_model_desc, bank, shared_rec, x, logits, B: int, y,
                                       stream=None) -> int:
    """Layer over a caller-owned bank of resident experts; allocates nothing (see include/moecache.h)."""
    return lib.moe_layer_forward_resident_noalloc(ctypes.byref(desc), _ptr(bank), _ptr(shared_rec), _ptr(x),
                                                  _ptr(logits), B, _ptr(y), _stream(stream))


def moe_cache_destroy(cache: int) -> None:
    check(lib.moe_cache_destroy(cache), "moe_cache_destroy")


def moe_last_error() -> str:
    return lib.moe_last_error().decode(errors="replace")


def moe_version() -> int:
    return lib.moe_version()
