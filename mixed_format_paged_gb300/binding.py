"""ctypes binding of ``libmkv.so`` (C ABI in ``include/mkv.h``).

Argument marshalling only: every function here forwards to the C call of the
same name.  Device buffers are passed as raw pointers (``tensor.data_ptr()``)
and streams as ``torch.cuda.Stream.cuda_stream`` integers; nothing here
computes on cache data.  Importing fails loudly when the library has not been
built (there is no fallback path).
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmkv.so")

MKV_OK = 0
STATUS_NAMES = {
    0: "MKV_OK", 1: "MKV_ERR_INVALID_ARGUMENT", 2: "MKV_ERR_UNSUPPORTED", 3: "MKV_ERR_OUT_OF_PAGES",
    4: "MKV_ERR_INVALID_STATE", 5: "MKV_ERR_CUDA", 6: "MKV_ERR_DEVICE_CHECK", 7: "MKV_ERR_CAPACITY",
}
MKV_TIER_NONE, MKV_TIER_RECENT, MKV_TIER_ANCHOR, MKV_TIER_STALE = 0, 1, 2, 3
MKV_F32, MKV_BF16 = 0, 1
MKV_POOL_HOST_ONLY = 1

# every exported symbol of include/mkv.h
EXPORTED = [
    "mkv_pool_required_bytes", "mkv_pool_create", "mkv_pool_destroy", "mkv_seq_extend", "mkv_seq_release",
    "mkv_seq_info", "mkv_page_info", "mkv_append_tokens", "mkv_set_tier", "mkv_demote_pages",
    "mkv_decode_attention", "mkv_decode_attention_multi", "mkv_decode_attention_noalloc", "mkv_append_decode", "mkv_dequantize_pages", "mkv_pool_stats", "mkv_export_page", "mkv_rotation_signs", "mkv_tq3_codebook",
    "mkv_plan_decode", "mkv_plan_decode_multi", "mkv_check_device_errors", "mkv_selftest_wait_timeout", "mkv_inject_plan_slot", "mkv_set_timing_events", "mkv_last_error", "mkv_version",
    "mkv_step_graph_create", "mkv_step_graph_launch", "mkv_step_graph_destroy", "mkv_page_relevance",
]


class MkvError(RuntimeError):
    def __init__(self, status: int, where: str, message: str):
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


class PoolConfig(ctypes.Structure):
    _fields_ = [
        ("num_layers", ctypes.c_int32), ("num_q_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32), ("page_size", ctypes.c_int32), ("fp8_slots", ctypes.c_int32),
        ("tq3_slots", ctypes.c_int32), ("max_seqs", ctypes.c_int32), ("max_pages_per_seq", ctypes.c_int32),
        ("max_batch", ctypes.c_int32), ("flags", ctypes.c_int32), ("reserved", ctypes.c_int32),
        ("rotation_seed", ctypes.c_uint64),
    ]


class Stats(ctypes.Structure):
    _fields_ = [
        ("recent_pages", ctypes.c_int64), ("anchor_pages", ctypes.c_int64), ("stale_pages", ctypes.c_int64),
        ("live_tokens", ctypes.c_int64), ("fp8_bytes", ctypes.c_int64), ("tq3_bytes", ctypes.c_int64),
        ("kv_bytes_per_live_token", ctypes.c_double), ("fp8_slots_free", ctypes.c_int32),
        ("tq3_slots_free", ctypes.c_int32), ("device_bytes", ctypes.c_int64), ("workspace_bytes", ctypes.c_int64),
    ]


_lib = None


def lib() -> ctypes.CDLL:
    """Load libmkv.so (once).  Raises if it is missing: build it first with
    ``python -m mixed_format_paged_gb300.build``."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing; build it with `python -m mixed_format_paged_gb300.build`")
    L = ctypes.CDLL(LIB_PATH)
    P = ctypes.c_void_p
    I32 = ctypes.c_int32
    I32P = ctypes.POINTER(ctypes.c_int32)
    sig = {
        "mkv_pool_required_bytes": [ctypes.POINTER(PoolConfig), ctypes.POINTER(ctypes.c_size_t)],
        "mkv_pool_create": [ctypes.POINTER(PoolConfig), P, ctypes.c_size_t, P, ctypes.POINTER(P)],
        "mkv_pool_destroy": [P],
        "mkv_seq_extend": [P, I32, I32P, I32P],
        "mkv_seq_release": [P, I32],
        "mkv_seq_info": [P, I32, I32P, I32P],
        "mkv_page_info": [P, I32, I32, I32P, I32P],
        "mkv_append_tokens": [P, I32, I32, I32P, I32P, P, P, ctypes.c_int, P],
        "mkv_set_tier": [P, I32, I32, ctypes.c_int],
        "mkv_demote_pages": [P, I32, I32P, I32P, P],
        "mkv_decode_attention": [P, I32, I32, I32P, P, ctypes.c_int, P, P, P],
        "mkv_decode_attention_multi": [P, I32, I32, I32P, I32, P, ctypes.c_int, P, P, P],
        "mkv_decode_attention_noalloc": [P, I32, I32, I32P, P, ctypes.c_int, P, P, P],
        "mkv_append_decode": [P, I32, I32, I32P, P, P, ctypes.c_int, P, ctypes.c_int, P, P, P],
        "mkv_dequantize_pages": [P, I32, I32, I32, I32, P, P, ctypes.c_int, P],
        "mkv_pool_stats": [P, ctypes.POINTER(Stats)],
        "mkv_export_page": [P, I32, I32, I32, P, ctypes.c_size_t, I32P, I32P, P],
        "mkv_rotation_signs": [P, ctypes.POINTER(ctypes.c_int8), I32],
        "mkv_tq3_codebook": [ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_float)],
        "mkv_plan_decode": [P, I32, I32P, I32P, I32, I32P],
        "mkv_plan_decode_multi": [P, I32, I32P, I32, I32P, I32, I32P],
        "mkv_check_device_errors": [P, P],
        "mkv_selftest_wait_timeout": [P, ctypes.c_int64, P],
        "mkv_inject_plan_slot": [P, I32, I32, P],
        "mkv_set_timing_events": [P, P, P],
        "mkv_step_graph_create": [P, I32, I32P, ctypes.POINTER(P), ctypes.POINTER(P), ctypes.POINTER(P),
                                  ctypes.c_int, ctypes.c_int, ctypes.POINTER(P), ctypes.POINTER(P), P,
                                  ctypes.POINTER(P)],
        "mkv_step_graph_launch": [P, P],
        "mkv_page_relevance": [P, I32, I32, I32P, P, ctypes.c_int, P, P, I32, P],
        "mkv_step_graph_destroy": [P],
        "mkv_last_error": [],
        "mkv_version": [],
    }
    for name, args in sig.items():
        f = getattr(L, name)
        f.argtypes = args
        f.restype = ctypes.c_char_p if name in ("mkv_last_error", "mkv_version") else ctypes.c_int
    _lib = L
    return L


def check(status: int, where: str) -> None:
    if status != MKV_OK:
        raise MkvError(status, where, lib().mkv_last_error().decode())


_I32_CACHE: dict = {}


def _i32(values):
    """int32 C array of `values` (small arrays are cached: the same batch is
    passed for every layer of a decode step)."""
    key = tuple(int(v) for v in values)
    hit = _I32_CACHE.get(key)
    if hit is None:
        hit = ((ctypes.c_int32 * max(1, len(key)))(*key), len(key))
        if len(key) <= 256:
            if len(_I32_CACHE) > 4096:
                _I32_CACHE.clear()
            _I32_CACHE[key] = hit
    return hit


def _ptr(x) -> ctypes.c_void_p:
    if x is None:
        return ctypes.c_void_p(None)
    if isinstance(x, int):
        return ctypes.c_void_p(x)
    return ctypes.c_void_p(x.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        return ctypes.c_void_p(None)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


# ----------------------------------------------------------------- C names
def mkv_pool_required_bytes(cfg: PoolConfig) -> int:
    out = ctypes.c_size_t()
    check(lib().mkv_pool_required_bytes(ctypes.byref(cfg), ctypes.byref(out)), "mkv_pool_required_bytes")
    return out.value


def mkv_pool_create(cfg: PoolConfig, device_buf, nbytes: int, stream=None) -> ctypes.c_void_p:
    h = ctypes.c_void_p()
    check(lib().mkv_pool_create(ctypes.byref(cfg), _ptr(device_buf), nbytes, _stream(stream), ctypes.byref(h)),
          "mkv_pool_create")
    return h


def mkv_pool_destroy(pool) -> None:
    check(lib().mkv_pool_destroy(pool), "mkv_pool_destroy")


def mkv_seq_extend(pool, seq_ids, n_new) -> None:
    a, n = _i32(seq_ids)
    b, _ = _i32(n_new)
    check(lib().mkv_seq_extend(pool, n, a, b), "mkv_seq_extend")


def mkv_seq_release(pool, seq: int) -> None:
    check(lib().mkv_seq_release(pool, seq), "mkv_seq_release")


def mkv_seq_info(pool, seq: int):
    ln, npg = ctypes.c_int32(), ctypes.c_int32()
    check(lib().mkv_seq_info(pool, seq, ctypes.byref(ln), ctypes.byref(npg)), "mkv_seq_info")
    return ln.value, npg.value


def mkv_page_info(pool, seq: int, page: int):
    t, s = ctypes.c_int32(), ctypes.c_int32()
    check(lib().mkv_page_info(pool, seq, page, ctypes.byref(t), ctypes.byref(s)), "mkv_page_info")
    return t.value, s.value


def mkv_append_tokens(pool, layer: int, seq_ids, n_new, k, v, dtype: int, stream=None) -> None:
    a, n = _i32(seq_ids)
    b, _ = _i32(n_new)
    check(lib().mkv_append_tokens(pool, layer, n, a, b, _ptr(k), _ptr(v), dtype, _stream(stream)),
          "mkv_append_tokens")


def mkv_set_tier(pool, seq: int, page: int, tier: int) -> None:
    check(lib().mkv_set_tier(pool, seq, page, tier), "mkv_set_tier")


def mkv_demote_pages(pool, seq_ids, pages, stream=None) -> None:
    a, n = _i32(seq_ids)
    b, _ = _i32(pages)
    check(lib().mkv_demote_pages(pool, n, a, b, _stream(stream)), "mkv_demote_pages")


def mkv_decode_attention(pool, layer: int, seq_ids, q, dtype: int, out, lse, stream=None) -> None:
    a, n = _i32(seq_ids)
    check(lib().mkv_decode_attention(pool, layer, n, a, _ptr(q), dtype, _ptr(out), _ptr(lse), _stream(stream)),
          "mkv_decode_attention")


def mkv_decode_attention_multi(pool, layer: int, seq_ids, nq: int, q, dtype: int, out, lse, stream=None) -> None:
    a, n = _i32(seq_ids)
    check(lib().mkv_decode_attention_multi(pool, layer, n, a, nq, _ptr(q), dtype, _ptr(out), _ptr(lse),
                                           _stream(stream)), "mkv_decode_attention_multi")


def mkv_decode_attention_noalloc(pool, layer: int, seq_ids, q, dtype: int, out, lse, stream=None) -> None:
    """mkv_decode_attention with its scratch in the library's fixed device
    array: for callers that may not allocate device memory during a call."""
    a, n = _i32(seq_ids)
    check(lib().mkv_decode_attention_noalloc(pool, layer, n, a, _ptr(q), dtype, _ptr(out), _ptr(lse),
                                             _stream(stream)), "mkv_decode_attention_noalloc")


def mkv_append_decode(pool, layer: int, seq_ids, k, v, kv_dtype: int, q, q_dtype: int, out, lse,
                      stream=None) -> None:
    a, n = _i32(seq_ids)
    check(lib().mkv_append_decode(pool, layer, n, a, _ptr(k), _ptr(v), kv_dtype, _ptr(q), q_dtype, _ptr(out),
                                  _ptr(lse), _stream(stream)), "mkv_append_decode")


def mkv_page_relevance(pool, layer: int, seq_ids, q, q_dtype: int, lse, mass, mass_stride: int,
                       stream=None) -> None:
    a, n = _i32(seq_ids)
    check(lib().mkv_page_relevance(pool, layer, n, a, _ptr(q), q_dtype, _ptr(lse), _ptr(mass), mass_stride,
                                   _stream(stream)), "mkv_page_relevance")


def _ptr_array(xs):
    """Array of device pointers (one per layer), or NULL for None."""
    if xs is None:
        return None
    arr = (ctypes.c_void_p * len(xs))(*[_ptr(x).value for x in xs])
    return ctypes.cast(arr, ctypes.POINTER(ctypes.c_void_p)), arr


def mkv_step_graph_create(pool, seq_ids, q, k, v, q_dtype: int, kv_dtype: int, out, lse, stream=None):
    """q, k, v, out, lse: one device buffer per layer (k = v = None: no fused
    append).  Returns the graph handle."""
    a, n = _i32(seq_ids)
    keep = [_ptr_array(x) for x in (q, k, v, out, lse)]
    args = [x[0] if x is not None else None for x in keep]
    g = ctypes.c_void_p()
    check(lib().mkv_step_graph_create(pool, n, a, args[0], args[1], args[2], q_dtype, kv_dtype, args[3], args[4],
                                      _stream(stream), ctypes.byref(g)), "mkv_step_graph_create")
    return g


def mkv_step_graph_launch(graph, stream=None) -> None:
    check(lib().mkv_step_graph_launch(graph, _stream(stream)), "mkv_step_graph_launch")


def mkv_step_graph_destroy(graph) -> None:
    check(lib().mkv_step_graph_destroy(graph), "mkv_step_graph_destroy")


def mkv_dequantize_pages(pool, layer: int, seq: int, page0: int, npages: int, k_out, v_out, out_dtype: int,
                         stream=None) -> None:
    check(lib().mkv_dequantize_pages(pool, layer, seq, page0, npages, _ptr(k_out), _ptr(v_out), out_dtype,
                                     _stream(stream)), "mkv_dequantize_pages")


def mkv_pool_stats(pool) -> Stats:
    st = Stats()
    check(lib().mkv_pool_stats(pool, ctypes.byref(st)), "mkv_pool_stats")
    return st


def mkv_export_page(pool, layer: int, seq: int, page: int, nbytes: int, stream=None):
    """Returns (bytes, tier, n_valid)."""
    buf = (ctypes.c_uint8 * nbytes)()
    t, nv = ctypes.c_int32(), ctypes.c_int32()
    check(lib().mkv_export_page(pool, layer, seq, page, ctypes.cast(buf, ctypes.c_void_p), nbytes,
                                ctypes.byref(t), ctypes.byref(nv), _stream(stream)), "mkv_export_page")
    return bytes(buf), t.value, nv.value


def mkv_rotation_signs(pool, d: int = 256):
    buf = (ctypes.c_int8 * d)()
    check(lib().mkv_rotation_signs(pool, buf, d), "mkv_rotation_signs")
    return list(buf)


def mkv_tq3_codebook():
    lv = (ctypes.c_float * 8)()
    th = (ctypes.c_float * 7)()
    check(lib().mkv_tq3_codebook(lv, th), "mkv_tq3_codebook")
    return list(lv), list(th)


PLAN_RECORD = 9   # ints per split: b, kv head, tier, first entry, pages, tokens, CTA, first block, blocks


def mkv_plan_decode(pool, seq_ids):
    a, n = _i32(seq_ids)
    nc = ctypes.c_int32()
    check(lib().mkv_plan_decode(pool, n, a, None, 0, ctypes.byref(nc)), "mkv_plan_decode")
    buf = (ctypes.c_int32 * max(1, PLAN_RECORD * nc.value))()
    check(lib().mkv_plan_decode(pool, n, a, buf, nc.value, ctypes.byref(nc)), "mkv_plan_decode")
    return [tuple(buf[PLAN_RECORD * i: PLAN_RECORD * (i + 1)]) for i in range(nc.value)]


def mkv_plan_decode_multi(pool, seq_ids, nq: int):
    a, n = _i32(seq_ids)
    nc = ctypes.c_int32()
    check(lib().mkv_plan_decode_multi(pool, n, a, nq, None, 0, ctypes.byref(nc)), "mkv_plan_decode_multi")
    buf = (ctypes.c_int32 * max(1, PLAN_RECORD * nc.value))()
    check(lib().mkv_plan_decode_multi(pool, n, a, nq, buf, nc.value, ctypes.byref(nc)), "mkv_plan_decode_multi")
    return [tuple(buf[PLAN_RECORD * i: PLAN_RECORD * (i + 1)]) for i in range(nc.value)]


def mkv_check_device_errors(pool, stream=None) -> None:
    check(lib().mkv_check_device_errors(pool, _stream(stream)), "mkv_check_device_errors")


def mkv_selftest_wait_timeout(pool, limit_cycles: int, stream=None) -> None:
    check(lib().mkv_selftest_wait_timeout(pool, limit_cycles, _stream(stream)), "mkv_selftest_wait_timeout")


def mkv_inject_plan_slot(pool, entry: int, slot: int, stream=None) -> None:
    check(lib().mkv_inject_plan_slot(pool, entry, slot, _stream(stream)), "mkv_inject_plan_slot")


def mkv_set_timing_events(pool, start_event, stop_event) -> None:
    """start/stop: torch.cuda.Event (created with enable_timing=True) or None."""
    def h(e):
        if e is None:
            return ctypes.c_void_p(None)
        if not e.cuda_event:
            raise ValueError("torch creates a CUDA event on its first record(); record it once before passing it")
        return ctypes.c_void_p(e.cuda_event)
    check(lib().mkv_set_timing_events(pool, h(start_event), h(stop_event)), "mkv_set_timing_events")


def mkv_version() -> str:
    return lib().mkv_version().decode()
