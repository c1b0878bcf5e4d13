"""ctypes binding of libpagedattn (``include/pagedattn.h``): argument marshalling only.

Every function here forwards to the C entry point of the same name; all compute runs in
the library's CUDA kernels. Tensor arguments may be torch CUDA tensors or raw device
addresses (int). There is no fallback: if the shared library is missing or fails to load,
``load()`` raises.
"""

from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libpagedattn.so")

PA_OK = 0
STATUS_NAMES = {0: "PA_OK", 1: "PA_ERR_INVALID_ARG", 2: "PA_ERR_UNSUPPORTED",
                3: "PA_ERR_MISALIGNED", 4: "PA_ERR_WORKSPACE", 5: "PA_ERR_CUDA",
                6: "PA_ERR_NO_DEVICE"}
PA_DEVERR_PAGE_ID = 1
PA_DEVERR_CONTEXT = 2
PA_DEVERR_TIMEOUT = 4
PA_DEVERR_QUERY_START = 8
PA_TEST_EXPIRE_WAITS = 1
SCHEDULE = {"auto": 0, "single": 1, "balanced": 2}
MATH = {"auto": 0, "simt": 1, "mma": 2}
COMBINE = {"auto": 0, "fused": 1, "kernel": 2}

# Every entry point include/pagedattn.h declares.
EXPORTS = ("pa_plan", "pa_workspace_size", "pa_workspace_init", "pa_decode", "pa_decode_ex",
           "pa_decode_noalloc", "pa_append_kv", "pa_prefill",
           "pa_split_kv_partial", "pa_split_kv_combine", "pa_get_device_error",
           "pa_status_string", "pa_version")


class PagedAttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}")


class pa_problem_t(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("query_heads", ctypes.c_int32),
                ("kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("max_pages_per_sequence", ctypes.c_int32),
                ("num_physical_pages", ctypes.c_int32), ("cache_layout", ctypes.c_int32)]


class pa_options_t(ctypes.Structure):
    _fields_ = [("schedule", ctypes.c_int32), ("math", ctypes.c_int32),
                ("combine", ctypes.c_int32), ("workers", ctypes.c_int32),
                ("stages", ctypes.c_int32), ("warps_per_cta", ctypes.c_int32),
                ("tile_tokens", ctypes.c_int32), ("test_flags", ctypes.c_int32)]


class pa_plan_t(ctypes.Structure):
    _fields_ = [("schedule", ctypes.c_int32), ("math", ctypes.c_int32),
                ("combine", ctypes.c_int32), ("workers", ctypes.c_int32),
                ("warps_per_cta", ctypes.c_int32), ("ctas", ctypes.c_int32),
                ("stages", ctypes.c_int32), ("tile_tokens", ctypes.c_int32),
                ("units", ctypes.c_int32), ("heads_per_unit", ctypes.c_int32),
                ("group", ctypes.c_int32),
                ("smem_bytes", ctypes.c_int64), ("workspace_bytes", ctypes.c_int64)]


_lib = None
_lock = threading.Lock()


def load(path: Optional[str] = None):
    """Load (building first if the library is absent and nvcc is available)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if path is None:
            from . import build as _build

            p = _build.build()
        lib = ctypes.CDLL(p)
        vp, i32, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float
        P = ctypes.POINTER
        lib.pa_plan.argtypes = [P(pa_problem_t), P(pa_options_t), i32, P(pa_plan_t)]
        lib.pa_workspace_size.argtypes = [P(pa_problem_t), P(pa_options_t), P(ctypes.c_size_t)]
        lib.pa_workspace_init.argtypes = [vp, ctypes.c_size_t, vp]
        lib.pa_decode.argtypes = [P(pa_problem_t), vp, vp, vp, vp, vp, f32, vp, vp]
        lib.pa_decode_ex.argtypes = [P(pa_problem_t), vp, vp, vp, vp, vp, f32, vp, P(pa_options_t),
                                     vp, ctypes.c_size_t, vp]
        lib.pa_decode_noalloc.argtypes = [P(pa_problem_t), vp, vp, vp, vp, vp, f32, vp, vp]
        lib.pa_append_kv.argtypes = [P(pa_problem_t), vp, vp, vp, vp, vp, vp, vp]
        lib.pa_prefill.argtypes = [P(pa_problem_t), vp, vp, ctypes.c_int64, i32, vp, vp, vp, vp,
                                   f32, vp, P(pa_options_t), vp]
        lib.pa_split_kv_partial.argtypes = [P(pa_problem_t), vp, vp, vp, vp, vp, f32, i32, i32, vp,
                                            vp, vp, vp]
        lib.pa_split_kv_combine.argtypes = [P(pa_problem_t), i32, vp, vp, vp, vp, vp]
        lib.pa_get_device_error.argtypes = [vp, P(ctypes.c_uint32)]
        lib.pa_status_string.argtypes = [ctypes.c_int]
        lib.pa_status_string.restype = ctypes.c_char_p
        lib.pa_version.argtypes = []
        for name in EXPORTS:
            if name not in ("pa_status_string",):
                getattr(lib, name).restype = ctypes.c_int
        if path is None:
            _lib = lib
        return lib


# ------------------------------------------------------------------ marshalling helpers
def problem(batch, query_heads, kv_heads, head_dim, page_size, max_pages_per_sequence,
            num_physical_pages, cache_layout=0) -> pa_problem_t:
    return pa_problem_t(batch, query_heads, kv_heads, head_dim, page_size,
                        max_pages_per_sequence, num_physical_pages, cache_layout)


def problem_of(w) -> pa_problem_t:
    """pa_problem_t of a ``workloads.Workload`` (or any object with the same fields)."""
    return problem(w.batch, w.query_heads, w.kv_heads, w.head_dim, w.page_size,
                   w.max_pages_per_sequence, w.num_physical_pages,
                   getattr(w, "cache_layout", 0))


def options(schedule="auto", math="auto", combine="auto", workers=0, stages=0,
            warps_per_cta=0, tile_tokens=0, test_flags=0) -> pa_options_t:
    o = pa_options_t()
    o.schedule = SCHEDULE[schedule] if isinstance(schedule, str) else int(schedule)
    o.math = MATH[math] if isinstance(math, str) else int(math)
    o.combine = COMBINE[combine] if isinstance(combine, str) else int(combine)
    o.workers, o.stages, o.warps_per_cta = int(workers), int(stages), int(warps_per_cta)
    o.tile_tokens = int(tile_tokens)
    o.test_flags = int(test_flags)
    return o


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s):
    if s is None:
        try:
            import torch

            if torch.cuda.is_available():
                return torch.cuda.current_stream().cuda_stream
        except ImportError:
            pass
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(rc: int, where: str):
    if rc != PA_OK:
        raise PagedAttnError(rc, where)


# ------------------------------------------------------------------ entry points
def pa_plan(prob: pa_problem_t, opts: Optional[pa_options_t] = None, sm_count: int = 152) -> dict:
    plan = pa_plan_t()
    _check(load().pa_plan(ctypes.byref(prob), ctypes.byref(opts) if opts else None,
                          int(sm_count), ctypes.byref(plan)), "pa_plan")
    return {name: getattr(plan, name) for name, _ in pa_plan_t._fields_}


def pa_workspace_size(prob: pa_problem_t, opts: Optional[pa_options_t] = None) -> int:
    n = ctypes.c_size_t(0)
    _check(load().pa_workspace_size(ctypes.byref(prob), ctypes.byref(opts) if opts else None,
                                    ctypes.byref(n)), "pa_workspace_size")
    return int(n.value)


def pa_workspace_init(workspace, workspace_bytes: int, stream=None):
    _check(load().pa_workspace_init(_ptr(workspace), int(workspace_bytes), _stream(stream)),
           "pa_workspace_init")


def pa_decode(prob, query, key_cache, value_cache, block_tables, context_lengths, scale, out,
              stream=None):
    _check(load().pa_decode(ctypes.byref(prob), _ptr(query), _ptr(key_cache), _ptr(value_cache),
                            _ptr(block_tables), _ptr(context_lengths), float(scale), _ptr(out),
                            _stream(stream)), "pa_decode")


def pa_decode_ex(prob, query, key_cache, value_cache, block_tables, context_lengths, scale, out,
                 opts: Optional[pa_options_t] = None, workspace=None, workspace_bytes: int = 0,
                 stream=None):
    _check(load().pa_decode_ex(ctypes.byref(prob), _ptr(query), _ptr(key_cache),
                               _ptr(value_cache), _ptr(block_tables), _ptr(context_lengths),
                               float(scale), _ptr(out), ctypes.byref(opts) if opts else None,
                               _ptr(workspace), int(workspace_bytes), _stream(stream)),
           "pa_decode_ex")


def pa_decode_noalloc(prob, query, key_cache, value_cache, block_tables, context_lengths, scale,
                      out, stream=None):
    """pa_decode without any device allocation: split-K scratch comes from a fixed 16 MiB
    array inside the library (for callers that may not allocate; see the header)."""
    _check(load().pa_decode_noalloc(ctypes.byref(prob), _ptr(query), _ptr(key_cache),
                                    _ptr(value_cache), _ptr(block_tables), _ptr(context_lengths),
                                    float(scale), _ptr(out), _stream(stream)), "pa_decode_noalloc")


PA_NOALLOC_SCRATCH_BYTES = 16 * 1024 * 1024


def pa_append_kv(prob, new_key, new_value, block_tables, context_lengths, key_cache, value_cache,
                 stream=None):
    """Write one new K/V row per (sequence, K/V head) at token index context_lengths[b]."""
    _check(load().pa_append_kv(ctypes.byref(prob), _ptr(new_key), _ptr(new_value),
                               _ptr(block_tables), _ptr(context_lengths), _ptr(key_cache),
                               _ptr(value_cache), _stream(stream)), "pa_append_kv")


def pa_prefill(prob, query, query_start, total_tokens, max_query_len, key_cache, value_cache,
               block_tables, context_lengths, scale, out, opts: Optional[pa_options_t] = None,
               stream=None):
    """Causal attention of each sequence's last n_b tokens (query rows query_start[b] ..
    query_start[b + 1]) over its paged cache; fp32 out [total_tokens][query_heads][head_dim]."""
    _check(load().pa_prefill(ctypes.byref(prob), _ptr(query), _ptr(query_start),
                             int(total_tokens), int(max_query_len), _ptr(key_cache),
                             _ptr(value_cache), _ptr(block_tables), _ptr(context_lengths),
                             float(scale), _ptr(out),
                             ctypes.byref(opts) if opts is not None else None,
                             _stream(stream)), "pa_prefill")


def pa_split_kv_partial(prob, query, key_cache, value_cache, block_tables, context_lengths, scale,
                        num_splits, partial_max, partial_sum, partial_out, math="auto",
                        stream=None):
    m = MATH[math] if isinstance(math, str) else int(math)
    _check(load().pa_split_kv_partial(ctypes.byref(prob), _ptr(query), _ptr(key_cache),
                                      _ptr(value_cache), _ptr(block_tables),
                                      _ptr(context_lengths), float(scale), int(num_splits), m,
                                      _ptr(partial_max), _ptr(partial_sum), _ptr(partial_out),
                                      _stream(stream)), "pa_split_kv_partial")


def pa_split_kv_combine(prob, num_splits, partial_max, partial_sum, partial_out, out, stream=None):
    _check(load().pa_split_kv_combine(ctypes.byref(prob), int(num_splits), _ptr(partial_max),
                                      _ptr(partial_sum), _ptr(partial_out), _ptr(out),
                                      _stream(stream)), "pa_split_kv_combine")


def pa_get_device_error(stream=None) -> int:
    flags = ctypes.c_uint32(0)
    _check(load().pa_get_device_error(_stream(stream), ctypes.byref(flags)),
           "pa_get_device_error")
    return int(flags.value)


def pa_status_string(status: int) -> str:
    return load().pa_status_string(int(status)).decode()


def pa_version() -> int:
    return int(load().pa_version())


def status_of(fn, *args, **kw) -> int:
    """Call a binding and return the C status instead of raising (for tests)."""
    try:
        fn(*args, **kw)
    except PagedAttnError as e:
        return e.status
    return PA_OK
