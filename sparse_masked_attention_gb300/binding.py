"""ctypes binding of libflashmask's C ABI (include/flashmask.h).

Argument marshalling only.  The functions keep the C names and take the same
arguments; a device pointer is a Python int.  Every step of the computation
runs in the CUDA library.  If that library has not been built, loading it
raises, because no other path exists.
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libflashmask.so")

FM_OK = 0
FM_ERR_INVALID_ARG = 1
FM_ERR_UNSUPPORTED = 2
FM_ERR_WORKSPACE = 3
FM_ERR_CUDA = 4
FM_ERR_DEVICE_TIMEOUT = 5
FM_ERR_DEVICE_BOUNDS = 6

FM_TILE_SKIP = 0
FM_TILE_PARTIAL = 1
FM_TILE_UNMASKED = 2


class fm_problem(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("H", ctypes.c_int), ("Hm", ctypes.c_int),
                ("N", ctypes.c_int), ("d", ctypes.c_int), ("dv", ctypes.c_int),
                ("scale", ctypes.c_float), ("causal", ctypes.c_int)]


class fm_options(ctypes.Structure):
    _fields_ = [("deterministic", ctypes.c_int), ("debug_bounds", ctypes.c_int),
                ("wait_timeout_ns", ctypes.c_ulonglong),
                ("kernel_events", ctypes.POINTER(ctypes.c_void_p)),
                ("n_kernel_events", ctypes.c_int),
                ("sink", ctypes.c_void_p), ("dsink", ctypes.c_void_p),
                ("reuse_tile_map", ctypes.c_int), ("accumulate_f32", ctypes.c_int),
                ("debug_drop_load", ctypes.c_int)]


EXPORTS = ("flashmask_workspace_size", "flashmask_fwd", "flashmask_bwd", "flashmask_classify",
           "flashmask_count_unmasked", "flashmask_get_error", "flashmask_error_string",
           "flashmask_last_error_detail", "flashmask_fwd_noalloc", "flashmask_localize",
           "flashmask_merge_init", "flashmask_merge", "flashmask_merge_finish",
           "flashmask_accumulate", "flashmask_to_bf16", "flashmask_selftest_wait")

FM_NOALLOC_SCRATCH_BYTES = 16 * 1024 * 1024

_lock = threading.Lock()
_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libflashmask.so and declare its signatures (raises if missing)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(
                f"libflashmask.so not found at {path}; build it with "
                "`python -m sparse_masked_attention_gb300.build` (no fallback exists)")
        lib = ctypes.CDLL(path)
        P = ctypes.POINTER
        vp = ctypes.c_void_p
        prob, opt = P(fm_problem), P(fm_options)
        lib.flashmask_workspace_size.argtypes = [prob, opt, ctypes.c_int]
        lib.flashmask_workspace_size.restype = ctypes.c_size_t
        lib.flashmask_fwd.argtypes = [prob, opt, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                      ctypes.c_size_t, vp]
        lib.flashmask_fwd.restype = ctypes.c_int
        lib.flashmask_bwd.argtypes = [prob, opt, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                      vp, vp, ctypes.c_size_t, vp]
        lib.flashmask_bwd.restype = ctypes.c_int
        lib.flashmask_classify.argtypes = [prob, vp, vp, vp, vp, vp, vp, ctypes.c_size_t, vp]
        lib.flashmask_classify.restype = ctypes.c_int
        lib.flashmask_count_unmasked.argtypes = [prob, vp, vp, vp, vp, vp, vp]
        lib.flashmask_count_unmasked.restype = ctypes.c_int
        lib.flashmask_get_error.argtypes = [vp]
        lib.flashmask_get_error.restype = ctypes.c_int
        lib.flashmask_selftest_wait.argtypes = [ctypes.c_ulonglong, vp]
        lib.flashmask_selftest_wait.restype = ctypes.c_int
        lib.flashmask_error_string.argtypes = [ctypes.c_int]
        lib.flashmask_error_string.restype = ctypes.c_char_p
        lib.flashmask_fwd_noalloc.argtypes = [prob, opt, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
        lib.flashmask_fwd_noalloc.restype = ctypes.c_int
        ci, ll = ctypes.c_int, ctypes.c_longlong
        lib.flashmask_localize.argtypes = [prob, vp, vp, vp, vp, ci, ci, ci, vp, vp, vp, vp,
                                           P(ci), vp]
        lib.flashmask_merge_init.argtypes = [ci, ci, ci, vp, vp, vp]
        lib.flashmask_merge.argtypes = [ci, ci, ci, vp, vp, vp, vp, vp]
        lib.flashmask_merge_finish.argtypes = [ci, ci, ci, vp, vp, vp, vp, ll, vp]
        lib.flashmask_accumulate.argtypes = [ll, vp, vp, vp]
        lib.flashmask_to_bf16.argtypes = [ll, vp, vp, vp]
        for name in ("flashmask_localize", "flashmask_merge_init", "flashmask_merge",
                     "flashmask_merge_finish", "flashmask_accumulate", "flashmask_to_bf16"):
            getattr(lib, name).restype = ctypes.c_int
        lib.flashmask_last_error_detail.argtypes = []
        lib.flashmask_last_error_detail.restype = ctypes.c_char_p
        _lib = lib
        return lib


def _ref(x):
    return None if x is None else ctypes.byref(x)


def flashmask_workspace_size(problem: fm_problem, options=None, is_bwd: int = 0) -> int:
    return int(load().flashmask_workspace_size(ctypes.byref(problem), _ref(options), is_bwd))


def flashmask_fwd(problem, options, q, k, v, lts, lte, uts, ute, o, lse, workspace, ws_bytes,
                  stream) -> int:
    return int(load().flashmask_fwd(ctypes.byref(problem), _ref(options), q, k, v, lts, lte, uts,
                                    ute, o, lse, workspace, ws_bytes, stream))


def flashmask_bwd(problem, options, q, k, v, o, lse, dout, lts, lte, uts, ute, dq, dk, dv,
                  workspace, ws_bytes, stream) -> int:
    return int(load().flashmask_bwd(ctypes.byref(problem), _ref(options), q, k, v, o, lse, dout,
                                    lts, lte, uts, ute, dq, dk, dv, workspace, ws_bytes, stream))


def flashmask_classify(problem, lts, lte, uts, ute, tile_class, workspace, ws_bytes,
                       stream) -> int:
    return int(load().flashmask_classify(ctypes.byref(problem), lts, lte, uts, ute, tile_class,
                                         workspace, ws_bytes, stream))


def flashmask_count_unmasked(problem, lts, lte, uts, ute, counts, stream) -> int:
    return int(load().flashmask_count_unmasked(ctypes.byref(problem), lts, lte, uts, ute, counts,
                                               stream))


def flashmask_get_error(stream) -> int:
    return int(load().flashmask_get_error(stream))


def flashmask_selftest_wait(timeout_ns, stream) -> int:
    return int(load().flashmask_selftest_wait(int(timeout_ns), stream))


def flashmask_error_string(status: int) -> str:
    return load().flashmask_error_string(status).decode()


def flashmask_last_error_detail() -> str:
    return load().flashmask_last_error_detail().decode()


def flashmask_fwd_noalloc(problem, options, q, k, v, lts, lte, uts, ute, o, lse, stream) -> int:
    return int(load().flashmask_fwd_noalloc(ctypes.byref(problem), _ref(options), q, k, v, lts,
                                            lte, uts, ute, o, lse, stream))


def flashmask_localize(problem, lts, lte, uts, ute, q0, k0, length, out_lts, out_lte, out_uts,
                       out_ute, stream):
    """Returns (status, local causal flag: 1, 0, or -1 for a fully masked pair)."""
    flag = ctypes.c_int(0)
    st = int(load().flashmask_localize(ctypes.byref(problem), lts, lte, uts, ute, q0, k0, length,
                                       out_lts, out_lte, out_uts, out_ute, ctypes.byref(flag),
                                       stream))
    return st, int(flag.value)


def flashmask_merge_init(L, H, dv, o_acc, lse_acc, stream) -> int:
    return int(load().flashmask_merge_init(L, H, dv, o_acc, lse_acc, stream))


def flashmask_merge(L, H, dv, o_part, lse_part, o_acc, lse_acc, stream) -> int:
    return int(load().flashmask_merge(L, H, dv, o_part, lse_part, o_acc, lse_acc, stream))


def flashmask_merge_finish(L, H, dv, o_acc, lse_acc, o_out, lse_out, lse_stride, stream) -> int:
    return int(load().flashmask_merge_finish(L, H, dv, o_acc, lse_acc, o_out, lse_out,
                                             lse_stride, stream))


def flashmask_accumulate(n, part, acc, stream) -> int:
    return int(load().flashmask_accumulate(n, part, acc, stream))


def flashmask_to_bf16(n, src, dst, stream) -> int:
    return int(load().flashmask_to_bf16(n, src, dst, stream))
