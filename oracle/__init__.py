"""fp64 CPU oracle for FlashMask masked attention (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its binding) never imports, links or runs it, and the two share no code.

The arithmetic lives in ``oracle.c`` (plain C, double precision, OpenMP over
rows); this module only compiles it with the host C compiler and marshals
numpy arrays.  What it computes, with the passages it follows:

* FlashMask README (PaddlePaddle/FlashMask), "Formulation":
  ``O = softmax(Q K^T / sqrt(d) + M) V``, ``d`` the Q/K head dim.
* FlashMask README "Overview" and the FlashMask-3 abstract: the mask is given
  per key column ``j`` as query-row intervals ``[LTS_j, LTE_j)`` and
  ``[UTS_j, UTE_j)``; ``causal`` also masks ``i < j``.
* Fully masked rows give ``O = 0``, ``LSE = -inf`` and no gradient (stated
  convention; the pages are silent).
* Attention-sink bias (FlashMask README, "News", which names it without a
  formula; reading taken): a per-head logit ``sink`` joins every row's
  softmax denominator as a term ``exp(sink)`` with no value, so
  ``O_i = sum_j exp(s_ij) v_j / (exp(sink) + sum_j exp(s_ij))`` and
  ``LSE_i = log(exp(sink) + sum_j exp(s_ij))``; its gradient is
  ``-sum_i P_sink,i D_i`` with ``P_sink,i = exp(sink - LSE_i)``.
* The backward pass is the plain derivative of the formula.
* The tile map is a brute-force count of masked elements per tile.
"""
from __future__ import annotations

import ctypes
import os
import platform
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, f"liboracle_{platform.machine()}.so")

TILE_SKIP = 0
TILE_PARTIAL = 1
TILE_UNMASKED = 2

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into a shared library for this host; return its path."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c99",
               "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        dp = ctypes.POINTER(ctypes.c_double)
        ip = ctypes.POINTER(ctypes.c_int32)
        lp = ctypes.POINTER(ctypes.c_int64)
        i8p = ctypes.POINTER(ctypes.c_int8)
        head = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_int,
                ctypes.c_double, dp, dp, dp]
        vec = [ip, ip, ip, ip]
        lib.oracle_fwd.argtypes = head + vec + [ctypes.c_long, lp, dp, dp]
        lib.oracle_fwd.restype = ctypes.c_int
        lib.oracle_bwd_dq.argtypes = head + [dp] + vec + [ctypes.c_long, lp, dp, dp, dp]
        lib.oracle_bwd_dq.restype = ctypes.c_int
        lib.oracle_bwd_dkdv.argtypes = head + [dp] + vec + [ctypes.c_long, lp, dp, dp]
        lib.oracle_bwd_dkdv.restype = ctypes.c_int
        lib.oracle_tilemap.argtypes = [ctypes.c_int, ctypes.c_int] + vec + [
            ctypes.c_int, ctypes.c_int, i8p]
        lib.oracle_tilemap.restype = ctypes.c_longlong
        lib.oracle_num_threads.argtypes = []
        lib.oracle_num_threads.restype = ctypes.c_int
        _lib = lib
        return lib


def num_threads() -> int:
    return int(_load().oracle_num_threads())


# ---------------------------------------------------------------- marshalling
def _f64(a, shape=None) -> np.ndarray:
    a = np.ascontiguousarray(np.asarray(a, dtype=np.float64))
    if shape is not None and a.shape != tuple(shape):
        raise ValueError(f"expected shape {shape}, got {a.shape}")
    return a


def _vecs(mask, N):
    """mask: dict with optional int32 vectors lts/lte/uts/ute of length N."""
    out = []
    keep = []
    for name in ("lts", "lte", "uts", "ute"):
        x = None if mask is None else mask.get(name)
        if x is None:
            out.append(None)
            continue
        x = np.ascontiguousarray(np.asarray(x, dtype=np.int32))
        if x.shape != (N,):
            raise ValueError(f"{name}: expected shape ({N},), got {x.shape}")
        keep.append(x)
        out.append(x.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)))
    return out, keep


def _idx(idx):
    if idx is None:
        return None, None
    a = np.ascontiguousarray(np.asarray(idx, dtype=np.int64))
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))


def _dptr(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _sink(sink):
    return -np.inf if sink is None else float(sink)


def attention_fwd(q, k, v, mask=None, causal=False, scale=None, rows=None, sink=None):
    """One (batch, head) slice.  q, k: [N, d]; v: [N, dv].  `sink`: the head's
    attention-sink logit (None: no sink), a term exp(sink) of every row's
    softmax denominator that carries no value.

    Returns (o [n_rows, dv], lse [n_rows]) in float64.
    """
    q = _f64(q)
    N, d = q.shape
    k = _f64(k, (N, d))
    v = _f64(v)
    dv = v.shape[1]
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    vec, _keep = _vecs(mask, N)
    rows_a, rows_p = _idx(rows)
    n = N if rows_a is None else len(rows_a)
    o = np.zeros((n, dv), np.float64)
    lse = np.zeros((n,), np.float64)
    rc = _load().oracle_fwd(N, d, dv, float(scale), int(bool(causal)), _sink(sink), _dptr(q),
                            _dptr(k), _dptr(v), *vec, n, rows_p, _dptr(o), _dptr(lse))
    if rc:
        raise MemoryError("oracle_fwd: allocation failed")
    return o, lse


def attention_bwd_dq(q, k, v, dout, mask=None, causal=False, scale=None, rows=None, sink=None,
                     with_dsink=False):
    """Returns (dq [n_rows, d], delta [n_rows]) for one (batch, head) slice, and
    with `with_dsink` also the rows' terms of the sink logit's gradient."""
    q = _f64(q)
    N, d = q.shape
    k = _f64(k, (N, d))
    v = _f64(v)
    dv = v.shape[1]
    dout = _f64(dout, (N, dv))
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    vec, _keep = _vecs(mask, N)
    rows_a, rows_p = _idx(rows)
    n = N if rows_a is None else len(rows_a)
    dq = np.zeros((n, d), np.float64)
    delta = np.zeros((n,), np.float64)
    dsink = np.zeros((n,), np.float64)
    rc = _load().oracle_bwd_dq(N, d, dv, float(scale), int(bool(causal)), _sink(sink), _dptr(q),
                               _dptr(k), _dptr(v), _dptr(dout), *vec, n, rows_p, _dptr(dq),
                               _dptr(delta), _dptr(dsink))
    if rc:
        raise MemoryError("oracle_bwd_dq: allocation failed")
    return (dq, delta, dsink) if with_dsink else (dq, delta)


def attention_bwd_dkdv(q, k, v, dout, mask=None, causal=False, scale=None, cols=None,
                       sink=None):
    """Returns (dk [n_cols, d], dv [n_cols, dv]) for one (batch, head) slice."""
    q = _f64(q)
    N, d = q.shape
    k = _f64(k, (N, d))
    v = _f64(v)
    dv = v.shape[1]
    dout = _f64(dout, (N, dv))
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    vec, _keep = _vecs(mask, N)
    cols_a, cols_p = _idx(cols)
    n = N if cols_a is None else len(cols_a)
    dk = np.zeros((n, d), np.float64)
    dvv = np.zeros((n, dv), np.float64)
    rc = _load().oracle_bwd_dkdv(N, d, dv, float(scale), int(bool(causal)), _sink(sink),
                                 _dptr(q), _dptr(k), _dptr(v), _dptr(dout), *vec, n, cols_p,
                                 _dptr(dk), _dptr(dvv))
    if rc:
        raise MemoryError("oracle_bwd_dkdv: allocation failed")
    return dk, dvv


def attention_bwd(q, k, v, dout, mask=None, causal=False, scale=None, sink=None):
    """Full backward of one (batch, head) slice: (dq, dk, dv), and with a sink
    also the gradient of its logit: (dq, dk, dv, dsink)."""
    dq, _, ds = attention_bwd_dq(q, k, v, dout, mask, causal, scale, sink=sink, with_dsink=True)
    dk, dvv = attention_bwd_dkdv(q, k, v, dout, mask, causal, scale, sink=sink)
    return (dq, dk, dvv) if sink is None else (dq, dk, dvv, float(ds.sum()))


def tilemap(N, mask=None, causal=False, tq=128, tk=128):
    """Brute-force tile classes [ceil(N/tq), ceil(N/tk)] (int8) and the number
    of unmasked pairs over the N x N square."""
    vec, _keep = _vecs(mask, N)
    nq, nk = -(-N // tq), -(-N // tk)
    cls = np.zeros((nq, nk), np.int8)
    total = _load().oracle_tilemap(int(N), int(bool(causal)), *vec, int(tq), int(tk),
                                   cls.ctypes.data_as(ctypes.POINTER(ctypes.c_int8)))
    return cls, int(total)


def count_unmasked(N, mask=None, causal=False):
    """Brute-force number of unmasked (i, j) pairs of one mask."""
    vec, _keep = _vecs(mask, N)
    return int(_load().oracle_tilemap(int(N), int(bool(causal)), *vec, 128, 128, None))


# ------------------------------------------------ context-parallel chunks
def localize(mask, N, causal, q0, k0, length):
    """Column-wise vectors of the local problem of one (query chunk, key chunk)
    pair, the sequence being cut into chunks of `length` rows and keys that
    start at multiples of `length` (FlashMask-3 abstract: under a multi-chunk
    context-parallel assignment, mask localization is a zero-communication
    clip-shift-max on the boundary vectors).

    Local row i' = i - q0 and local key j' = j - k0.  Each interval of key
    column j, clamped to [0, N] as everywhere, is clipped to the query chunk,
    shifted by its start and kept non-negative:
    ``x' = max(min(x, q0 + length) - q0, 0)``.  The causal flag ``i < j``:
    on the diagonal pair (q0 == k0) it is the local flag ``i' < j'``; a key
    chunk before the query chunk has ``i > j`` everywhere, so no flag; a key
    chunk after it is masked everywhere.

    Returns (dict of four [length] int32 arrays, local causal flag), or
    (None, None) when every element of the pair is masked."""
    assert 0 <= q0 and q0 + length <= N and 0 <= k0 and k0 + length <= N
    assert (q0 - k0) % length == 0
    if causal and k0 > q0:
        return None, None
    local_causal = bool(causal) and k0 == q0
    mask = mask or {}
    empty = {"lts": N, "lte": N, "uts": 0, "ute": 0}
    out = {}
    for name in ("lts", "lte", "uts", "ute"):
        x = mask.get(name)
        x = (np.full(length, empty[name], np.int64) if x is None
             else np.clip(np.asarray(x, np.int64)[k0:k0 + length], 0, N))
        out[name] = np.maximum(np.minimum(x, q0 + length) - q0, 0).astype(np.int32)
    return out, local_causal
