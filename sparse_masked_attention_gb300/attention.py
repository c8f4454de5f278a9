"""PyTorch front end over the C ABI.

torch supplies device memory and the current stream; the work runs in the
CUDA library through ``binding``.  Layouts follow the C ABI:
q, k ``[B, N, H, d]``; v ``[B, N, H, dv]`` (bf16, contiguous); mask vectors
``[B, Hm, N]`` int32 with ``Hm`` in ``{1, H}``; lse ``[B, H, N]`` fp32.
"""
from __future__ import annotations

import ctypes
import math
from typing import Optional

import torch

from . import binding as _b


class FlashMaskError(RuntimeError):
    """An error of the library or of its arguments; `status` is the library's
    fm_status code, or None for a check made in Python."""

    def __init__(self, message, status=None):
        super().__init__(message)
        self.status = status


def _check(status: int, what: str):
    if status != _b.FM_OK:
        detail = _b.flashmask_last_error_detail() if status == _b.FM_ERR_CUDA else ""
        raise FlashMaskError(f"{what}: {_b.flashmask_error_string(status)} (status {status})"
                             + (f" [{detail}]" if detail else ""), status)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


_nvtx = False


def set_nvtx(enabled: bool) -> None:
    """Wrap every forward and backward launch sequence in an NVTX range
    ("flashmask_fwd N=... d=..."), so profiler timelines show which kernels
    belong to which call.  Off by default: a range costs host time per call."""
    global _nvtx
    _nvtx = bool(enabled)


class _Range:
    def __init__(self, name):
        self.name = name

    def __enter__(self):
        if _nvtx:
            torch.cuda.nvtx.range_push(self.name)

    def __exit__(self, *exc):
        if _nvtx:
            torch.cuda.nvtx.range_pop()
        return False


def _same_device(a: torch.device, b: torch.device) -> bool:
    if a.type != b.type:
        return False
    ia = a.index if a.index is not None else torch.cuda.current_device()
    ib = b.index if b.index is not None else torch.cuda.current_device()
    return ia == ib


def _mask_args(masks, B: int, H: int, N: int, device):
    """Validate the four boundary vectors; returns (Hm, [ptr x 4], keep-alive)."""
    Hm = None
    keep = []
    for name, t in zip(("lts", "lte", "uts", "ute"), masks):
        if t is None:
            keep.append(None)
            continue
        if t.dtype != torch.int32 or not _same_device(t.device, device) or not t.is_contiguous():
            raise FlashMaskError(f"{name} must be a contiguous int32 tensor on {device}")
        if t.dim() != 3 or t.shape[0] != B or t.shape[2] != N or t.shape[1] not in (1, H):
            raise FlashMaskError(f"{name} must have shape [B, 1 or H, N], got {tuple(t.shape)}")
        if Hm is not None and t.shape[1] != Hm:
            raise FlashMaskError("all mask vectors must share the same head count")
        Hm = t.shape[1]
        keep.append(t)
    return (Hm or 1), [_ptr(t) for t in keep], keep


def make_problem(B, H, Hm, N, d, dv, scale, causal) -> _b.fm_problem:
    return _b.fm_problem(B, H, Hm, N, d, dv, float(scale if scale is not None else 0.0),
                         int(bool(causal)))


def make_options(deterministic=False, wait_timeout_ns=0, kernel_events=None, sink=None,
                 dsink=None, reuse_tile_map=False, debug_bounds=False,
                 accumulate_f32=False, debug_drop_load=0) -> _b.fm_options:
    """kernel_events: optional list of raw cudaEvent_t handles (ints), recorded in
    pairs around each kernel launch of the call.  sink / dsink: optional [H]
    fp32 CUDA tensors, the attention-sink logits and (backward) their gradient.
    reuse_tile_map: the workspace already holds this problem's tile map and
    lists from an earlier call on it (see flashmask.h).  debug_bounds: every
    attention CTA checks its work list first; a bad one makes get_error()
    raise (status FM_ERR_DEVICE_BOUNDS) instead of reading out of range.
    accumulate_f32: the backward adds its gradients to fp32 dq, dk, dv instead
    of writing bf16.  debug_drop_load: failure-detection tests only (see
    flashmask.h): the forward skips one key-tile load so its waits run out."""
    opt = _b.fm_options(int(bool(deterministic)), int(bool(debug_bounds)), int(wait_timeout_ns),
                        None, 0,
                        None if sink is None else sink.data_ptr(),
                        None if dsink is None else dsink.data_ptr(), int(bool(reuse_tile_map)),
                        int(bool(accumulate_f32)), int(debug_drop_load))
    opt._tensors = (sink, dsink)
    if kernel_events:
        arr = (ctypes.c_void_p * len(kernel_events))(*kernel_events)
        opt.kernel_events = ctypes.cast(arr, ctypes.POINTER(ctypes.c_void_p))
        opt.n_kernel_events = len(kernel_events)
        opt._keep = arr
    return opt


def _check_qkv(q, k, v):
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous() or t.dim() != 4:
            raise FlashMaskError(f"{name} must be a contiguous 4-D bf16 CUDA tensor [B,N,H,dim]")
    B, N, H, d = q.shape
    if k.shape != (B, N, H, d) or v.shape[:3] != (B, N, H):
        raise FlashMaskError("q, k, v shapes disagree")
    if not (_same_device(k.device, q.device) and _same_device(v.device, q.device)):
        raise FlashMaskError("q, k, v must be on one device")
    return B, N, H, d, v.shape[3]


def workspace_size(B, H, Hm, N, d, dv, is_bwd: bool, deterministic=False) -> int:
    prob = make_problem(B, H, Hm, N, d, dv, None, False)
    n = _b.flashmask_workspace_size(prob, make_options(deterministic), int(is_bwd))
    if n == 0:
        raise FlashMaskError("invalid problem for workspace query")
    return n


def _check_out(name, t, shape, dtype, device):
    """A caller-supplied output: the kernels write every element of `shape`
    through its data pointer, so anything else would write out of bounds."""
    if (t.dtype != dtype or tuple(t.shape) != tuple(shape) or not t.is_contiguous()
            or not _same_device(t.device, device)):
        raise FlashMaskError(f"{name} must be a contiguous {dtype} tensor of shape "
                             f"{tuple(shape)} on {device}")


def _check_workspace(ws, device):
    if ws.dtype != torch.uint8 or ws.dim() != 1 or not ws.is_contiguous() or \
            not _same_device(ws.device, device):
        raise FlashMaskError(f"workspace must be a contiguous 1-D uint8 tensor on {device}")


def _check_sink(sink, H, device):
    if sink is not None and (sink.dtype != torch.float32 or tuple(sink.shape) != (H,) or
                             not sink.is_contiguous() or not _same_device(sink.device, device)):
        raise FlashMaskError(f"sink must be a contiguous float32 tensor of shape ({H},) on "
                             f"{device}")


def fwd(q, k, v, lts=None, lte=None, uts=None, ute=None, causal=False, scale=None,
        out=None, lse=None, workspace=None, stream=None, options=None, sink=None,
        reuse_tile_map=False):
    """Masked attention forward; returns (o [B,N,H,dv] bf16, lse [B,H,N] fp32).
    sink: optional [H] fp32 attention-sink logits (see flashmask.h).
    reuse_tile_map: `workspace` already holds this problem's tile map and lists."""
    B, N, H, d, dv = _check_qkv(q, k, v)
    Hm, mp, _keep = _mask_args((lts, lte, uts, ute), B, H, N, q.device)
    prob = make_problem(B, H, Hm, N, d, dv, scale, causal)
    _check_sink(sink, H, q.device)
    if options is not None and sink is not None:
        raise FlashMaskError("pass the sink either in options or as sink=, not both")
    if reuse_tile_map and workspace is None:
        raise FlashMaskError("reuse_tile_map needs the workspace that holds the tile map")
    opt = make_options(sink=sink, reuse_tile_map=reuse_tile_map) if options is None else options
    if out is None:
        out = torch.empty((B, N, H, dv), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    _check_out("out", out, (B, N, H, dv), torch.bfloat16, q.device)
    _check_out("lse", lse, (B, H, N), torch.float32, q.device)
    ws_bytes = _b.flashmask_workspace_size(prob, opt, 0)
    if workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
    _check_workspace(workspace, q.device)
    with _Range(f"flashmask_fwd B={B} H={H} N={N} d={d} dv={dv}" if _nvtx else ""):
        st = _b.flashmask_fwd(prob, opt, q.data_ptr(), k.data_ptr(), v.data_ptr(), *mp,
                              out.data_ptr(), lse.data_ptr(), workspace.data_ptr(),
                              workspace.numel(), _stream(stream))
    _check(st, "flashmask_fwd")
    return out, lse


def bwd(q, k, v, o, lse, dout, lts=None, lte=None, uts=None, ute=None, causal=False,
        scale=None, deterministic=False, dq=None, dk=None, dv=None, workspace=None,
        stream=None, options=None, sink=None, reuse_tile_map=False, accumulate_f32=False):
    """Masked attention backward; returns (dq, dk, dv) in bf16, and with a sink
    (the forward's [H] fp32 logits) also their gradient: (dq, dk, dv, dsink).
    reuse_tile_map: `workspace` (sized for the backward) already holds this
    problem's tile map and lists, e.g. from the forward call on it.
    accumulate_f32: dq, dk, dv are given as fp32 tensors and the gradients
    are added to them (no bf16 rounding)."""
    B, N, H, d, dvd = _check_qkv(q, k, v)
    _check_sink(sink, H, q.device)
    if options is not None and sink is not None:
        raise FlashMaskError("pass the sink either in options or as sink=, not both")
    for name, t, shape in (("o", o, (B, N, H, dvd)), ("dout", dout, (B, N, H, dvd))):
        if t.dtype != torch.bfloat16 or not t.is_contiguous() or tuple(t.shape) != shape or \
                not _same_device(t.device, q.device):
            raise FlashMaskError(f"{name} must be contiguous bf16 {shape} on {q.device}")
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, N) or \
            not lse.is_contiguous() or not _same_device(lse.device, q.device):
        raise FlashMaskError(f"lse must be contiguous fp32 [B, H, N] on {q.device}")
    Hm, mp, _keep = _mask_args((lts, lte, uts, ute), B, H, N, q.device)
    prob = make_problem(B, H, Hm, N, d, dvd, scale, causal)
    dsink = None if sink is None else torch.empty(H, dtype=torch.float32, device=q.device)
    if reuse_tile_map and workspace is None:
        raise FlashMaskError("reuse_tile_map needs the workspace that holds the tile map")
    if options is not None and accumulate_f32:
        raise FlashMaskError("pass accumulate_f32 either in options or as an argument")
    opt = make_options(deterministic, sink=sink, dsink=dsink, reuse_tile_map=reuse_tile_map,
                       accumulate_f32=accumulate_f32) if options is None else options
    acc32 = bool(opt.accumulate_f32)
    if acc32 and (dq is None or dk is None or dv is None):
        raise FlashMaskError("accumulate_f32 adds to the caller's fp32 dq, dk and dv")
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    gdt = torch.float32 if acc32 else torch.bfloat16
    _check_out("dq", dq, (B, N, H, d), gdt, q.device)
    _check_out("dk", dk, (B, N, H, d), gdt, q.device)
    _check_out("dv", dv, (B, N, H, dvd), gdt, q.device)
    ws_bytes = _b.flashmask_workspace_size(prob, opt, 1)
    if workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
    _check_workspace(workspace, q.device)
    with _Range(f"flashmask_bwd B={B} H={H} N={N} d={d} dv={dvd}" if _nvtx else ""):
        st = _b.flashmask_bwd(prob, opt, q.data_ptr(), k.data_ptr(), v.data_ptr(),
                              o.data_ptr(), lse.data_ptr(), dout.data_ptr(), *mp,
                              dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                              workspace.data_ptr(), workspace.numel(), _stream(stream))
    _check(st, "flashmask_bwd")
    return (dq, dk, dv) if sink is None else (dq, dk, dv, dsink)


def classify(N, B=1, H=1, lts=None, lte=None, uts=None, ute=None, causal=False, device="cuda",
             stream=None):
    """Tile map [B*Hm, T, T] uint8 (0 skip, 1 partial, 2 unmasked) of 128x128 tiles."""
    device = torch.device(device)
    Hm, mp, _keep = _mask_args((lts, lte, uts, ute), B, H, N, device)
    prob = make_problem(B, H, Hm, N, 128, 128, None, causal)
    T = -(-N // 128)
    out = torch.empty((B * Hm, T, T), dtype=torch.uint8, device=device)
    ws_bytes = _b.flashmask_workspace_size(prob, None, 0)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=device)
    st = _b.flashmask_classify(prob, *mp, out.data_ptr(), ws.data_ptr(), ws.numel(),
                               _stream(stream))
    _check(st, "flashmask_classify")
    return out


def count_unmasked(N, B=1, H=1, lts=None, lte=None, uts=None, ute=None, causal=False,
                   device="cuda", stream=None):
    """Unmasked (i, j) pairs per mask head: int64 tensor [B*Hm] on the device."""
    device = torch.device(device)
    Hm, mp, _keep = _mask_args((lts, lte, uts, ute), B, H, N, device)
    prob = make_problem(B, H, Hm, N, 128, 128, None, causal)
    out = torch.empty((B * Hm,), dtype=torch.int64, device=device)
    st = _b.flashmask_count_unmasked(prob, *mp, out.data_ptr(), _stream(stream))
    _check(st, "flashmask_count_unmasked")
    return out


def get_error(stream=None):
    """Synchronise the stream and raise if a kernel gave up on a bounded wait or
    (debug_bounds) found its work list out of range."""
    _check(_b.flashmask_get_error(_stream(stream)), "device")


def selftest_wait(timeout_ns=20_000_000, stream=None):
    """Failure-detection self-test: a device wait that nothing completes gives
    up after `timeout_ns`; the next get_error() raises with status
    FM_ERR_DEVICE_TIMEOUT, and the context stays usable."""
    _check(_b.flashmask_selftest_wait(timeout_ns, _stream(stream)), "flashmask_selftest_wait")


class FlashMaskAttention(torch.autograd.Function):
    """Autograd wrapper: forward and backward both run in the CUDA library."""

    @staticmethod
    def forward(ctx, q, k, v, lts, lte, uts, ute, causal, scale, deterministic, sink):
        o, lse = fwd(q, k, v, lts, lte, uts, ute, causal, scale, sink=sink)
        ctx.save_for_backward(q, k, v, o, lse, lts, lte, uts, ute, sink)
        ctx.causal, ctx.scale, ctx.deterministic = causal, scale, deterministic
        return o

    @staticmethod
    def backward(ctx, do):
        q, k, v, o, lse, lts, lte, uts, ute, sink = ctx.saved_tensors
        g = bwd(q, k, v, o, lse, do.contiguous(), lts, lte, uts, ute, ctx.causal, ctx.scale,
                ctx.deterministic, sink=sink)
        dsink = g[3] if sink is not None else None
        return g[0], g[1], g[2], None, None, None, None, None, None, None, dsink


def flashmask_attention(q, k, v, lts=None, lte=None, uts=None, ute=None, causal=False,
                        scale=None, deterministic=False, sink=None):
    """O = softmax(Q K^T * scale + M) V with the column-wise mask; differentiable.
    sink: optional [H] fp32 attention-sink logits (differentiable as well)."""
    return FlashMaskAttention.apply(q, k, v, lts, lte, uts, ute, causal, scale, deterministic,
                                    sink)


def default_scale(d: int) -> float:
    return 1.0 / math.sqrt(d)


# --------------------------------------------------- context-parallel chunks
def zigzag_assignment(chunks: int, ranks: int) -> list:
    """Query chunks per rank of the usual causal load-balancing assignment:
    with 2R chunks, rank r owns chunks r and 2R - 1 - r."""
    if chunks != 2 * ranks:
        raise FlashMaskError("the zigzag assignment needs chunks == 2 * ranks")
    return [[r, chunks - 1 - r] for r in range(ranks)]


def localize(lts, lte, uts, ute, B, H, N, causal, q0, k0, length, stream=None):
    """Boundary vectors of the local problem of the pair (query chunk at q0, key
    chunk at k0) of chunks of `length` (clip to the query chunk, shift by its
    start, max with 0).  Returns ([lts, lte, uts, ute] as [B, Hm, length] int32
    tensors, local causal flag), or (None, -1) when every element of the pair is
    masked."""
    device = next(t.device for t in (lts, lte, uts, ute) if t is not None) \
        if any(t is not None for t in (lts, lte, uts, ute)) else torch.device("cuda")
    Hm, mp, _keep = _mask_args((lts, lte, uts, ute), B, H, N, device)
    prob = make_problem(B, H, Hm, N, 64, 64, None, causal)
    out = [torch.empty((B, Hm, length), dtype=torch.int32, device=device) for _ in range(4)]
    st, flag = _b.flashmask_localize(prob, *mp, int(q0), int(k0), int(length),
                                     *(t.data_ptr() for t in out), _stream(stream))
    _check(st, "flashmask_localize")
    return (None, -1) if flag < 0 else (out, flag)


def _chunk_plan(N, chunks, ranks):
    if chunks < 1 or N % chunks != 0:
        raise FlashMaskError("chunks must divide N")
    L = N // chunks
    owned = zigzag_assignment(chunks, ranks) if ranks else [[c] for c in range(chunks)]
    return L, owned


def fwd_chunked(q, k, v, lts=None, lte=None, uts=None, ute=None, causal=False, scale=None,
                chunks=2, ranks=None, stream=None):
    """The forward of the whole sequence as a context-parallel run emulated on
    this GPU: the sequence is cut into `chunks` equal chunks; each rank (the
    zigzag assignment when `ranks` is given, one chunk per rank otherwise)
    takes its query chunks against every key chunk, each pair a local problem
    with localized vectors, and merges the pairs of a query chunk by
    log-sum-exp.  Returns (o [B,N,H,dv] bf16, lse [B,H,N] fp32), equal to fwd()
    up to rounding."""
    B, N, H, d, dv = _check_qkv(q, k, v)
    L, owned = _chunk_plan(N, chunks, ranks)
    dev = q.device
    s = _stream(stream)
    o = torch.empty((B, N, H, dv), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    o_part = torch.empty((1, L, H, dv), dtype=torch.bfloat16, device=dev)
    lse_part = torch.empty((1, H, L), dtype=torch.float32, device=dev)
    o_acc = torch.empty((L, H, dv), dtype=torch.float32, device=dev)
    lse_acc = torch.empty((H, L), dtype=torch.float32, device=dev)
    vecs = (lts, lte, uts, ute)
    ws = None
    for b in range(B):
        vb = [None if t is None else t[b:b + 1] for t in vecs]
        for rank_chunks in owned:
            for qc in rank_chunks:
                q0 = qc * L
                _check(_b.flashmask_merge_init(L, H, dv, o_acc.data_ptr(), lse_acc.data_ptr(),
                                               s), "flashmask_merge_init")
                for kc in range(chunks):
                    k0 = kc * L
                    local, lc = localize(*vb, 1, H, N, causal, q0, k0, L, stream)
                    if local is None:
                        continue
                    if ws is None:
                        Hm = local[0].shape[1]
                        ws = torch.empty(workspace_size(1, H, Hm, L, d, dv, False),
                                         dtype=torch.uint8, device=dev)
                    fwd(q[b:b + 1, q0:q0 + L], k[b:b + 1, k0:k0 + L], v[b:b + 1, k0:k0 + L],
                        *local, causal=bool(lc), scale=scale if scale is not None
                        else default_scale(d), out=o_part, lse=lse_part, workspace=ws,
                        stream=stream)
                    _check(_b.flashmask_merge(L, H, dv, o_part.data_ptr(), lse_part.data_ptr(),
                                              o_acc.data_ptr(), lse_acc.data_ptr(), s),
                           "flashmask_merge")
                lse_out = lse.data_ptr() + (b * H * N + q0) * 4
                _check(_b.flashmask_merge_finish(L, H, dv, o_acc.data_ptr(), lse_acc.data_ptr(),
                                                 o[b:b + 1, q0:q0 + L].data_ptr(), lse_out, N, s),
                       "flashmask_merge_finish")
    return o, lse


def bwd_chunked(q, k, v, o, lse, dout, lts=None, lte=None, uts=None, ute=None, causal=False,
                scale=None, deterministic=False, chunks=2, ranks=None, stream=None):
    """The backward as the same emulated context-parallel run: every pair's
    local backward (with the whole sequence's O and LSE rows of its query
    chunk) adds its partial dQ for the query chunk and partial dK, dV for the
    key chunk, in fp32, straight into the whole sequence's accumulators
    (fm_options.accumulate_f32); they are rounded to bf16 once."""
    B, N, H, d, dvd = _check_qkv(q, k, v)
    L, owned = _chunk_plan(N, chunks, ranks)
    dev = q.device
    s = _stream(stream)
    acc = [torch.zeros((B, N, H, c), dtype=torch.float32, device=dev) for c in (d, d, dvd)]
    vecs = (lts, lte, uts, ute)
    ws = None
    for b in range(B):
        vb = [None if t is None else t[b:b + 1] for t in vecs]
        for rank_chunks in owned:
            for qc in rank_chunks:
                q0 = qc * L
                lse_c = lse[b:b + 1, :, q0:q0 + L].contiguous()
                for kc in range(chunks):
                    k0 = kc * L
                    local, lc = localize(*vb, 1, H, N, causal, q0, k0, L, stream)
                    if local is None:
                        continue
                    if ws is None:
                        Hm = local[0].shape[1]
                        ws = torch.empty(workspace_size(1, H, Hm, L, d, dvd, True, deterministic),
                                         dtype=torch.uint8, device=dev)
                    bwd(q[b:b + 1, q0:q0 + L], k[b:b + 1, k0:k0 + L], v[b:b + 1, k0:k0 + L],
                        o[b:b + 1, q0:q0 + L], lse_c, dout[b:b + 1, q0:q0 + L], *local,
                        causal=bool(lc), scale=scale if scale is not None else default_scale(d),
                        deterministic=deterministic, dq=acc[0][b:b + 1, q0:q0 + L],
                        dk=acc[1][b:b + 1, k0:k0 + L], dv=acc[2][b:b + 1, k0:k0 + L],
                        workspace=ws, stream=stream, accumulate_f32=True)
    outs = [torch.empty((B, N, H, c), dtype=torch.bfloat16, device=dev) for c in (d, d, dvd)]
    for a, out in zip(acc, outs):
        _check(_b.flashmask_to_bf16(a.numel(), a.data_ptr(), out.data_ptr(), s),
               "flashmask_to_bf16")
    return tuple(outs)
