"""Canary bands: every output the library writes (O, LSE, dQ, dK, dV, the sink
gradient) and the workspace sit in the middle of a larger buffer whose guard
bands hold a fixed bit pattern.  After the forward and the backward every
guard must be unchanged, so no kernel writes outside the tensor it was given,
at ragged sizes (N not a multiple of the 128-row tile) and every head dim.
This stands in for a memory checker on the output side.
"""
import math

import numpy as np
import pytest
import torch

from gpu_util import cuda_mask
from sparse_masked_attention_gb300 import attention as fm
from sparse_masked_attention_gb300 import workloads as W

pytestmark = pytest.mark.gpu

GUARD_BYTES = 8192  # keeps every view 256-byte aligned (TMA and workspace rules)
PATTERN = 0x5A


class Guarded:
    """A tensor of `shape` inside a byte buffer with guard bands on both sides."""

    def __init__(self, shape, dtype, device="cuda"):
        itemsize = torch.tensor([], dtype=dtype).element_size()
        self.nbytes = math.prod(shape) * itemsize
        self.buf = torch.full((self.nbytes + 2 * GUARD_BYTES,), PATTERN, dtype=torch.uint8,
                              device=device)
        self.t = self.buf[GUARD_BYTES:GUARD_BYTES + self.nbytes].view(dtype).view(shape)

    def intact(self):
        head = self.buf[:GUARD_BYTES]
        tail = self.buf[GUARD_BYTES + self.nbytes:]
        return bool((head == PATTERN).all()) and bool((tail == PATTERN).all())


def _mask(name, N, B):
    rng = np.random.default_rng(N)
    if name == "causal_document":
        return W.causal_document(N, [W.uniform_lengths(rng, 40, 300, N) for _ in range(B)])
    if name == "full":
        return W.full(N, B)
    return W.share_question(
        N, [W.share_question_groups(rng, N, (60, 200), (2, 3), (30, 120)) for _ in range(B)])


@pytest.mark.parametrize("d,dv", [(64, 64), (128, 128), (192, 128), (256, 256)])
@pytest.mark.parametrize("N", [130, 1000])
@pytest.mark.parametrize("family", ["causal_document", "full", "share_question"])
def test_outputs_and_workspace_stay_in_bounds(d, dv, N, family):
    B, H = 2, 2
    q, k, v, do = W.make_inputs(B, N, H, d, dv, seed=N + d, device="cuda")
    mask = _mask(family, N, B)
    vec = cuda_mask(mask)
    o = Guarded((B, N, H, dv), torch.bfloat16)
    lse = Guarded((B, H, N), torch.float32)
    dq = Guarded((B, N, H, d), torch.bfloat16)
    dk = Guarded((B, N, H, d), torch.bfloat16)
    dvv = Guarded((B, N, H, dv), torch.bfloat16)
    ws = Guarded((fm.workspace_size(B, H, 1, N, d, dv, True),), torch.uint8)
    fm.fwd(q, k, v, *vec, causal=mask.causal, out=o.t, lse=lse.t, workspace=ws.t)
    fm.bwd(q, k, v, o.t, lse.t, do, *vec, causal=mask.causal, deterministic=True, dq=dq.t,
           dk=dk.t, dv=dvv.t, workspace=ws.t, reuse_tile_map=True)
    fm.get_error()
    for name, g in (("O", o), ("LSE", lse), ("dQ", dq), ("dK", dk), ("dV", dvv),
                    ("workspace", ws)):
        assert g.intact(), f"{name}: a guard band was overwritten"
    # ...and every element inside was written: the same as with the library's
    # own allocations (the guard pattern is a finite value no output takes)
    ro, rl = fm.fwd(q, k, v, *vec, causal=mask.causal)
    rg = fm.bwd(q, k, v, ro, rl, do, *vec, causal=mask.causal, deterministic=True)
    fm.get_error()
    assert torch.equal(o.t, ro) and torch.equal(lse.t, rl)
    for got, ref in zip((dq.t, dk.t, dvv.t), rg):
        assert torch.equal(got, ref)


def test_sink_gradient_stays_in_bounds():
    B, H, N, d = 1, 3, 1000, 128
    q, k, v, do = W.make_inputs(B, N, H, d, d, seed=3, device="cuda")
    mask = _mask("causal_document", N, B)
    vec = cuda_mask(mask)
    sink = torch.tensor([0.5, -1.0, 2.0], dtype=torch.float32, device="cuda")
    o, lse = fm.fwd(q, k, v, *vec, causal=mask.causal, sink=sink)
    dsink = Guarded((H,), torch.float32)
    fm.bwd(q, k, v, o, lse, do, *vec, causal=mask.causal,
           options=fm.make_options(True, sink=sink, dsink=dsink.t))
    ref = fm.bwd(q, k, v, o, lse, do, *vec, causal=mask.causal, deterministic=True, sink=sink)
    fm.get_error()
    assert dsink.intact()
    assert torch.equal(dsink.t, ref[3])


def test_wrong_outputs_are_refused_before_launch():
    B, H, N, d = 1, 2, 300, 128
    q, k, v, do = W.make_inputs(B, N, H, d, d, seed=4, device="cuda")
    o, lse = fm.fwd(q, k, v, causal=True)
    bad = [dict(out=torch.empty((B, N - 1, H, d), dtype=torch.bfloat16, device="cuda")),
           dict(out=torch.empty((B, N, H, d), dtype=torch.float16, device="cuda")),
           dict(lse=torch.empty((B, H, N + 1), dtype=torch.float32, device="cuda")),
           dict(out=torch.empty((B, N, H, 2 * d), dtype=torch.bfloat16, device="cuda")[..., :d]),
           dict(workspace=torch.empty(1 << 20, dtype=torch.int32, device="cuda"))]
    for kw in bad:
        with pytest.raises(fm.FlashMaskError):
            fm.fwd(q, k, v, causal=True, **kw)
    for kw in (dict(dq=torch.empty((B, N, H, d - 64), dtype=torch.bfloat16, device="cuda")),
               dict(dk=torch.empty((B, N + 7, H, d), dtype=torch.bfloat16, device="cuda")),
               dict(dv=torch.empty((B, N, H, d), dtype=torch.float32, device="cuda"))):
        with pytest.raises(fm.FlashMaskError):
            fm.bwd(q, k, v, o, lse, do, causal=True, **kw)
    fm.get_error()
