"""The backward over the whole bf16 input range, against the fp64 oracle.

The backward's dP and dV products run in fp16 on copies of dO and V scaled by
a power of two per (batch, head), so that gradients far below fp16's smallest
normal (1e-9 and less, as unscaled losses in bf16 training give) and values
far above its largest (1e5) keep fp16's precision.

The method is homogeneous of degree one in dO (every gradient scales with it)
and in V (O, dQ and dK scale with it; P, hence dV, does not).  A scaled case
is therefore held to the same bar as an N(0, 1) case after dividing by the
scale: max-abs tolerance times the factor, relative L2 unchanged.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from sparse_masked_attention_gb300 import attention as fm
from sparse_masked_attention_gb300 import workloads as W

from gpu_util import MAX_ABS, REL_L2, assert_close, assert_lse, cuda_mask, head, mask_slice

pytestmark = pytest.mark.gpu

DIMS = [(64, 64), (128, 128), (192, 128), (256, 256)]

# (name, per-head factor on dO, per-head factor on V); two heads.
CASES = [
    ("dO x 1e-6", (1e-6, 1e-6), (1.0, 1.0)),
    ("dO x 1e-9", (1e-9, 1e-9), (1.0, 1.0)),
    ("V x 1e5", (1.0, 1.0), (1e5, 1e5)),
    ("dO x 1e-6 and V x 1e5", (1e-6, 1e-6), (1e5, 1e5)),
    ("heads apart: dO x 1e-9 | x 1e3", (1e-9, 1e3), (1.0, 1.0)),
]


def _scaled(t, factors):
    """bf16 tensor [B, N, H, c] with head h multiplied by factors[h] (in fp32,
    then rounded to bf16: the oracle reads the rounded values)."""
    f = torch.tensor(factors, dtype=torch.float32, device=t.device).view(1, 1, -1, 1)
    return (t.float() * f).to(torch.bfloat16).contiguous()


@pytest.mark.parametrize("d,dv", DIMS)
@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_backward_over_the_bf16_range(d, dv, case):
    name, f_do, f_v = case
    N, H = 1000, 2
    rng = np.random.default_rng(3)
    mask = W.causal_document(N, [W.uniform_lengths(rng, 60, 400, N)])
    q, k, v, do = W.make_inputs(1, N, H, d, dv, seed=40, device="cuda")
    v, do = _scaled(v, f_v), _scaled(do, f_do)
    vec = cuda_mask(mask)
    o, lse = fm.fwd(q, k, v, *vec, causal=mask.causal)
    dq, dk, dvv = fm.bwd(q, k, v, o, lse, do, *vec, causal=mask.causal)
    fm.get_error()
    scale = 1 / math.sqrt(d)
    for h in range(H):
        qh, kh, vh, doh = head(q, 0, h), head(k, 0, h), head(v, 0, h), head(do, 0, h)
        ms = mask_slice(mask, 0, h)
        ro, rl = oracle.attention_fwd(qh, kh, vh, ms, mask.causal, scale)
        rdq, rdk, rdv = oracle.attention_bwd(qh, kh, vh, doh, ms, mask.causal, scale)
        fo, fg = f_v[h], f_do[h] * f_v[h]  # factors of O and of dQ, dK
        assert_close(f"{name} h{h} O", head(o, 0, h), ro, MAX_ABS * fo, REL_L2)
        assert_lse(lse[0, h].cpu().numpy(), rl)
        assert_close(f"{name} h{h} dQ", head(dq, 0, h), rdq, MAX_ABS * fg, REL_L2)
        assert_close(f"{name} h{h} dK", head(dk, 0, h), rdk, MAX_ABS * fg, REL_L2)
        assert_close(f"{name} h{h} dV", head(dvv, 0, h), rdv, MAX_ABS * f_do[h], REL_L2)
        for t in (dq, dk, dvv):
            assert torch.isfinite(t[0, :, h].float()).all(), f"{name}: non-finite gradient"


def test_scaling_changes_no_bit_of_unit_range_results():
    """Powers of two change no rounding: for N(0, 1) inputs the gradients are
    the same as with dO and V both multiplied by 2^20 and the results divided
    by it (every product of the path sees the same mantissas)."""
    N, H, d = 640, 2, 128
    mask = W.causal(N, 1)
    q, k, v, do = W.make_inputs(1, N, H, d, d, seed=41, device="cuda")
    vec = cuda_mask(mask)
    o, lse = fm.fwd(q, k, v, *vec, causal=True)
    g1 = fm.bwd(q, k, v, o, lse, do, *vec, causal=True, deterministic=True)
    s = 2.0 ** 20
    do2 = (do.float() * s).to(torch.bfloat16)
    g2 = fm.bwd(q, k, v, o, lse, do2, *vec, causal=True, deterministic=True)
    fm.get_error()
    for a, b in zip(g1, g2):
        assert torch.equal(a.float() * s, b.float())
