"""Attention-sink logits on the GPU, through the C ABI, against the fp64 oracle.

The oracle's sink (a value-free term exp(sink) of every row's softmax
denominator) is pinned on the CPU against an extra zero-value key column.
Here the CUDA path must match it: O, LSE and dQ / dK / dV within the usual
tolerances, and the sink logits' gradient within a bound derived from its
terms.
"""
import numpy as np
import pytest
import torch

import oracle
from sparse_masked_attention_gb300 import attention as fm
from sparse_masked_attention_gb300 import workloads as W

from gpu_util import assert_close, assert_lse, cuda_mask, head, mask_slice

pytestmark = pytest.mark.gpu


def _check(q, k, v, do, mask, sink, o, lse, grads):
    B, N, H, d = q.shape
    scale = 1 / np.sqrt(d)
    dsink_ref = np.zeros(H)
    dsink_abs = np.zeros(H)  # sum of the terms' magnitudes
    for b in range(B):
        for h in range(H):
            qh, kh, vh, doh = head(q, b, h), head(k, b, h), head(v, b, h), head(do, b, h)
            ms = mask_slice(mask, b, h)
            s = float(sink[h])
            ro, rl = oracle.attention_fwd(qh, kh, vh, ms, mask.causal, scale, sink=s)
            assert_close("O", head(o, b, h), ro)
            assert_lse(lse[b, h].cpu().numpy(), rl)
            if grads is None:
                continue
            rdq, _, terms = oracle.attention_bwd_dq(qh, kh, vh, doh, ms, mask.causal, scale,
                                                    sink=s, with_dsink=True)
            rdk, rdv = oracle.attention_bwd_dkdv(qh, kh, vh, doh, ms, mask.causal, scale, sink=s)
            assert_close("dQ", head(grads[0], b, h), rdq)
            assert_close("dK", head(grads[1], b, h), rdk)
            assert_close("dV", head(grads[2], b, h), rdv)
            dsink_ref[h] += terms.sum()
            dsink_abs[h] += np.abs(terms).sum()
    if grads is not None:
        got = grads[3].cpu().numpy().astype(np.float64)
        # Each term -P_sink,i D_i comes from the fp32 LSE (|err| <= 1e-3, so
        # P_sink to 1e-3 relative) and D_i from the bf16 O (2^-9 relative per
        # element): 1e-2 of the terms' magnitudes bounds the sum's error.
        assert np.all(np.abs(got - dsink_ref) <= 1e-2 * dsink_abs + 1e-4), (got, dsink_ref)


@pytest.mark.parametrize("d,dv", [(64, 64), (128, 128), (192, 128), (256, 256)])
def test_sink_parity(d, dv):
    B, H, N = 2, 2, 1000
    rng = np.random.default_rng(31)
    q, k, v, do = W.make_inputs(B, N, H, d, dv, seed=5, device="cuda")
    mask = W.causal_document(N, [W.uniform_lengths(rng, 50, 300, N) for _ in range(B)])
    vec = cuda_mask(mask)
    sink = torch.tensor([0.75, -1.5], dtype=torch.float32, device="cuda")
    o, lse = fm.fwd(q, k, v, *vec, causal=mask.causal, sink=sink)
    grads = fm.bwd(q, k, v, o, lse, do, *vec, causal=mask.causal, sink=sink)
    fm.get_error()
    _check(q, k, v, do, mask, sink.cpu().numpy(), o, lse, grads)


def test_sink_fully_masked_rows_and_dominating_sink():
    """Rows [130, 260) see no key: O = 0 and LSE = sink.  A sink above every
    row's largest score (8 against scores of unit variance) takes the other
    normalisation branch; far larger sinks push the gradients below bf16
    resolution, where the relative-L2 criterion says nothing."""
    B, H, N, d = 1, 2, 400, 128
    q, k, v, do = W.make_inputs(B, N, H, d, d, seed=6, device="cuda")
    lts = np.full((1, 1, N), 130, np.int32)
    lte = np.full((1, 1, N), 260, np.int32)
    mask = W.Mask(N, False, lts=lts, lte=lte, family="custom", meta=[{}])
    vec = cuda_mask(mask)
    sink = torch.tensor([1.25, 8.0], dtype=torch.float32, device="cuda")
    o, lse = fm.fwd(q, k, v, *vec, causal=False, sink=sink)
    grads = fm.bwd(q, k, v, o, lse, do, *vec, causal=False, sink=sink)
    fm.get_error()
    assert bool((o[0, 130:260] == 0).all())
    assert torch.allclose(lse[0, 0, 130:260], torch.full((130,), 1.25, device="cuda"))
    _check(q, k, v, do, mask, sink.cpu().numpy(), o, lse, grads)


def test_sink_gradient_deterministic_and_autograd():
    B, H, N, d = 2, 3, 700, 64
    rng = np.random.default_rng(8)
    q, k, v, do = W.make_inputs(B, N, H, d, d, seed=7, device="cuda")
    mask = W.share_question(N, [W.share_question_groups(rng, N, (100, 200), (2, 3), (40, 120))
                                for _ in range(B)])
    vec = cuda_mask(mask)
    sink = torch.tensor([0.0, 1.0, -2.0], dtype=torch.float32, device="cuda")
    o, lse = fm.fwd(q, k, v, *vec, causal=True, sink=sink)
    g1 = fm.bwd(q, k, v, o, lse, do, *vec, causal=True, deterministic=True, sink=sink)
    g2 = fm.bwd(q, k, v, o, lse, do, *vec, causal=True, deterministic=True, sink=sink)
    for a, b_ in zip(g1, g2):
        assert torch.equal(a, b_)
    qq, kk, vv = (x.clone().requires_grad_(True) for x in (q, k, v))
    ss = sink.clone().requires_grad_(True)
    out = fm.flashmask_attention(qq, kk, vv, *vec, causal=True, deterministic=True, sink=ss)
    out.backward(do)
    fm.get_error()
    assert torch.equal(out, o)
    for a, b_ in zip((qq.grad, kk.grad, vv.grad, ss.grad), g1):
        assert torch.equal(a, b_)


def test_sink_with_per_head_masks():
    B, H, N, d = 1, 3, 500, 128
    rng = np.random.default_rng(41)
    q, k, v, do = W.make_inputs(B, N, H, d, d, seed=17, device="cuda")
    mask = W.random_vectors(N, rng, B, Hm=H, causal_flag=True, lo=0, hi=N)
    vec = cuda_mask(mask)
    sink = torch.tensor([-0.5, 0.0, 2.5], dtype=torch.float32, device="cuda")
    o, lse = fm.fwd(q, k, v, *vec, causal=True, sink=sink)
    grads = fm.bwd(q, k, v, o, lse, do, *vec, causal=True, sink=sink)
    fm.get_error()
    _check(q, k, v, do, mask, sink.cpu().numpy(), o, lse, grads)
