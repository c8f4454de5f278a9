"""Context-parallel chunks on one GPU, through the C ABI.

- flashmask_localize writes, bit for bit, the local vectors the oracle's
  localization gives (clip to the query chunk, shift, max with 0), and flags
  the pairs a causal mask masks entirely.
- The forward and backward of the whole sequence, run as the emulated
  context-parallel job (each rank's query chunks against every key chunk,
  log-sum-exp merge, partial gradients added in fp32 by the backward itself
  and rounded to bf16 once), match the fp64 oracle element by element at the
  single-call tolerance.
- flashmask_bwd with accumulate_f32 adds exactly its gradients to fp32
  arrays that already hold values.
"""
import numpy as np
import pytest
import torch

import oracle
from sparse_masked_attention_gb300 import attention as fm
from sparse_masked_attention_gb300 import workloads as W

from gpu_util import assert_close, assert_lse, cuda_mask, head, mask_slice

pytestmark = pytest.mark.gpu


def _family(name, N, B, rng, Hm=1):
    if name == "causal":
        return W.causal(N, B)
    if name == "causal_document":
        return W.causal_document(N, [W.uniform_lengths(rng, 60, 400, N) for _ in range(B)])
    if name == "document":
        return W.document(N, [W.uniform_lengths(rng, 60, 400, N) for _ in range(B)])
    if name == "share_question":
        return W.share_question(
            N, [W.share_question_groups(rng, N, (100, 300), (2, 4), (50, 200)) for _ in range(B)])
    if name == "block_sparse":
        return W.block_sparse(N, rng, B)
    if name == "random_causal":
        return W.random_vectors(N, rng, B, Hm, causal_flag=True)
    if name == "random":
        return W.random_vectors(N, rng, B, Hm, causal_flag=False)
    raise ValueError(name)


@pytest.mark.parametrize("family", ["causal_document", "share_question", "block_sparse",
                                    "random_causal", "random"])
@pytest.mark.parametrize("chunks", [2, 4])
def test_localize_matches_oracle(family, chunks):
    B, H, N = 2, 3, 1024
    rng = np.random.default_rng(chunks)
    Hm = H if family.startswith("random") else 1
    mask = _family(family, N, B, rng, Hm)
    vec = cuda_mask(mask)
    L = N // chunks
    for qc in range(chunks):
        for kc in range(chunks):
            local, flag = fm.localize(*vec, B, H, N, mask.causal, qc * L, kc * L, L)
            for b in range(B):
                for hm in range(Hm):
                    want, wc = oracle.localize(mask.slice(b, hm), N, mask.causal, qc * L,
                                               kc * L, L)
                    if want is None:
                        assert local is None and flag == -1
                        continue
                    assert flag == int(wc)
                    for i, name in enumerate(("lts", "lte", "uts", "ute")):
                        np.testing.assert_array_equal(local[i][b, hm].cpu().numpy(), want[name])
    torch.cuda.synchronize()


@pytest.mark.parametrize("family", ["causal", "causal_document", "document", "share_question",
                                    "block_sparse", "random_causal"])
@pytest.mark.parametrize("d", [64, 128])
def test_chunked_fwd_bwd_parity(family, d):
    B, H, N, C, R = 2, 2, 1024, 4, 2
    rng = np.random.default_rng(11)
    q, k, v, do = W.make_inputs(B, N, H, d, d, seed=3, device="cuda")
    mask = _family(family, N, B, rng)
    vec = cuda_mask(mask)
    o, lse = fm.fwd_chunked(q, k, v, *vec, causal=mask.causal, chunks=C, ranks=R)
    grads = fm.bwd_chunked(q, k, v, o, lse, do, *vec, causal=mask.causal, chunks=C, ranks=R)
    fm.get_error()
    scale = 1 / np.sqrt(d)
    for b in range(B):
        for h in range(H):
            qh, kh, vh, doh = head(q, b, h), head(k, b, h), head(v, b, h), head(do, b, h)
            ms = mask_slice(mask, b, h)
            ro, rl = oracle.attention_fwd(qh, kh, vh, ms, mask.causal, scale)
            assert_close("O", head(o, b, h), ro)
            assert_lse(lse[b, h].cpu().numpy(), rl)
            refs = oracle.attention_bwd(qh, kh, vh, doh, ms, mask.causal, scale)
            for name, g, ref in zip(("dQ", "dK", "dV"), grads, refs):
                # Every pair adds its partial gradient in fp32 (accumulate_f32),
                # and the sum is rounded to bf16 once: the single-call bar.
                assert_close(name, head(g, b, h), ref)


def test_chunked_equals_single_call_forward():
    """The emulated context-parallel forward and the single call agree to bf16
    rounding of O and fp32 rounding of LSE."""
    B, H, N, d = 1, 4, 2048, 128
    rng = np.random.default_rng(5)
    q, k, v, _ = W.make_inputs(B, N, H, d, d, seed=9, device="cuda", with_dout=False)
    mask = _family("share_question", N, B, rng)
    vec = cuda_mask(mask)
    o1, l1 = fm.fwd(q, k, v, *vec, causal=mask.causal)
    o2, l2 = fm.fwd_chunked(q, k, v, *vec, causal=mask.causal, chunks=8, ranks=4)
    fm.get_error()
    diff = (o1.float() - o2.float()).abs().max().item()
    assert diff <= 2.0 ** -6 * max(1.0, o1.float().abs().max().item()), diff
    fin = torch.isfinite(l1)
    assert torch.equal(torch.isneginf(l1), torch.isneginf(l2))
    assert (l1[fin] - l2[fin]).abs().max().item() <= 1e-4


def test_chunked_odd_chunk_count_one_chunk_per_rank():
    """Three chunks, no zigzag: every rank (here, loop step) owns one chunk."""
    B, H, N, d = 1, 2, 768, 64
    rng = np.random.default_rng(12)
    q, k, v, do = W.make_inputs(B, N, H, d, d, seed=4, device="cuda")
    mask = _family("share_question", N, B, rng)
    vec = cuda_mask(mask)
    o, lse = fm.fwd_chunked(q, k, v, *vec, causal=mask.causal, chunks=3)
    grads = fm.bwd_chunked(q, k, v, o, lse, do, *vec, causal=mask.causal, chunks=3)
    fm.get_error()
    scale = 1 / np.sqrt(d)
    for h in range(H):
        qh, kh, vh, doh = head(q, 0, h), head(k, 0, h), head(v, 0, h), head(do, 0, h)
        ms = mask_slice(mask, 0, h)
        ro, rl = oracle.attention_fwd(qh, kh, vh, ms, mask.causal, scale)
        assert_close("O", head(o, 0, h), ro)
        assert_lse(lse[0, h].cpu().numpy(), rl)
        for name, g, ref in zip(("dQ", "dK", "dV"), grads,
                                oracle.attention_bwd(qh, kh, vh, doh, ms, mask.causal, scale)):
            assert_close(name, head(g, 0, h), ref)


def test_chunked_ragged_chunk_length():
    """N = 1000 in 4 chunks of 250 rows: every local problem ends in a ragged
    tile, and chunk boundaries cut through tiles of the whole sequence."""
    B, H, N, d, C = 1, 2, 1000, 128, 4
    rng = np.random.default_rng(19)
    q, k, v, do = W.make_inputs(B, N, H, d, d, seed=16, device="cuda")
    mask = _family("causal_document", N, B, rng)
    vec = cuda_mask(mask)
    o, lse = fm.fwd_chunked(q, k, v, *vec, causal=mask.causal, chunks=C, ranks=C // 2)
    grads = fm.bwd_chunked(q, k, v, o, lse, do, *vec, causal=mask.causal, chunks=C, ranks=C // 2)
    fm.get_error()
    scale = 1 / np.sqrt(d)
    for h in range(H):
        qh, kh, vh, doh = head(q, 0, h), head(k, 0, h), head(v, 0, h), head(do, 0, h)
        ms = mask_slice(mask, 0, h)
        ro, rl = oracle.attention_fwd(qh, kh, vh, ms, mask.causal, scale)
        assert_close("O", head(o, 0, h), ro)
        assert_lse(lse[0, h].cpu().numpy(), rl)
        for name, g, ref in zip(("dQ", "dK", "dV"), grads,
                                oracle.attention_bwd(qh, kh, vh, doh, ms, mask.causal, scale)):
            assert_close(name, head(g, 0, h), ref)


@pytest.mark.parametrize("d,dv", [(64, 64), (128, 128), (192, 128), (256, 256)])
def test_accumulate_f32_adds_the_gradients(d, dv):
    """With accumulate_f32 the backward adds its fp32 gradients to what the
    arrays hold: starting from a known fill, the result minus the fill is the
    gradient (oracle bar), and it rounds to the bf16 call's output within one
    bf16 rounding."""
    N, H = 700, 2
    rng = np.random.default_rng(23)
    mask = _family("causal_document", N, 1, rng)
    q, k, v, do = W.make_inputs(1, N, H, d, dv, seed=27, device="cuda")
    vec = cuda_mask(mask)
    o, lse = fm.fwd(q, k, v, *vec, causal=mask.causal)
    g16 = fm.bwd(q, k, v, o, lse, do, *vec, causal=mask.causal, deterministic=True)
    fills = [torch.full((1, N, H, c), 0.25 * (i + 1), dtype=torch.float32, device="cuda")
             for i, c in enumerate((d, d, dv))]
    acc = [f.clone() for f in fills]
    fm.bwd(q, k, v, o, lse, do, *vec, causal=mask.causal, deterministic=True, dq=acc[0],
           dk=acc[1], dv=acc[2], accumulate_f32=True)
    fm.get_error()
    scale = 1 / np.sqrt(d)
    for h in range(H):
        qh, kh, vh, doh = head(q, 0, h), head(k, 0, h), head(v, 0, h), head(do, 0, h)
        refs = oracle.attention_bwd(qh, kh, vh, doh, mask_slice(mask, 0, h), mask.causal, scale)
        for name, a, f, g, ref in zip(("dQ", "dK", "dV"), acc, fills, g16, refs):
            got = (a - f)[0, :, h].double().cpu().numpy()
            assert_close(f"{name} accumulated", got, ref)
            # bf16 rounding is within 2^-9 relative; adding to and removing a
            # fill below 1 costs at most 2^-23 absolute in fp32.
            one = (a - f)[0, :, h]
            bound = 2.0 ** -8 * one.abs() + 2.0 ** -22
            assert ((one - g[0, :, h].float()).abs() <= bound).all(), name
