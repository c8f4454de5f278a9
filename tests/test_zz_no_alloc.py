"""flashmask_fwd_noalloc: the forward for callers that cannot allocate device
memory.

Such callers (a host that lends only its own tensors, code where cudaMalloc
is not allowed) cannot pass a workspace.  The entry point uses the library's
fixed 16 MiB device array instead.  These tests call it through the C ABI and
check it against flashmask_fwd with an ordinary workspace.  Two calls run in
a row with different masks and sizes, because the array keeps the previous
call's contents.  The file is named to run last, after every other test, and
it also passes alone in a fresh process.
"""
import numpy as np
import pytest
import torch

from sparse_masked_attention_gb300 import attention as fm
from sparse_masked_attention_gb300 import binding as B
from sparse_masked_attention_gb300 import build as build_mod
from sparse_masked_attention_gb300 import workloads as W

from gpu_util import LSE_ABS, assert_close, cuda_mask


@pytest.fixture(scope="module")
def lib():
    build_mod.build()
    return B.load()


def _ptrs(vec):
    return [None if t is None else t.data_ptr() for t in vec]


def _run_both(mask, Bn, H, N, d, dv, seed):
    q, k, v, _ = W.make_inputs(Bn, N, H, d, dv, seed=seed, device="cuda", with_dout=False)
    vec = cuda_mask(mask)
    prob = fm.make_problem(Bn, H, 1, N, d, dv, None, mask.causal)
    stream = torch.cuda.current_stream().cuda_stream
    # regular entry point, caller-provided workspace
    o_ref = torch.empty((Bn, N, H, dv), dtype=torch.bfloat16, device="cuda")
    lse_ref = torch.empty((Bn, H, N), dtype=torch.float32, device="cuda")
    ws = torch.empty(B.flashmask_workspace_size(prob, None, 0), dtype=torch.uint8,
                     device="cuda")
    st = B.flashmask_fwd(prob, None, q.data_ptr(), k.data_ptr(), v.data_ptr(), *_ptrs(vec),
                         o_ref.data_ptr(), lse_ref.data_ptr(), ws.data_ptr(), ws.numel(), stream)
    assert st == B.FM_OK
    # no-workspace entry point
    o = torch.full_like(o_ref, float("nan"))
    lse = torch.full_like(lse_ref, float("nan"))
    st = B.flashmask_fwd_noalloc(prob, None, q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                 *_ptrs(vec), o.data_ptr(), lse.data_ptr(), stream)
    assert st == B.FM_OK, B.flashmask_last_error_detail()
    assert B.flashmask_get_error(stream) == B.FM_OK
    return o, lse, o_ref, lse_ref


@pytest.mark.gpu
def test_noalloc_forward_matches_workspace_forward_twice(lib):
    rng = np.random.default_rng(5)
    cases = [
        (W.causal_document(1000, [W.uniform_lengths(rng, 60, 300, 1000)]), 1, 2, 1000, 128, 128),
        (W.sliding_window(777, 150, 2), 2, 3, 777, 64, 64),
    ]
    for i, (mask, Bn, H, N, d, dv) in enumerate(cases):
        o, lse, o_ref, lse_ref = _run_both(mask, Bn, H, N, d, dv, seed=20 + i)
        assert torch.isfinite(o.float()).all()
        assert_close(f"noalloc O call {i}", o.float().cpu().numpy(), o_ref.float().cpu().numpy())
        err = (lse - lse_ref).abs().max().item()
        assert err <= LSE_ABS, f"noalloc LSE call {i}: {err:.3e}"


def test_noalloc_rejects_problems_beyond_the_static_scratch(lib):
    # N = 131072 with two mask heads needs about 23 MiB of forward scratch.
    prob = fm.make_problem(2, 2, 1, 131072, 128, 128, None, True)
    need = B.flashmask_workspace_size(prob, None, 0)
    assert need > B.FM_NOALLOC_SCRATCH_BYTES
    st = B.flashmask_fwd_noalloc(prob, None, 256, 256, 256, None, None, None, None, 256, 256,
                                 None)
    assert st == B.FM_ERR_WORKSPACE
    assert "static scratch" in B.flashmask_last_error_detail()


def test_noalloc_refuses_a_reused_tile_map(lib):
    # The static array may hold another problem's tile map, so a call that asks
    # to reuse it is refused before any CUDA call (this runs without a GPU).
    prob = fm.make_problem(1, 2, 1, 1000, 128, 128, None, True)
    opt = fm.make_options(reuse_tile_map=True)
    st = B.flashmask_fwd_noalloc(prob, opt, 256, 256, 256, None, None, None, None, 256, 256,
                                 None)
    assert st == B.FM_ERR_INVALID_ARG
    assert "reuse_tile_map" in B.flashmask_last_error_detail()


@pytest.mark.gpu
def test_noalloc_passes_options_through(lib):
    # A sink and the list check (debug_bounds) reach the kernels exactly as they
    # do through flashmask_fwd: same outputs, and the check reports nothing.
    rng = np.random.default_rng(9)
    N, H, d = 900, 3, 128
    mask = W.causal_document(N, [W.uniform_lengths(rng, 80, 400, N)])
    q, k, v, _ = W.make_inputs(1, N, H, d, d, seed=31, device="cuda", with_dout=False)
    vec = cuda_mask(mask)
    sink = torch.tensor([0.5, -1.0, 2.0], dtype=torch.float32, device="cuda")
    prob = fm.make_problem(1, H, 1, N, d, d, None, mask.causal)
    opt = fm.make_options(sink=sink, debug_bounds=True)
    stream = torch.cuda.current_stream().cuda_stream
    o_ref = torch.empty((1, N, H, d), dtype=torch.bfloat16, device="cuda")
    lse_ref = torch.empty((1, H, N), dtype=torch.float32, device="cuda")
    ws = torch.empty(B.flashmask_workspace_size(prob, opt, 0), dtype=torch.uint8, device="cuda")
    st = B.flashmask_fwd(prob, opt, q.data_ptr(), k.data_ptr(), v.data_ptr(), *_ptrs(vec),
                         o_ref.data_ptr(), lse_ref.data_ptr(), ws.data_ptr(), ws.numel(), stream)
    assert st == B.FM_OK
    for call in range(2):
        o = torch.full_like(o_ref, float("nan"))
        lse = torch.full_like(lse_ref, float("nan"))
        st = B.flashmask_fwd_noalloc(prob, opt, q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                     *_ptrs(vec), o.data_ptr(), lse.data_ptr(), stream)
        assert st == B.FM_OK, B.flashmask_last_error_detail()
        assert B.flashmask_get_error(stream) == B.FM_OK
        assert torch.equal(o, o_ref), f"call {call}: O differs from flashmask_fwd"
        assert torch.equal(lse, lse_ref), f"call {call}: LSE differs from flashmask_fwd"
