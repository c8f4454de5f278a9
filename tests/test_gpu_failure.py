"""Failure detection on the GPU without a fault: a device wait that nothing
completes gives up after its limit, the host reads the timeout status, and the
context stays usable for the next calls."""
import time

import pytest
import torch

from gpu_util import check_head_full, cuda_mask
from sparse_masked_attention_gb300 import attention as fm
from sparse_masked_attention_gb300 import binding as _b
from sparse_masked_attention_gb300 import workloads as W



@pytest.mark.gpu
def test_bounded_wait_gives_up_and_the_context_stays_usable():
    torch.cuda.synchronize()
    fm.get_error()  # start clean
    t0 = time.perf_counter()
    fm.selftest_wait(50_000_000)  # 50 ms
    with pytest.raises(fm.FlashMaskError) as err:
        fm.get_error()
    elapsed = time.perf_counter() - t0
    assert err.value.status == _b.FM_ERR_DEVICE_TIMEOUT
    assert 0.05 <= elapsed < 5.0
    fm.get_error()  # reading the status cleared it

    # The library still computes correct results on this context.
    B, H, N, d = 1, 2, 300, 128
    q, k, v, do = W.make_inputs(B, N, H, d, d, seed=8, device="cuda")
    mask = W.causal(N, B)
    lts, lte, uts, ute = cuda_mask(mask)
    o, lse = fm.fwd(q, k, v, lts, lte, uts, ute, mask.causal)
    grads = fm.bwd(q, k, v, o, lse, do, lts, lte, uts, ute, mask.causal)
    fm.get_error()
    check_head_full(q, k, v, do, mask, o, lse, grads, 0, 1)


@pytest.mark.gpu
def test_nvtx_ranges_wrap_the_calls():
    B, H, N, d = 1, 2, 300, 64
    q, k, v, do = W.make_inputs(B, N, H, d, d, seed=9, device="cuda")
    ref_o, ref_lse = fm.fwd(q, k, v, causal=True)
    fm.set_nvtx(True)
    try:
        o, lse = fm.fwd(q, k, v, causal=True)
        fm.bwd(q, k, v, o, lse, do, causal=True)
    finally:
        fm.set_nvtx(False)
    fm.get_error()
    assert torch.equal(o, ref_o) and torch.equal(lse, ref_lse)


@pytest.mark.gpu
def test_forward_kernel_drains_after_its_waits_run_out():
    """An attention kernel's own drain: with debug_drop_load the forward never
    issues one key-tile load per CTA, so the waits for it run out after 20 ms.
    Every role leaves its loop, the producers wait for their loads still in
    flight, the MMA thread for its MMAs, TMEM is freed and the kernel returns:
    the host reads FM_ERR_DEVICE_TIMEOUT, and the same context then computes
    correct results."""
    torch.cuda.synchronize()
    fm.get_error()  # start clean
    B, H, N, d = 1, 2, 1000, 128  # causal: every query-tile pair has >= 2 key tiles
    q, k, v, do = W.make_inputs(B, N, H, d, d, seed=12, device="cuda")
    mask = W.causal(N, B)
    vec = cuda_mask(mask)
    opt = fm.make_options(wait_timeout_ns=20_000_000, debug_drop_load=2)
    t0 = time.perf_counter()
    fm.fwd(q, k, v, *vec, causal=True, options=opt)
    with pytest.raises(fm.FlashMaskError) as err:
        fm.get_error()
    elapsed = time.perf_counter() - t0
    assert err.value.status == _b.FM_ERR_DEVICE_TIMEOUT
    assert 0.02 <= elapsed < 5.0
    fm.get_error()  # reading the status cleared it

    o, lse = fm.fwd(q, k, v, *vec, causal=True)
    grads = fm.bwd(q, k, v, o, lse, do, *vec, causal=True)
    fm.get_error()
    for h in range(H):
        check_head_full(q, k, v, do, mask, o, lse, grads, 0, h)


def test_drop_load_option_is_checked():
    prob = fm.make_problem(1, 2, 1, 256, 128, 128, None, True)
    assert _b.flashmask_workspace_size(prob, fm.make_options(debug_drop_load=-1), 0) == 0
    assert _b.flashmask_workspace_size(prob, fm.make_options(debug_drop_load=3), 0) > 0
