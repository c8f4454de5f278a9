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

pytestmark = pytest.mark.gpu


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
