"""debug_bounds: the check kernel that reads every work list of the workspace
before the attention kernels run.

- With lists the library built itself the check passes, and every output is
  bit-identical to a run without it.
- With a reused workspace whose lists were damaged, the call reports
  FM_ERR_DEVICE_BOUNDS and the damaged lists are emptied before any attention
  kernel reads them.  Every damaged value is one step past its range, so even
  an access the check missed would stay inside the workspace: rows past N read
  as zeros through TMA, and the other reads land in the next workspace array.
  The workspace is allocated with slack at its end as well.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import cuda_mask
from sparse_masked_attention_gb300 import attention as fm
from sparse_masked_attention_gb300 import binding as _b
from sparse_masked_attention_gb300 import workloads as W

pytestmark = pytest.mark.gpu

WS_ALIGN = 256
SLACK = 1 << 20


def _layout(B, Hm, H, N, dv, bwd, fused_d=None):
    """Byte offsets of the workspace's tile map and lists, in the order the
    library lays them out, and the total size (pinned below against
    flashmask_workspace_size and the lists' contents)."""
    T = -(-N // 128)
    Npad, TP, BM = T * 128, (T + 1) // 2, B * Hm
    off, out = 0, {}

    def take(name, nbytes):
        nonlocal off
        out[name] = off
        off = -(-(off + nbytes) // WS_ALIGN) * WS_ALIGN

    take("vec", BM * Npad * 16)
    take("cls", BM * T * T)
    take("fwd_list", BM * T * T * 4)
    take("fwd_cnt", BM * T * 4)
    take("bwd_list", BM * T * T * 4)
    take("bwd_cnt", BM * T * 4)
    take("pair_list", BM * TP * T * 4)
    take("pair_cnt", BM * TP * 4)
    take("pair_order", BM * TP * 4)
    if bwd:
        rows = B * H * Npad
        take("lse2", rows * 4)
        take("delta", rows * 4)
        if not fused_d:  # the one-pass backward converts V in its own kernel
            take("v16", B * N * H * dv * 2)
        take("do16", B * N * H * dv * 2)
        take("sink_part", rows // 16 * 4)
        take("range_part", B * H * T * 8)
        take("scales", B * H * 16)
        if fused_d:  # the one-pass backward's fp32 dQ sums (not in deterministic mode)
            take("dqacc", rows * fused_d * 4)
    return out, off, T, TP


def _inputs(d, dv, N=1000, H=2):
    q, k, v, do = W.make_inputs(1, N, H, d, dv, seed=5, device="cuda")
    rng = np.random.default_rng(11)
    mask = W.causal_document(N, [W.uniform_lengths(rng, 60, 400, N)])
    return q, k, v, do, mask


def _step(q, k, v, do, vec, causal, ws, debug, reuse=False):
    o, lse = fm.fwd(q, k, v, *vec, causal=causal, workspace=ws,
                    options=fm.make_options(debug_bounds=debug, reuse_tile_map=reuse))
    # deterministic: the sums' order, and so their last bits, fixed
    grads = fm.bwd(q, k, v, o, lse, do, *vec, causal=causal, workspace=ws,
                   options=fm.make_options(deterministic=True, debug_bounds=debug,
                                           reuse_tile_map=True))
    return o, lse, grads


@pytest.mark.parametrize("d,dv", [(128, 128), (256, 256)])
def test_debug_bounds_passes_and_changes_nothing(d, dv):
    q, k, v, do, mask = _inputs(d, dv)
    vec = cuda_mask(mask)
    N, H = q.shape[1], q.shape[2]
    ws = torch.zeros(fm.workspace_size(1, H, 1, N, d, dv, True) + SLACK, dtype=torch.uint8,
                     device="cuda")
    ref = _step(q, k, v, do, vec, mask.causal, ws, debug=False)
    fm.get_error()
    got = _step(q, k, v, do, vec, mask.causal, ws, debug=True)
    fm.get_error()  # raises on any device error
    assert torch.equal(got[0], ref[0]) and torch.equal(got[1], ref[1])
    for g, r in zip(got[2], ref[2]):
        assert torch.equal(g, r)


def test_damaged_reused_lists_are_reported_and_emptied():
    d = dv = 128
    q, k, v, do, mask = _inputs(d, dv)
    vec = cuda_mask(mask)
    N, H = q.shape[1], q.shape[2]
    lay, total, T, TP = _layout(1, 1, H, N, dv, bwd=True)
    # the steps below run the deterministic backward, whose workspace has no
    # dQ buffer; the default backward's adds one at the end
    assert total == fm.workspace_size(1, H, 1, N, d, dv, True, deterministic=True)
    assert _layout(1, 1, H, N, dv, bwd=True, fused_d=d)[1] == \
        fm.workspace_size(1, H, 1, N, d, dv, True)
    ws = torch.zeros(total + SLACK, dtype=torch.uint8, device="cuda")
    _step(q, k, v, do, vec, mask.causal, ws, debug=False)
    fm.get_error()

    wsi = ws.view(torch.int32)

    def ints(name, n, first=0):
        s = lay[name] // 4 + first
        return wsi[s:s + n]

    # Pin the mirrored layout to the lists' contents before touching anything.
    cls, _ = oracle.tilemap(N, mask.slice(0), mask.causal)
    keep = cls != _b.FM_TILE_SKIP
    assert sorted(ints("pair_order", TP).tolist()) == list(range(TP))
    assert ints("fwd_cnt", T).tolist() == keep.sum(axis=1).tolist()
    assert ints("bwd_cnt", T).tolist() == keep.sum(axis=0).tolist()
    pairs = [int((keep[2 * p] | (keep[2 * p + 1] if 2 * p + 1 < T else False)).sum())
             for p in range(TP)]
    assert ints("pair_cnt", TP).tolist() == pairs
    assert pairs[0] > 0  # the damaged entry below is inside pair 0's list
    qt = int(np.argmax(keep.sum(axis=1) > 0))
    kt = int(np.argmax(keep.sum(axis=0) > 0))
    assert ints("fwd_list", 1, qt * T).item() >> 1 == int(np.argmax(keep[qt]))
    assert ints("bwd_list", 1, kt * T).item() >> 1 == int(np.argmax(keep[:, kt]))

    # One step past each range: a key tile T, a query tile T, a pair TP.
    ints("pair_list", 1, 0)[0] = T << 2
    ints("fwd_list", 1, qt * T)[0] = T << 1
    ints("bwd_list", 1, kt * T)[0] = T << 1
    ints("pair_order", 1, 1)[0] = TP
    o, lse = fm.fwd(q, k, v, *vec, causal=mask.causal, workspace=ws,
                    options=fm.make_options(debug_bounds=True, reuse_tile_map=True))
    with pytest.raises(fm.FlashMaskError) as err:
        fm.get_error()
    assert err.value.status == _b.FM_ERR_DEVICE_BOUNDS
    # emptied before the attention kernels read them
    assert ints("pair_cnt", 1, 0).item() == 0
    assert ints("fwd_cnt", 1, qt).item() == 0
    assert ints("bwd_cnt", 1, kt).item() == 0
    assert ints("pair_order", 1, 1).item() == 1
    fm.get_error()  # the error word was cleared by the read

    # A count past its range, seen by the backward.
    ints("bwd_cnt", 1, kt)[0] = T + 1
    fm.bwd(q, k, v, o, lse, do, *vec, causal=mask.causal, workspace=ws,
           options=fm.make_options(deterministic=True, debug_bounds=True, reuse_tile_map=True))
    with pytest.raises(fm.FlashMaskError) as err:
        fm.get_error()
    assert err.value.status == _b.FM_ERR_DEVICE_BOUNDS
    assert ints("bwd_cnt", 1, kt).item() == 0
    fm.get_error()

    # Without reuse the call rebuilds every list, and the check passes again.
    _step(q, k, v, do, vec, mask.causal, ws, debug=True)
    fm.get_error()
