"""Helpers shared by the GPU parity tests: run the CUDA path through the
C-ABI front end and the fp64 oracle on the same seeded inputs."""
import math

import numpy as np
import torch

import oracle
from sparse_masked_attention_gb300 import attention as fm
from sparse_masked_attention_gb300 import workloads as W

# Tolerance on O, dQ, dK, dV against the fp64 oracle: bf16 inputs, fp32
# accumulation, bf16 outputs.
MAX_ABS = 2e-2
REL_L2 = 1e-2
# LSE is written in fp32 from fp32 row statistics.
LSE_ABS = 1e-3


def cuda_mask(mask: W.Mask, device="cuda"):
    out = []
    for name in ("lts", "lte", "uts", "ute"):
        x = getattr(mask, name)
        out.append(None if x is None else torch.from_numpy(np.ascontiguousarray(x)).to(device))
    return out


def head(t, b, h):
    """[B, N, H, c] tensor -> fp64 numpy [N, c] of one (b, h)."""
    return t[b, :, h, :].float().cpu().numpy().astype(np.float64)


def mask_slice(mask: W.Mask, b, h):
    Hm = 1 if mask.lts is None and mask.uts is None else (
        (mask.lts if mask.lts is not None else mask.uts).shape[1])
    return mask.slice(b, 0 if Hm == 1 else h)


def errors(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    diff = got - ref
    max_abs = float(np.max(np.abs(diff))) if diff.size else 0.0
    den = float(np.linalg.norm(ref))
    rel = float(np.linalg.norm(diff) / den) if den > 0 else float(np.linalg.norm(diff))
    return max_abs, rel


def assert_close(name, got, ref, max_abs=MAX_ABS, rel_l2=REL_L2):
    ma, rl = errors(got, ref)
    assert ma <= max_abs and rl <= rel_l2, (
        f"{name}: max|err|={ma:.3e} (tol {max_abs}), relL2={rl:.3e} (tol {rel_l2}), "
        f"max|ref|={float(np.max(np.abs(ref))) if np.size(ref) else 0:.3e}")
    return ma, rl


def assert_lse(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    inf = np.isneginf(ref)
    assert np.array_equal(np.isneginf(got), inf), "fully masked rows must have LSE = -inf"
    if (~inf).any():
        d = float(np.max(np.abs(got[~inf] - ref[~inf])))
        assert d <= LSE_ABS, f"lse max|err| {d:.3e}"


def run_fwd_bwd(q, k, v, dout, mask: W.Mask, scale=None, deterministic=False, bwd=True):
    lts, lte, uts, ute = cuda_mask(mask, q.device)
    o, lse = fm.fwd(q, k, v, lts, lte, uts, ute, mask.causal, scale)
    grads = None
    if bwd:
        grads = fm.bwd(q, k, v, o, lse, dout, lts, lte, uts, ute, mask.causal, scale,
                       deterministic)
    fm.get_error()
    return o, lse, grads


def check_head_full(q, k, v, dout, mask, o, lse, grads, b, h, scale=None):
    """Element-by-element comparison of one (b, h) slice with the oracle."""
    d = q.shape[-1]
    scale = 1 / math.sqrt(d) if scale is None else scale
    qh, kh, vh = head(q, b, h), head(k, b, h), head(v, b, h)
    ms = mask_slice(mask, b, h)
    ro, rl = oracle.attention_fwd(qh, kh, vh, ms, mask.causal, scale)
    assert_close("O", head(o, b, h), ro)
    assert_lse(lse[b, h].cpu().numpy(), rl)
    if grads is not None:
        doh = head(dout, b, h)
        rdq, rdk, rdv = oracle.attention_bwd(qh, kh, vh, doh, ms, mask.causal, scale)
        assert_close("dQ", head(grads[0], b, h), rdq)
        assert_close("dK", head(grads[1], b, h), rdk)
        assert_close("dV", head(grads[2], b, h), rdv)
