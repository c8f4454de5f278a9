"""Parity at the workloads' full sizes, in the launch configuration bench.py times.

Every workload runs at full size through the public API, and is checked four
ways against the oracle:
- the tile map, bit-exact against the oracle's brute-force count;
- O, LSE and dQ on sampled query rows (rows are independent given K and V,
  so the oracle can compute each one alone);
- dK and dV on the key columns whose visible rows the oracle can afford;
- unmasked-pair counts against closed forms, where one exists.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from sparse_masked_attention_gb300 import attention as fm
from sparse_masked_attention_gb300 import workloads as W

from gpu_util import assert_close, assert_lse, cuda_mask, head, mask_slice

pytestmark = pytest.mark.gpu

NAMES = [n for n in W.CONFIGS if n != "tiny_causal_document"]


def _rows(N, rng, n=48):
    fixed = [0, 1, 127, 128, N // 2, N - 129, N - 128, N - 1]
    rnd = rng.choice(N, size=n - len(fixed), replace=False).tolist()
    return sorted(set(r for r in fixed + rnd if 0 <= r < N))


def _visible_rows_per_column(ms, causal, N):
    """Number of rows that see each key column (closed form per column)."""
    j = np.arange(N, dtype=np.int64)
    clamp = lambda x: np.clip(np.asarray(x, np.int64), 0, N)
    a0, b0 = np.zeros(N, np.int64), (j if causal else np.zeros(N, np.int64))
    a1 = clamp(ms["lts"]) if ms["lts"] is not None else np.full(N, N)
    b1 = clamp(ms["lte"]) if ms["lte"] is not None else np.full(N, N)
    a2 = clamp(ms["uts"]) if ms["uts"] is not None else np.zeros(N, np.int64)
    b2 = clamp(ms["ute"]) if ms["ute"] is not None else np.zeros(N, np.int64)
    ln = lambda a, b: np.maximum(b - a, 0)
    ln2 = lambda a, b, c, d: ln(np.maximum(a, c), np.minimum(b, d))
    s1 = ln(a0, b0) + ln(a1, b1) + ln(a2, b2)
    s2 = ln2(a0, b0, a1, b1) + ln2(a0, b0, a2, b2) + ln2(a1, b1, a2, b2)
    s3 = ln(np.maximum(a0, np.maximum(a1, a2)), np.minimum(b0, np.minimum(b1, b2)))
    return N - (s1 - s2 + s3)


def _cols(ms, causal, N, rng, budget_rows=3000, n=10):
    vis = _visible_rows_per_column(ms, causal, N)
    last = list(range(max(0, N - 128), N, 29)) + [N - 1]
    cand = [c for c in rng.choice(N, size=400, replace=False).tolist()
            if 0 < vis[c] <= budget_rows]
    cols = sorted(set(last + cand[: n - len(last)]))
    return [c for c in cols if vis[c] <= budget_rows or c >= N - 128]


@pytest.fixture(scope="module", params=NAMES)
def run(request):
    name = request.param
    cfg = W.CONFIGS[name]
    B, H, N, d, dv = cfg["B"], cfg["H"], cfg["N"], cfg["d"], cfg["dv"]
    torch.cuda.empty_cache()
    q, k, v, do = W.make_inputs(B, N, H, d, dv, seed=0, device="cuda")
    mask = W.make_mask(cfg, seed=0)
    vec = cuda_mask(mask)
    o, lse = fm.fwd(q, k, v, *vec, causal=mask.causal)
    grads = None
    if "bwd" in cfg["passes"]:
        grads = fm.bwd(q, k, v, o, lse, do, *vec, causal=mask.causal,
                       deterministic=cfg.get("deterministic", False))
    fm.get_error()
    yield name, cfg, q, k, v, do, mask, vec, o, lse, grads
    del q, k, v, do, o, lse, grads
    torch.cuda.empty_cache()


def test_tile_map_full_size(run):
    name, cfg, q, k, v, do, mask, vec, o, lse, grads = run
    N, B = cfg["N"], cfg["B"]
    got = fm.classify(N, B, 1, *vec, causal=mask.causal).cpu().numpy()
    want, visible = oracle.tilemap(N, mask.slice(0), mask.causal)
    np.testing.assert_array_equal(got[0], want)
    cnt = fm.count_unmasked(N, B, 1, *vec, causal=mask.causal).cpu().numpy()
    assert int(cnt[0]) == visible
    if cfg["mask"] == "causal":
        assert int(cnt[0]) == N * (N + 1) // 2
    if cfg["mask"] == "sliding":
        w = cfg["w"]
        assert int(cnt[0]) == sum(min(i + 1, w) for i in range(N))
    if cfg["mask"] == "prefix_lm":
        P = cfg["prefix"]
        assert int(cnt[0]) == P * N + (N - P) * (N - P + 1) // 2


def test_sampled_rows(run):
    name, cfg, q, k, v, do, mask, vec, o, lse, grads = run
    B, H, N, d = cfg["B"], cfg["H"], cfg["N"], cfg["d"]
    rng = np.random.default_rng(1)
    scale = 1 / math.sqrt(d)
    for (b, h) in sorted({(0, 0), (B - 1, H - 1)}):
        rows = _rows(N, rng)
        qh, kh, vh = head(q, b, h), head(k, b, h), head(v, b, h)
        ms = mask_slice(mask, b, h)
        ro, rl = oracle.attention_fwd(qh, kh, vh, ms, mask.causal, scale, rows=rows)
        assert_close(f"{name} O rows", head(o, b, h)[rows], ro)
        assert_lse(lse[b, h].cpu().numpy()[rows], rl)
        if grads is not None:
            rdq, _ = oracle.attention_bwd_dq(qh, kh, vh, head(do, b, h), ms, mask.causal, scale,
                                             rows=rows)
            assert_close(f"{name} dQ rows", head(grads[0], b, h)[rows], rdq)


def test_sampled_columns(run):
    name, cfg, q, k, v, do, mask, vec, o, lse, grads = run
    if grads is None:
        pytest.skip("forward-only workload")
    B, H, N, d = cfg["B"], cfg["H"], cfg["N"], cfg["d"]
    rng = np.random.default_rng(2)
    scale = 1 / math.sqrt(d)
    b, h = B - 1, H - 1
    ms = mask_slice(mask, b, h)
    cols = _cols(ms, mask.causal, N, rng)
    qh, kh, vh, doh = head(q, b, h), head(k, b, h), head(v, b, h), head(do, b, h)
    rdk, rdv = oracle.attention_bwd_dkdv(qh, kh, vh, doh, ms, mask.causal, scale, cols=cols)
    assert_close(f"{name} dK cols", head(grads[1], b, h)[cols], rdk)
    assert_close(f"{name} dV cols", head(grads[2], b, h)[cols], rdv)


def test_deterministic_full_size(run):
    name, cfg, q, k, v, do, mask, vec, o, lse, grads = run
    if not cfg.get("deterministic", False):
        pytest.skip("workload does not ask for the deterministic mode")
    g2 = fm.bwd(q, k, v, o, lse, do, *vec, causal=mask.causal, deterministic=True)
    fm.get_error()
    for a, b_ in zip(grads, g2):
        assert torch.equal(a, b_)
