"""Pins of the fp64 oracle against facts fixed outside the oracle itself.

Each test ties the oracle to an independent source: a hand-worked closed form,
a library routine (torch fp64 softmax/logsumexp/autograd), a mask family's
semantic definition, finite differences, or an invariant of the formula.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from sparse_masked_attention_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def _torch_masked_attention(q, k, v, masked, scale):
    """fp64 torch: softmax(q k^T * scale + M) v with M = -inf where masked."""
    q, k, v = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
    s = (q @ k.T) * scale
    s = s.masked_fill(torch.tensor(masked), float("-inf"))
    p = torch.softmax(s, dim=-1)
    o = p @ v
    lse = torch.logsumexp(s, dim=-1)
    return q, k, v, o, lse


# ------------------------------------------------------------- closed form


@pytest.mark.parametrize("case", ["full", "causal"])
def test_hand_worked_two_keys(case):
    g = json.load(open(os.path.join(GOLDEN, "two_keys_hand_worked.json")))
    c = g["cases"][case]
    q, k, v, do = (np.array(g[x]) for x in ("q", "k", "v", "dout"))
    o, lse = oracle.attention_fwd(q, k, v, causal=c["causal"], scale=g["scale"])
    np.testing.assert_allclose(o, c["o"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, c["lse"], rtol=0, atol=1e-12)
    dq, dk, dvv = oracle.attention_bwd(q, k, v, do, causal=c["causal"], scale=g["scale"])
    np.testing.assert_allclose(dq, c["dq"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(dk, c["dk"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(dvv, c["dv"], rtol=0, atol=1e-12)


# ------------------------------------------------- library routine (torch)


@pytest.mark.parametrize("N,d,dv", [(37, 8, 5), (64, 16, 16)])
def test_unmasked_equals_plain_attention(N, d, dv):
    q, k, v, do = (_rand((N, c), s) for s, c in enumerate((d, d, dv, dv)))
    scale = 1 / math.sqrt(d)
    tq, tk, tv, to, tl = _torch_masked_attention(q, k, v, np.zeros((N, N), bool), scale)
    o, lse = oracle.attention_fwd(q, k, v, scale=scale)
    np.testing.assert_allclose(o, to.detach().numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, tl.detach().numpy(), rtol=1e-12, atol=1e-12)
    (to * torch.tensor(do)).sum().backward()
    dq, dk, dvv = oracle.attention_bwd(q, k, v, do, scale=scale)
    np.testing.assert_allclose(dq, tq.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dk, tk.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dvv, tv.grad.numpy(), rtol=1e-10, atol=1e-12)


def test_default_scale_is_inverse_sqrt_d():
    N, d, dv = 20, 9, 4
    q, k, v = (_rand((N, c), s) for s, c in enumerate((d, d, dv)))
    a, la = oracle.attention_fwd(q, k, v)
    b, lb = oracle.attention_fwd(q, k, v, scale=1 / 3.0)
    np.testing.assert_array_equal(a, b)
    np.testing.assert_array_equal(la, lb)


def test_causal_equals_bruteforce_triangle():
    N, d, dv = 45, 8, 6
    q, k, v, do = (_rand((N, c), 10 + s) for s, c in enumerate((d, d, dv, dv)))
    scale = 0.4
    tri = np.triu(np.ones((N, N), bool), k=1)          # i < j masked
    tq, tk, tv, to, tl = _torch_masked_attention(q, k, v, tri, scale)
    o, lse = oracle.attention_fwd(q, k, v, causal=True, scale=scale)
    np.testing.assert_allclose(o, to.detach().numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, tl.detach().numpy(), rtol=1e-12, atol=1e-12)
    (to * torch.tensor(do)).sum().backward()
    dq, dk, dvv = oracle.attention_bwd(q, k, v, do, causal=True, scale=scale)
    np.testing.assert_allclose(dq, tq.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dk, tk.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dvv, tv.grad.numpy(), rtol=1e-10, atol=1e-12)


# ---------------------------------------- mask families vs their semantics


def _families(N, seed=3):
    rng = np.random.default_rng(seed)
    return [
        W.causal(N),
        W.sliding_window(N, 7),
        W.causal_document(N, [W.uniform_lengths(rng, 5, 17, N)]),
        W.causal_document(N, [W.three_documents(rng, N)]),
        W.prefix_lm(N, 11),
        W.share_question(N, [W.share_question_groups(rng, N, (4, 9), (2, 4), (2, 6))]),
        W.block_sparse(N, rng, blk=8),
        W.global_sliding(N, 5, 9),
    ]


@pytest.mark.parametrize("idx", range(8))
def test_family_attention_equals_dense_semantic(idx):
    N, d, dv = 50, 8, 7
    mask = _families(N)[idx]
    sem = W.dense_semantic(mask, 0)
    assert not sem.all(axis=1).any(), "families keep every row visible"
    q, k, v, do = (_rand((N, c), 20 + s) for s, c in enumerate((d, d, dv, dv)))
    scale = 1 / math.sqrt(d)
    tq, tk, tv, to, tl = _torch_masked_attention(q, k, v, sem, scale)
    o, lse = oracle.attention_fwd(q, k, v, mask.slice(0), mask.causal, scale)
    np.testing.assert_allclose(o, to.detach().numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, tl.detach().numpy(), rtol=1e-12, atol=1e-12)
    (to * torch.tensor(do)).sum().backward()
    dq, dk, dvv = oracle.attention_bwd(q, k, v, do, mask.slice(0), mask.causal, scale)
    np.testing.assert_allclose(dq, tq.grad.numpy(), rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(dk, tk.grad.numpy(), rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(dvv, tv.grad.numpy(), rtol=1e-10, atol=1e-11)


@pytest.mark.parametrize("idx", range(8))
def test_element_map_equals_dense_semantic(idx):
    """The oracle's 1x1 tile map is its dense expansion of the vectors."""
    N = 61
    mask = _families(N, seed=5)[idx]
    cls, visible = oracle.tilemap(N, mask.slice(0), mask.causal, tq=1, tk=1)
    sem = W.dense_semantic(mask, 0)
    np.testing.assert_array_equal(cls == oracle.TILE_SKIP, sem)
    assert set(np.unique(cls)) <= {oracle.TILE_SKIP, oracle.TILE_UNMASKED}
    assert visible == int((~sem).sum())


# -------------------------------------------------------------- invariants


def test_finite_differences():
    N, d, dv = 13, 4, 3
    rng = np.random.default_rng(7)
    mask = W.causal_document(N, [[4, 6, 3]])
    q, k, v, do = (rng.standard_normal((N, c)) for c in (d, d, dv, dv))
    scale = 0.7

    def loss(q_, k_, v_):
        o, _ = oracle.attention_fwd(q_, k_, v_, mask.slice(0), True, scale)
        return float((o * do).sum())

    dq, dk, dvv = oracle.attention_bwd(q, k, v, do, mask.slice(0), True, scale)
    h = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dvv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(*x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args = {"q": (q, k, v), "k": (q, k, v), "v": (q, k, v)}[name]
            ap = [xp if a is x else a for a in args]
            am = [xm if a is x else a for a in args]
            num[idx] = (loss(*ap) - loss(*am)) / (2 * h)
        np.testing.assert_allclose(g, num, rtol=1e-6, atol=1e-8, err_msg=name)


@pytest.mark.parametrize("f", [1e-9, 3.0, 1e5])
def test_homogeneity_in_dout_and_v(f):
    """The derivative is linear in dO, so every gradient scales with it; O and
    dP are linear in V while P is not affected, so O, dQ and dK scale with V
    and dV does not.  The GPU tests of extreme input ranges lean on this."""
    N, d, dv = 40, 8, 6
    rng = np.random.default_rng(17)
    mask = W.causal_document(N, [[15, 25]]).slice(0)
    q, k, v, do = (rng.standard_normal((N, c)) for c in (d, d, dv, dv))
    o, lse = oracle.attention_fwd(q, k, v, mask, True)
    g = oracle.attention_bwd(q, k, v, do, mask, True)
    g_do = oracle.attention_bwd(q, k, v, do * f, mask, True)
    for a, b in zip(g, g_do):
        np.testing.assert_allclose(b, a * f, rtol=1e-12, atol=0)
    o_v, lse_v = oracle.attention_fwd(q, k, v * f, mask, True)
    np.testing.assert_allclose(o_v, o * f, rtol=1e-12, atol=0)
    np.testing.assert_array_equal(lse_v, lse)
    gq, gk, gv = oracle.attention_bwd(q, k, v * f, do, mask, True)
    np.testing.assert_allclose(gq, g[0] * f, rtol=1e-9, atol=0)
    np.testing.assert_allclose(gk, g[1] * f, rtol=1e-9, atol=0)
    np.testing.assert_allclose(gv, g[2], rtol=1e-12, atol=0)


def test_softmax_rows_sum_to_one():
    """With V = 1 every visible row of O is sum_j P_ij = 1."""
    N, d = 70, 8
    rng = np.random.default_rng(1)
    mask = W.share_question(N, [W.share_question_groups(rng, N, (5, 12), (2, 4), (3, 8))])
    q, k = (rng.standard_normal((N, d)) for _ in range(2))
    o, _ = oracle.attention_fwd(q, k, np.ones((N, 3)), mask.slice(0), True)
    np.testing.assert_allclose(o, 1.0, rtol=0, atol=1e-13)


def test_fully_masked_rows_convention():
    """Rows 3 and 4 see no key: O = 0, LSE = -inf, dQ = 0, no dK/dV share."""
    N, d, dv = 10, 4, 3
    rng = np.random.default_rng(2)
    q, k, v, do = (rng.standard_normal((N, c)) for c in (d, d, dv, dv))
    mask = {"lts": np.full(N, 3, np.int32), "lte": np.full(N, 5, np.int32)}
    o, lse = oracle.attention_fwd(q, k, v, mask)
    assert np.all(o[3:5] == 0.0) and np.all(lse[3:5] == -np.inf)
    assert np.all(np.isfinite(lse[:3])) and np.all(np.isfinite(lse[5:]))
    dq, dk, dvv = oracle.attention_bwd(q, k, v, do, mask)
    assert np.all(dq[3:5] == 0.0)
    do2 = do.copy()
    do2[3:5] = 100.0 * rng.standard_normal((2, dv))
    q2 = q.copy()
    q2[3:5] = 100.0 * rng.standard_normal((2, d))
    _, dk2, dv2 = oracle.attention_bwd(q2, k, v, do2, mask)
    np.testing.assert_array_equal(dk, dk2)
    np.testing.assert_array_equal(dvv, dv2)


def test_document_mask_equals_separate_documents():
    N, d, dv = 40, 6, 5
    lengths = [9, 17, 14]
    rng = np.random.default_rng(4)
    q, k, v, do = (rng.standard_normal((N, c)) for c in (d, d, dv, dv))
    mask = W.causal_document(N, [lengths])
    o, lse = oracle.attention_fwd(q, k, v, mask.slice(0), True)
    dq, dk, dvv = oracle.attention_bwd(q, k, v, do, mask.slice(0), True)
    a = 0
    for n in lengths:
        s = slice(a, a + n)
        o1, l1 = oracle.attention_fwd(q[s], k[s], v[s], None, True, 1 / math.sqrt(d))
        g1 = oracle.attention_bwd(q[s], k[s], v[s], do[s], None, True, 1 / math.sqrt(d))
        np.testing.assert_allclose(o[s], o1, rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(lse[s], l1, rtol=1e-13, atol=1e-14)
        for got, ref in zip((dq[s], dk[s], dvv[s]), g1):
            np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-13)
        a += n


def test_causal_flag_equals_upper_interval_encoding():
    """causal=1 with no vectors == causal=0 with UTS_j = 0, UTE_j = j."""
    N, d, dv = 33, 5, 4
    rng = np.random.default_rng(6)
    q, k, v, do = (rng.standard_normal((N, c)) for c in (d, d, dv, dv))
    enc = {"uts": np.zeros(N, np.int32), "ute": np.arange(N, dtype=np.int32)}
    a = oracle.attention_fwd(q, k, v, None, True)
    b = oracle.attention_fwd(q, k, v, enc, False)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)
    ga = oracle.attention_bwd(q, k, v, do, None, True)
    gb = oracle.attention_bwd(q, k, v, do, enc, False)
    for x, y in zip(ga, gb):
        np.testing.assert_array_equal(x, y)


def test_rows_and_columns_subsets_match_full():
    N, d, dv = 57, 8, 8
    rng = np.random.default_rng(8)
    q, k, v, do = (rng.standard_normal((N, c)) for c in (d, d, dv, dv))
    mask = W.sliding_window(N, 9)
    full_o, full_l = oracle.attention_fwd(q, k, v, mask.slice(0), True)
    full_dq, full_dk, full_dv = oracle.attention_bwd(q, k, v, do, mask.slice(0), True)
    rows = [0, 5, 56, 30]
    o, l = oracle.attention_fwd(q, k, v, mask.slice(0), True, rows=rows)
    np.testing.assert_array_equal(o, full_o[rows])
    np.testing.assert_array_equal(l, full_l[rows])
    dq, _ = oracle.attention_bwd_dq(q, k, v, do, mask.slice(0), True, rows=rows)
    np.testing.assert_array_equal(dq, full_dq[rows])
    cols = [56, 1, 20]
    dk, dvv = oracle.attention_bwd_dkdv(q, k, v, do, mask.slice(0), True, cols=cols)
    np.testing.assert_allclose(dk, full_dk[cols], rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(dvv, full_dv[cols], rtol=1e-14, atol=1e-15)


# --------------------------------------------------- tile map closed forms


@pytest.mark.parametrize("N", [512, 128 * 5 + 77])
def test_tilemap_causal_closed_form(N):
    cls, visible = oracle.tilemap(N, None, True)
    n = cls.shape[0]
    qt, kt = np.meshgrid(np.arange(n), np.arange(n), indexing="ij")
    want = np.where(kt > qt, oracle.TILE_SKIP,
                    np.where(kt < qt, oracle.TILE_UNMASKED, oracle.TILE_PARTIAL))
    np.testing.assert_array_equal(cls, want)
    assert visible == N * (N + 1) // 2


def test_tilemap_sliding_closed_form():
    N, w = 2048, 384                          # w = 3 tiles
    mask = W.sliding_window(N, w)
    cls, visible = oracle.tilemap(N, mask.slice(0), True)
    n = N // 128
    qt, kt = np.meshgrid(np.arange(n), np.arange(n), indexing="ij")
    dlt = qt - kt
    want = np.full((n, n), oracle.TILE_PARTIAL)
    want[(dlt >= 1) & (dlt < w // 128)] = oracle.TILE_UNMASKED
    want[(dlt < 0) | (dlt >= w // 128 + 1)] = oracle.TILE_SKIP
    np.testing.assert_array_equal(cls, want)
    assert visible == sum(min(i + 1, w) for i in range(N))


def test_tilemap_empty_mask_all_unmasked():
    cls, visible = oracle.tilemap(300, None, False)
    assert (cls == oracle.TILE_UNMASKED).all() and visible == 300 * 300


def test_count_closed_forms():
    N = 1000
    assert oracle.count_unmasked(N, None, True) == N * (N + 1) // 2
    P = 256
    m = W.prefix_lm(N, P)
    assert oracle.count_unmasked(N, m.slice(0), m.causal) == P * N + sum(N - j for j in range(P, N))
    g, w = 64, 100
    m = W.global_sliding(N, g, w)
    want = sum(N - j for j in range(g)) + sum(min(w, N - j) for j in range(g, N))
    assert oracle.count_unmasked(N, m.slice(0), m.causal) == want


# ---------------------------------------------------------- attention sink
def _torch_sink_reference(q, k, v, do, mask, causal, scale, sink):
    """The sink as one more key column whose logit is `sink` and whose value is
    zero, through fp64 torch softmax and autograd (independent of the oracle)."""
    import torch
    N = q.shape[0]
    dense = torch.from_numpy(oracle.tilemap(N, mask, causal, tq=1, tk=1)[0] == oracle.TILE_SKIP)
    qt, kt, vt = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
    st = torch.tensor(sink, dtype=torch.float64, requires_grad=True)
    s = (qt @ kt.T) * scale
    s = s.masked_fill(dense, float("-inf"))
    logits = torch.cat([s, st.expand(N, 1)], dim=1)
    p = torch.softmax(logits, dim=1)
    o = p[:, :N] @ vt
    lse = torch.logsumexp(logits, dim=1)
    o.backward(torch.from_numpy(do))
    return (o.detach().numpy(), lse.detach().numpy(), qt.grad.numpy(), kt.grad.numpy(),
            vt.grad.numpy(), float(st.grad))


@pytest.mark.parametrize("sink", [-2.0, 0.5, 3.0])
def test_sink_is_an_extra_zero_value_key(sink):
    rng = np.random.default_rng(21)
    N, d = 96, 16
    q, k, v, do = (rng.standard_normal((N, d)) for _ in range(4))
    mask = W.causal_document(N, [W.uniform_lengths(rng, 10, 40, N)]).slice(0)
    scale = 1 / np.sqrt(d)
    o, lse = oracle.attention_fwd(q, k, v, mask, True, scale, sink=sink)
    dq, dk, dv, ds = oracle.attention_bwd(q, k, v, do, mask, True, scale, sink=sink)
    ro, rl, rdq, rdk, rdv, rds = _torch_sink_reference(q, k, v, do, mask, True, scale, sink)
    for got, ref in ((o, ro), (lse, rl), (dq, rdq), (dk, rdk), (dv, rdv)):
        np.testing.assert_allclose(got, ref, atol=1e-12, rtol=1e-12)
    assert abs(ds - rds) <= 1e-12 * max(1.0, abs(rds))


def test_sink_limits():
    """A vanishing sink is no sink; a row whose keys are all masked gives O = 0,
    LSE = sink and adds nothing to the sink's gradient."""
    rng = np.random.default_rng(22)
    N, d = 64, 8
    q, k, v, do = (rng.standard_normal((N, d)) for _ in range(4))
    mask = {"lts": np.full(N, 20, np.int32), "lte": np.full(N, 30, np.int32)}
    o0, l0 = oracle.attention_fwd(q, k, v, mask, False)
    o1, l1 = oracle.attention_fwd(q, k, v, mask, False, sink=-1e4)
    np.testing.assert_allclose(o1, o0, atol=1e-15)
    np.testing.assert_allclose(l1[np.isfinite(l0)], l0[np.isfinite(l0)], atol=1e-15)
    o2, l2 = oracle.attention_fwd(q, k, v, mask, False, sink=1.25)
    assert (o2[20:30] == 0).all() and np.allclose(l2[20:30], 1.25)
    _, _, terms = oracle.attention_bwd_dq(q, k, v, do, mask, False, sink=1.25, with_dsink=True)
    assert (terms[20:30] == 0).all() and (terms[:20] != 0).all()
