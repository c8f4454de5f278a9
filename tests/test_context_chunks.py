"""Mask localization for context-parallel chunks, pinned on the CPU.

The local vectors of every (query chunk, key chunk) pair must describe
exactly the block of the global mask the pair covers (brute force: the dense
expansion of the global vectors, sliced), and the fp64 attention of a query
chunk rebuilt from its pairs by the log-sum-exp merge must equal the
attention of the whole sequence.
"""
import numpy as np
import pytest

import oracle
from sparse_masked_attention_gb300 import workloads as W


def _dense(N, ms, causal):
    cls, _ = oracle.tilemap(N, ms, causal, tq=1, tk=1)
    return cls == oracle.TILE_SKIP


def _masks(N, seed):
    rng = np.random.default_rng(seed)
    yield W.causal(N)
    yield W.full(N)
    yield W.sliding_window(N, 90)
    yield W.causal_document(N, [W.uniform_lengths(rng, 30, 200, N)])
    yield W.document(N, [W.uniform_lengths(rng, 30, 200, N)])
    yield W.prefix_lm(N, 150)
    yield W.share_question(N, [W.share_question_groups(rng, N, (60, 150), (2, 3), (20, 80))])
    yield W.block_sparse(N, rng, blk=32)
    yield W.bidirectional_window(N, 70)
    yield W.random_eviction(N, rng)
    yield W.random_vectors(N, rng, causal_flag=True)
    yield W.random_vectors(N, rng, causal_flag=False)


@pytest.mark.parametrize("chunks", [2, 3, 4])
def test_local_vectors_cover_the_global_block(chunks):
    N = 480
    L = N // chunks
    for mask in _masks(N, seed=chunks):
        ms = mask.slice(0)
        full = _dense(N, ms, mask.causal)
        for qc in range(chunks):
            for kc in range(chunks):
                q0, k0 = qc * L, kc * L
                block = full[q0:q0 + L, k0:k0 + L]
                local, lc = oracle.localize(ms, N, mask.causal, q0, k0, L)
                if local is None:
                    assert block.all(), (mask.family, qc, kc)
                    continue
                np.testing.assert_array_equal(_dense(L, local, lc), block,
                                              err_msg=f"{mask.family} {qc} {kc}")


def _lse_merge(parts, L, dv):
    """Plain log-sum-exp merge of partial (O, LSE) over the key chunks."""
    o = np.zeros((L, dv))
    lse = np.full(L, -np.inf)
    for po, pl in parts:
        new = np.logaddexp(lse, pl)
        wa = np.where(np.isneginf(new), 0.0, np.exp(lse - np.where(np.isneginf(new), 0, new)))
        wb = np.where(np.isneginf(new), 0.0, np.exp(pl - np.where(np.isneginf(new), 0, new)))
        o = o * wa[:, None] + po * wb[:, None]
        lse = new
    return o, lse


@pytest.mark.parametrize("family", ["causal_document", "share_question", "block_sparse",
                                    "random"])
def test_chunked_attention_equals_whole(family):
    N, C, d = 384, 4, 32
    L = N // C
    rng = np.random.default_rng(7)
    mask = {
        "causal_document": lambda: W.causal_document(N, [W.uniform_lengths(rng, 40, 150, N)]),
        "share_question": lambda: W.share_question(
            N, [W.share_question_groups(rng, N, (50, 120), (2, 3), (20, 60))]),
        "block_sparse": lambda: W.block_sparse(N, rng, blk=32),
        "random": lambda: W.random_vectors(N, rng, causal_flag=True),
    }[family]()
    ms = mask.slice(0)
    q, k, v = (rng.standard_normal((N, d)) for _ in range(3))
    scale = 1 / np.sqrt(d)
    o_ref, lse_ref = oracle.attention_fwd(q, k, v, ms, mask.causal, scale)
    for qc in range(C):
        q0 = qc * L
        parts = []
        for kc in range(C):
            k0 = kc * L
            local, lc = oracle.localize(ms, N, mask.causal, q0, k0, L)
            if local is None:
                continue
            parts.append(oracle.attention_fwd(q[q0:q0 + L], k[k0:k0 + L], v[k0:k0 + L], local,
                                              lc, scale))
        o, lse = _lse_merge(parts, L, d)
        np.testing.assert_allclose(o, o_ref[q0:q0 + L], atol=1e-12)
        fin = np.isfinite(lse_ref[q0:q0 + L])
        np.testing.assert_allclose(lse[fin], lse_ref[q0:q0 + L][fin], atol=1e-12)
        assert np.array_equal(np.isneginf(lse), np.isneginf(lse_ref[q0:q0 + L]))
