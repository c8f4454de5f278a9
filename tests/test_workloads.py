"""The mask generators encode each family's semantics exactly.

The dense expansion of the generated vectors (the oracle's 1x1 tile map) must
equal the family's semantic predicate, built from the drawn structure.
"""
import numpy as np
import pytest

import oracle
from sparse_masked_attention_gb300 import workloads as W


@pytest.mark.parametrize("name", sorted(W.CONFIGS))
def test_config_mask_matches_semantics(name):
    cfg = W.CONFIGS[name]
    N = min(cfg["N"], 3000)
    mask = W.make_mask(cfg, seed=0, N=N, B=min(cfg["B"], 2))
    for b in range(len(mask.meta)):
        cls, visible = oracle.tilemap(N, mask.slice(b), mask.causal, tq=1, tk=1)
        sem = W.dense_semantic(mask, b)
        np.testing.assert_array_equal(cls == oracle.TILE_SKIP, sem)
        assert not sem.all(axis=1).any()


def test_three_documents_partition():
    rng = np.random.default_rng(0)
    lens = W.three_documents(rng, 256)
    assert len(lens) == 3 and sum(lens) == 256 and min(lens) >= 1


def test_uniform_lengths_cover_exactly():
    rng = np.random.default_rng(0)
    lens = W.uniform_lengths(rng, 512, 4096, 8192)
    assert sum(lens) == 8192 and all(1 <= x <= 4096 for x in lens)
    assert all(x >= 512 for x in lens[:-1])


def test_block_sparse_fraction_near_target():
    N = 128 * 64
    mask = W.block_sparse(N, np.random.default_rng(0))
    runs = mask.meta[0]["runs"]
    masked = sum((r1[1] - r1[0]) + (r2[1] - r2[0]) for r1, r2 in runs)
    cand = sum(64 - 1 - kb for kb in range(64))
    assert abs(masked / cand - 0.3) < 0.02
    # the diagonal block is never masked
    for kb, (r1, r2) in enumerate(runs):
        assert r1[0] > kb or r1[0] == r1[1]
        assert r2[0] > kb or r2[0] == r2[1]


def test_inputs_are_seeded():
    a = W.make_inputs(1, 16, 2, 8, 8, seed=3)
    b = W.make_inputs(1, 16, 2, 8, 8, seed=3)
    for x, y in zip(a, b):
        assert x.dtype.is_floating_point and x.shape[-1] == 8
        assert bool((x == y).all())


def _dense(mask, b=0):
    cls, _ = oracle.tilemap(mask.N, mask.slice(b), mask.causal, tq=1, tk=1)
    return cls == oracle.TILE_SKIP


def test_prefix_document_reduces_to_its_limits():
    """No prefix: causal documents; a prefix as long as the document: plain
    bidirectional documents."""
    rng = np.random.default_rng(3)
    N = 700
    lengths = W.uniform_lengths(rng, 40, 200, N)
    none = W.prefix_document(N, [lengths], [[0] * len(lengths)])
    whole = W.prefix_document(N, [lengths], [list(lengths)])
    np.testing.assert_array_equal(_dense(none), _dense(W.causal_document(N, [lengths])))
    np.testing.assert_array_equal(_dense(whole), _dense(W.document(N, [lengths])))


def test_document_is_block_diagonal_and_symmetric():
    rng = np.random.default_rng(4)
    N = 500
    lengths = W.uniform_lengths(rng, 30, 150, N)
    m = _dense(W.document(N, [lengths]))
    np.testing.assert_array_equal(m, m.T)
    ends = np.cumsum(lengths)
    starts = ends - np.asarray(lengths)
    for s0, e0 in zip(starts, ends):
        assert not m[s0:e0, s0:e0].any()
        assert m[s0:e0, :s0].all() and m[s0:e0, e0:].all()


def test_bidirectional_window_limits():
    N = 300
    assert not _dense(W.bidirectional_window(N, N)).any()          # window covers all: no mask
    one = _dense(W.bidirectional_window(N, 1))                      # only the diagonal
    np.testing.assert_array_equal(~one, np.eye(N, dtype=bool))
    m = _dense(W.bidirectional_window(N, 37))
    np.testing.assert_array_equal(m, m.T)
    assert (~m).sum(axis=1).max() == 2 * 37 - 1


def test_random_eviction_limits():
    """Keys never evicted give plain causal attention; every row keeps its
    diagonal, and the causal part is always masked."""
    N = 400
    kept = _dense(W.random_eviction(N, np.random.default_rng(5), keep=1.0))
    np.testing.assert_array_equal(kept, _dense(W.causal(N)))
    m = _dense(W.random_eviction(N, np.random.default_rng(6)))
    assert not np.diag(m).any()
    assert m[np.triu(np.ones((N, N), bool), 1)].all()
    assert m.sum() > kept.sum()  # some keys were evicted


# The benchmarked shapes, as the workload definitions state them: batch, heads,
# sequence length, head dims, passes, and the mask's own parameters.
STATED = {
    "tiny_causal_document": dict(B=1, H=2, N=256, d=64, dv=64, passes="fwd+bwd"),
    "std_causal": dict(B=1, H=32, N=8192, d=128, dv=128, passes="fwd"),
    "std_sliding": dict(B=1, H=32, N=8192, d=128, dv=128, passes="fwd", w=1024),
    "std_causal_document": dict(B=1, H=32, N=8192, d=128, dv=128, passes="fwd",
                                doc_len=(512, 4096)),
    "std_prefix_lm": dict(B=1, H=32, N=8192, d=128, dv=128, passes="fwd", prefix=2048),
    "share_question": dict(B=2, H=16, N=32768, d=128, dv=128, passes="fwd+bwd"),
    "long_block_sparse": dict(B=1, H=8, N=131072, d=128, dv=128, passes="fwd+bwd"),
    "long_global_sliding": dict(B=1, H=8, N=131072, d=128, dv=128, passes="fwd+bwd",
                                n_global=512, w=4096),
    "large_head_d192": dict(B=1, H=16, N=16384, d=192, dv=128, passes="fwd+bwd",
                            doc_len=(1024, 8192), deterministic=True),
    "large_head_d256": dict(B=1, H=16, N=16384, d=256, dv=256, passes="fwd+bwd",
                            doc_len=(1024, 8192), deterministic=True),
}


@pytest.mark.parametrize("name", sorted(STATED))
def test_benchmarked_shapes_are_the_stated_ones(name):
    cfg = W.CONFIGS[name]
    for key, want in STATED[name].items():
        assert cfg[key] == want, (name, key)
