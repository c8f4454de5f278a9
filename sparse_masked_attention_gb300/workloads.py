"""Seeded synthetic workloads: attention inputs and column-wise mask vectors.

This module generates inputs only.  It holds none of the attention
arithmetic, and it serves the CUDA path and the CPU oracle alike.

Mask families are those named in the FlashMask-3 abstract: document,
prefix-LM, share-question, sliding-window and block-sparse, plus causal and
global+sliding.  Further structured variants of the same kind widen the set:
bidirectional documents, documents with a bidirectional prefix each, a
symmetric (bidirectional) sliding window, and causal attention with random
key eviction.  Each family is first drawn as a structure, such as document
lengths or a window width.  That structure is then encoded in the column-wise
form of the FlashMask README "Overview".  Key column ``j`` gets query-row
intervals ``[LTS_j, LTE_j)`` and ``[UTS_j, UTE_j)``.  Row ``i`` is masked
when it lies in either interval, and the ``causal`` flag also masks ``i < j``.

An empty lower interval is stored as ``LTS = LTE = N``.  An empty upper
interval is stored as ``UTS = UTE = 0``.  Vectors are int32 with shape
``[B, 1, N]``: each sample has its own mask, shared by all heads.

``dense_semantic`` rebuilds a small mask densely from the drawn structure,
never from the vectors.  Tests use it to check the encoding.

Input tensors are drawn with ``torch.Generator(device).manual_seed(seed)`` in
the order q, k, v, dO.  Each is ``randn`` in fp32 with the BNHD shape, then
cast to bf16.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import numpy as np

# --------------------------------------------------------------- structures


@dataclass
class Mask:
    """Column-wise mask of a batch: vectors [B, 1, N] (None = interval absent)."""
    N: int
    causal: bool
    lts: Optional[np.ndarray] = None
    lte: Optional[np.ndarray] = None
    uts: Optional[np.ndarray] = None
    ute: Optional[np.ndarray] = None
    family: str = ""
    meta: list = field(default_factory=list)  # per-sample drawn structure

    def slice(self, b: int, hm: int = 0) -> dict:
        """Vectors of one (sample, mask-head) as a dict of [N] int32 arrays."""
        out = {}
        for name in ("lts", "lte", "uts", "ute"):
            x = getattr(self, name)
            out[name] = None if x is None else np.ascontiguousarray(x[b, hm])
        return out


def uniform_lengths(rng: np.random.Generator, lo: int, hi: int, N: int) -> list:
    """Integer lengths ~ U[lo, hi] drawn until they cover N; the last one is cut."""
    out, tot = [], 0
    while tot < N:
        x = int(rng.integers(lo, hi + 1))
        x = min(x, N - tot)
        out.append(x)
        tot += x
    return out


def three_documents(rng: np.random.Generator, N: int) -> list:
    """Two distinct cut points uniform in {1..N-1}, sorted: three documents."""
    cuts = np.sort(rng.choice(np.arange(1, N), size=2, replace=False))
    return [int(cuts[0]), int(cuts[1] - cuts[0]), int(N - cuts[1])]


# ------------------------------------------------------------ mask families


def causal(N: int, B: int = 1) -> Mask:
    return Mask(N, True, family="causal", meta=[{} for _ in range(B)])


def full(N: int, B: int = 1) -> Mask:
    """No mask at all (dense bidirectional attention)."""
    return Mask(N, False, family="full", meta=[{} for _ in range(B)])


def sliding_window(N: int, w: int, B: int = 1) -> Mask:
    """Causal window of w keys, self included: row i sees keys i-w+1 .. i."""
    j = np.arange(N, dtype=np.int64)
    lts = np.minimum(j + w, N).astype(np.int32)
    lte = np.full(N, N, np.int32)
    rep = lambda x: np.repeat(x[None, None], B, axis=0)
    return Mask(N, True, lts=rep(lts), lte=rep(lte), family="sliding",
                meta=[{"w": w} for _ in range(B)])


def _doc_lower(N, lengths):
    ends = np.cumsum(lengths)
    doc_end = np.repeat(ends, lengths).astype(np.int32)
    return doc_end, np.full(N, N, np.int32)


def causal_document(N: int, lengths_per_sample: list) -> Mask:
    """Causal within a document, nothing across documents."""
    B = len(lengths_per_sample)
    lts = np.zeros((B, 1, N), np.int32)
    lte = np.zeros((B, 1, N), np.int32)
    for b, lengths in enumerate(lengths_per_sample):
        assert sum(lengths) == N
        lts[b, 0], lte[b, 0] = _doc_lower(N, lengths)
    return Mask(N, True, lts=lts, lte=lte, family="causal_document",
                meta=[{"lengths": list(map(int, x))} for x in lengths_per_sample])


def prefix_lm(N: int, prefix: int, B: int = 1) -> Mask:
    """Bidirectional prefix of `prefix` tokens, causal suffix (no causal flag)."""
    j = np.arange(N, dtype=np.int64)
    uts = np.zeros(N, np.int32)
    ute = np.where(j >= prefix, j, 0).astype(np.int32)
    rep = lambda x: np.repeat(x[None, None], B, axis=0)
    return Mask(N, False, uts=rep(uts), ute=rep(ute), family="prefix_lm",
                meta=[{"prefix": prefix} for _ in range(B)])


def _doc_bounds(N, lengths):
    ends = np.cumsum(lengths)
    starts = ends - np.asarray(lengths)
    return (np.repeat(starts, lengths).astype(np.int32),
            np.repeat(ends, lengths).astype(np.int32))


def document(N: int, lengths_per_sample: list) -> Mask:
    """Bidirectional within a document, nothing across documents (no causal
    flag): column j is masked above its document's start and from its end."""
    B = len(lengths_per_sample)
    lts = np.zeros((B, 1, N), np.int32)
    lte = np.full((B, 1, N), N, np.int32)
    uts = np.zeros((B, 1, N), np.int32)
    ute = np.zeros((B, 1, N), np.int32)
    for b, lengths in enumerate(lengths_per_sample):
        assert sum(lengths) == N
        start, end = _doc_bounds(N, lengths)
        lts[b, 0], ute[b, 0] = end, start
    return Mask(N, False, lts=lts, lte=lte, uts=uts, ute=ute, family="document",
                meta=[{"lengths": list(map(int, x))} for x in lengths_per_sample])


def document_prefixes(rng: np.random.Generator, lengths: list) -> list:
    """A bidirectional prefix per document, its length ~ U{0 .. document length}."""
    return [int(rng.integers(0, n + 1)) for n in lengths]


def prefix_document(N: int, lengths_per_sample: list, prefixes_per_sample: list) -> Mask:
    """Documents with a bidirectional prefix each: inside a document every row
    sees the prefix keys, and the keys after the prefix causally; nothing
    across documents (no causal flag)."""
    B = len(lengths_per_sample)
    lts = np.zeros((B, 1, N), np.int32)
    lte = np.full((B, 1, N), N, np.int32)
    uts = np.zeros((B, 1, N), np.int32)
    ute = np.zeros((B, 1, N), np.int32)
    j = np.arange(N, dtype=np.int32)
    for b, (lengths, prefixes) in enumerate(zip(lengths_per_sample, prefixes_per_sample)):
        assert sum(lengths) == N and len(prefixes) == len(lengths)
        start, end = _doc_bounds(N, lengths)
        pref_end = np.repeat(np.cumsum(lengths) - np.asarray(lengths) + np.asarray(prefixes),
                             lengths).astype(np.int32)
        lts[b, 0] = end
        ute[b, 0] = np.where(j < pref_end, start, j)
    return Mask(N, False, lts=lts, lte=lte, uts=uts, ute=ute, family="prefix_document",
                meta=[{"lengths": list(map(int, x)), "prefixes": list(map(int, y))}
                      for x, y in zip(lengths_per_sample, prefixes_per_sample)])


def bidirectional_window(N: int, w: int, B: int = 1) -> Mask:
    """Symmetric local window (no causal flag): row i sees the keys j with
    |i - j| < w."""
    j = np.arange(N, dtype=np.int64)
    lts = np.minimum(j + w, N).astype(np.int32)
    lte = np.full(N, N, np.int32)
    uts = np.zeros(N, np.int32)
    ute = np.maximum(j - w + 1, 0).astype(np.int32)
    rep = lambda x: np.repeat(x[None, None], B, axis=0)
    return Mask(N, False, lts=rep(lts), lte=rep(lte), uts=rep(uts), ute=rep(ute),
                family="bidirectional_window", meta=[{"w": w} for _ in range(B)])


def eviction_rows(rng: np.random.Generator, N: int, keep: float = 0.5) -> np.ndarray:
    """Per key j the first row that no longer sees it: N (never evicted) with
    probability `keep`, otherwise ~ U{j+1 .. N}."""
    j = np.arange(N, dtype=np.int64)
    ev = j + 1 + np.floor(rng.random(N) * (N - j)).astype(np.int64)
    never = rng.random(N) < keep
    return np.where(never, N, np.minimum(ev, N)).astype(np.int32)


def random_eviction(N: int, rng: np.random.Generator, B: int = 1, keep: float = 0.5) -> Mask:
    """Causal, and key j is evicted from row e_j on (a key-value cache that
    drops keys at random times; the diagonal always stays visible)."""
    lts = np.zeros((B, 1, N), np.int32)
    lte = np.full((B, 1, N), N, np.int32)
    meta = []
    for b in range(B):
        ev = eviction_rows(rng, N, keep)
        lts[b, 0] = ev
        meta.append({"evict": ev})
    return Mask(N, True, lts=lts, lte=lte, family="random_eviction", meta=meta)


def share_question_groups(rng, N, q_len=(1024, 4096), n_ans=(2, 4), a_len=(512, 2048)):
    """Packed groups [question, answer_1 .. answer_k] until N; the last is cut."""
    groups, pos = [], 0
    while pos < N:
        parts = [int(rng.integers(q_len[0], q_len[1] + 1))]
        k = int(rng.integers(n_ans[0], n_ans[1] + 1))
        parts += [int(rng.integers(a_len[0], a_len[1] + 1)) for _ in range(k)]
        cut = []
        for p in parts:
            if pos >= N:
                break
            p = min(p, N - pos)
            cut.append(p)
            pos += p
        groups.append(cut)
    return groups


def share_question(N: int, groups_per_sample: list) -> Mask:
    """Answers see their own question and themselves (causally), never a sibling
    answer; groups are independent.  Causal flag on."""
    B = len(groups_per_sample)
    lts = np.zeros((B, 1, N), np.int32)
    lte = np.full((B, 1, N), N, np.int32)
    for b, groups in enumerate(groups_per_sample):
        pos = 0
        for parts in groups:
            g_end = pos + sum(parts)
            # question columns are visible up to the end of the group
            lts[b, 0, pos:pos + parts[0]] = g_end
            a = pos + parts[0]
            for p in parts[1:]:
                lts[b, 0, a:a + p] = a + p     # an answer is visible only inside itself
                a += p
            pos = g_end
        assert pos == N
    return Mask(N, True, lts=lts, lte=lte, family="share_question",
                meta=[{"groups": g} for g in groups_per_sample])


def block_sparse(N: int, rng: np.random.Generator, B: int = 1, frac: float = 0.3,
                 blk: int = 128) -> Mask:
    """Causal, plus per key block kb a random `frac` of the query blocks below the
    diagonal masked, as two non-overlapping runs (run 1 -> LT, run 2 -> UT)."""
    nB = -(-N // blk)
    lts = np.zeros((B, 1, N), np.int32)
    lte = np.zeros((B, 1, N), np.int32)
    uts = np.zeros((B, 1, N), np.int32)
    ute = np.zeros((B, 1, N), np.int32)
    meta = []
    for b in range(B):
        runs = []
        for kb in range(nB):
            c = nB - 1 - kb                      # candidate query blocks kb+1 .. nB-1
            m = int(round(frac * c))
            m1 = int(rng.integers(0, m + 1))
            m2 = m - m1
            free = c - m
            g1, g2 = np.sort(rng.integers(0, free + 1, size=2))
            s1 = int(g1)
            s2 = int(g2) + m1
            r1 = (kb + 1 + s1, kb + 1 + s1 + m1)  # in query blocks, half-open
            r2 = (kb + 1 + s2, kb + 1 + s2 + m2)
            runs.append((r1, r2))
            c0, c1 = kb * blk, min((kb + 1) * blk, N)
            to_rows = lambda r: (min(r[0] * blk, N), min(r[1] * blk, N))
            a, e = to_rows(r1) if m1 > 0 else (N, N)
            lts[b, 0, c0:c1], lte[b, 0, c0:c1] = a, e
            a, e = to_rows(r2) if m2 > 0 else (0, 0)
            uts[b, 0, c0:c1], ute[b, 0, c0:c1] = a, e
        meta.append({"blk": blk, "runs": runs})
    return Mask(N, True, lts=lts, lte=lte, uts=uts, ute=ute, family="block_sparse",
                meta=meta)


def global_sliding(N: int, n_global: int, w: int, B: int = 1) -> Mask:
    """Causal; the first n_global keys are seen by every later row, the other keys
    only inside a causal window of w keys."""
    j = np.arange(N, dtype=np.int64)
    lts = np.where(j < n_global, N, np.minimum(j + w, N)).astype(np.int32)
    lte = np.full(N, N, np.int32)
    rep = lambda x: np.repeat(x[None, None], B, axis=0)
    return Mask(N, True, lts=rep(lts), lte=rep(lte), family="global_sliding",
                meta=[{"n_global": n_global, "w": w} for _ in range(B)])


def random_vectors(N: int, rng: np.random.Generator, B: int = 1, Hm: int = 1,
                   causal_flag: bool = False, lo: int = -8, hi: Optional[int] = None) -> Mask:
    """Arbitrary int32 vectors, including inverted (empty), negative and
    out-of-range boundaries; no semantic structure."""
    hi = N + 8 if hi is None else hi
    shape = (B, Hm, N)
    v = [rng.integers(lo, hi + 1, size=shape).astype(np.int32) for _ in range(4)]
    return Mask(N, causal_flag, lts=v[0], lte=v[1], uts=v[2], ute=v[3], family="random",
                meta=[{} for _ in range(B)])


# ------------------------------------------------------------ dense semantic


def dense_semantic(mask: Mask, b: int = 0) -> np.ndarray:
    """bool [N, N], True = masked, built from the drawn structure (not from the
    vectors).  For small N only."""
    N, fam, meta = mask.N, mask.family, mask.meta[b]
    i = np.arange(N)[:, None]
    j = np.arange(N)[None, :]
    if fam == "full":
        return np.zeros((N, N), bool)
    if fam == "causal":
        return i < j
    if fam == "sliding":
        return (i < j) | (i - j >= meta["w"])
    if fam == "causal_document":
        doc = np.repeat(np.arange(len(meta["lengths"])), meta["lengths"])
        return (i < j) | (doc[:, None] != doc[None, :])
    if fam == "prefix_lm":
        P = meta["prefix"]
        return (j >= P) & (i < j)
    if fam == "share_question":
        grp = np.zeros(N, np.int64)
        seg = np.zeros(N, np.int64)        # 0 = question, k = k-th answer
        pos = 0
        for g, parts in enumerate(meta["groups"]):
            for s, p in enumerate(parts):
                grp[pos:pos + p] = g
                seg[pos:pos + p] = s
                pos += p
        same_group = grp[:, None] == grp[None, :]
        visible = same_group & ((seg[None, :] == 0) | (seg[:, None] == seg[None, :]))
        return (i < j) | ~visible
    if fam == "block_sparse":
        blk = meta["blk"]
        qb, kb = i // blk, j // blk
        m = i < j
        masked_blocks = np.zeros((-(-N // blk),) * 2, bool)
        for k_blk, (r1, r2) in enumerate(meta["runs"]):
            masked_blocks[r1[0]:r1[1], k_blk] = True
            masked_blocks[r2[0]:r2[1], k_blk] = True
        return m | masked_blocks[qb, kb]
    if fam == "global_sliding":
        g, w = meta["n_global"], meta["w"]
        return (i < j) | ((j >= g) & (i - j >= w))
    if fam == "document":
        doc = np.repeat(np.arange(len(meta["lengths"])), meta["lengths"])
        return doc[:, None] != doc[None, :]
    if fam == "prefix_document":
        lengths = meta["lengths"]
        doc = np.repeat(np.arange(len(lengths)), lengths)
        offset = np.arange(N) - np.repeat(np.cumsum(lengths) - np.asarray(lengths), lengths)
        in_prefix = offset < np.repeat(meta["prefixes"], lengths)
        return (doc[:, None] != doc[None, :]) | (~in_prefix[None, :] & (i < j))
    if fam == "bidirectional_window":
        return np.abs(i - j) >= meta["w"]
    if fam == "random_eviction":
        return (i < j) | (i >= np.asarray(meta["evict"])[None, :])
    raise ValueError(f"no semantic definition for family {fam!r}")


# ----------------------------------------------------------------- configs

#: Workloads: shapes, mask family and passes.  Seeds default to 0.
CONFIGS = {
    "tiny_causal_document": dict(B=1, H=2, N=256, d=64, dv=64, mask="three_documents",
                                 passes="fwd+bwd"),
    "std_causal": dict(B=1, H=32, N=8192, d=128, dv=128, mask="causal", passes="fwd"),
    "std_sliding": dict(B=1, H=32, N=8192, d=128, dv=128, mask="sliding", w=1024,
                        passes="fwd"),
    "std_causal_document": dict(B=1, H=32, N=8192, d=128, dv=128, mask="causal_document",
                                doc_len=(512, 4096), passes="fwd"),
    "std_prefix_lm": dict(B=1, H=32, N=8192, d=128, dv=128, mask="prefix_lm", prefix=2048,
                          passes="fwd"),
    "share_question": dict(B=2, H=16, N=32768, d=128, dv=128, mask="share_question",
                           passes="fwd+bwd"),
    "long_block_sparse": dict(B=1, H=8, N=131072, d=128, dv=128, mask="block_sparse",
                              passes="fwd+bwd"),
    "long_global_sliding": dict(B=1, H=8, N=131072, d=128, dv=128, mask="global_sliding",
                                n_global=512, w=4096, passes="fwd+bwd"),
    "std_document": dict(B=1, H=32, N=8192, d=128, dv=128, mask="document",
                         doc_len=(512, 4096), passes="fwd"),
    "std_prefix_document": dict(B=1, H=32, N=8192, d=128, dv=128, mask="prefix_document",
                                doc_len=(512, 4096), passes="fwd"),
    "std_bidirectional_window": dict(B=1, H=32, N=8192, d=128, dv=128,
                                     mask="bidirectional_window", w=1024, passes="fwd"),
    "std_random_eviction": dict(B=1, H=32, N=8192, d=128, dv=128, mask="random_eviction",
                                passes="fwd"),
    "large_head_d192": dict(B=1, H=16, N=16384, d=192, dv=128, mask="causal_document",
                            doc_len=(1024, 8192), passes="fwd+bwd", deterministic=True),
    "large_head_d256": dict(B=1, H=16, N=16384, d=256, dv=256, mask="causal_document",
                            doc_len=(1024, 8192), passes="fwd+bwd", deterministic=True),
}


def make_mask(cfg: dict, seed: int = 0, N: Optional[int] = None, B: Optional[int] = None) -> Mask:
    """Draw the mask of a workload (optionally at another N / B)."""
    N = cfg["N"] if N is None else N
    B = cfg["B"] if B is None else B
    rng = np.random.default_rng(seed)
    kind = cfg["mask"]
    if kind == "causal":
        return causal(N, B)
    if kind == "full":
        return full(N, B)
    if kind == "sliding":
        return sliding_window(N, cfg["w"], B)
    if kind == "three_documents":
        return causal_document(N, [three_documents(rng, N) for _ in range(B)])
    if kind == "causal_document":
        lo, hi = cfg["doc_len"]
        return causal_document(N, [uniform_lengths(rng, lo, hi, N) for _ in range(B)])
    if kind == "prefix_lm":
        return prefix_lm(N, cfg["prefix"], B)
    if kind == "share_question":
        return share_question(N, [share_question_groups(rng, N) for _ in range(B)])
    if kind == "block_sparse":
        return block_sparse(N, rng, B)
    if kind == "global_sliding":
        return global_sliding(N, cfg["n_global"], cfg["w"], B)
    if kind == "document":
        lo, hi = cfg["doc_len"]
        return document(N, [uniform_lengths(rng, lo, hi, N) for _ in range(B)])
    if kind == "prefix_document":
        lo, hi = cfg["doc_len"]
        lengths = [uniform_lengths(rng, lo, hi, N) for _ in range(B)]
        return prefix_document(N, lengths, [document_prefixes(rng, x) for x in lengths])
    if kind == "bidirectional_window":
        return bidirectional_window(N, cfg["w"], B)
    if kind == "random_eviction":
        return random_eviction(N, rng, B)
    raise ValueError(kind)


def make_inputs(B: int, N: int, H: int, d: int, dv: int, seed: int = 0,
                device="cpu", with_dout: bool = True):
    """q, k [B,N,H,d], v (and dO) [B,N,H,dv] in bf16, drawn in the order q, k, v, dO."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    mk = lambda c: torch.randn((B, N, H, c), generator=g, device=device,
                               dtype=torch.float32).to(torch.bfloat16)
    q, k, v = mk(d), mk(d), mk(dv)
    dout = mk(dv) if with_dout else None
    return q, k, v, dout
