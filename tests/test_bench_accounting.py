"""FLOP accounting and workload overrides of bench.py (CPU only).

The per-kernel credits must add up to the step's algorithmic FLOPs per
unmasked pair: 2(d + dv) forward, 2(3d + 2dv) backward (S recomputation, dP,
dV, dK, dQ), 8d + 6dv together.
"""
import os
import sys
import types

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402

HEADS = [(64, 64), (128, 128), (192, 128), (256, 256)]


@pytest.mark.parametrize("d,dv", HEADS)
def test_step_flops_per_pair(d, dv):
    f = bench.flops_per_pair(d, dv)
    # forward: S = Q K^T (2d per pair) and O = P V (2dv per pair)
    assert f["fwd"] == 2 * d + 2 * dv
    # backward: S again, dP = dO V^T, dV = P^T dO, dK = dS^T Q, dQ = dS K
    assert f["bwd"] == 2 * d + 2 * dv + 2 * dv + 2 * d + 2 * d
    assert f["fwd+bwd"] == f["fwd"] + f["bwd"]


@pytest.mark.parametrize("d,dv", HEADS)
@pytest.mark.parametrize("det", [False, True])
def test_kernel_credits_add_up(d, dv, det):
    credit = lambda n: bench.kernel_alg_flops_per_pair(n, d, dv)  # noqa: E731
    f = bench.flops_per_pair(d, dv)
    fwd_names, bwd_names = bench.kernel_names(d, dv, det)
    assert sum(credit(n) for n in fwd_names) == f["fwd"]
    assert sum(credit(n) for n in bwd_names) == f["bwd"]
    # every form of the backward is credited with the same products
    assert credit("bwd_dkdv_dv") + credit("bwd_split_dk") == credit("bwd_split")
    assert credit("bwd_dkdvq") == credit("bwd_split")


def test_kernel_names_follow_the_backward_variant():
    for d, dv in HEADS:
        for det in (False, True):
            _, bwd = bench.kernel_names(d, dv, det)
            fused = not det and d == dv and d <= 128
            assert bwd[0] == "bwd_preprocess"
            if fused:
                assert bwd[1:] == ["bwd_dkdvq", "bwd_dq_convert"]
            elif d == 256 and dv == 256:
                assert bwd[1:] == ["bwd_dkdv_dv", "bwd_split_dk"]
            else:
                assert bwd[1:] == ["bwd_split"]


def test_workload_overrides():
    args = types.SimpleNamespace(workload="large_head_d192", N=None, B=None, H=None,
                                 deterministic=None)
    base = bench.workload_cfg(args)
    assert base["deterministic"] is True
    args.deterministic = 0
    args.N, args.H = 4096, 2
    cfg = bench.workload_cfg(args)
    assert cfg["deterministic"] is False and cfg["N"] == 4096 and cfg["H"] == 2
    assert cfg["d"] == base["d"] and cfg["B"] == base["B"]


def test_code_hash_ignores_comments_only(tmp_path):
    base = ('// header\n#include <x.h>\n/* block\n comment */\nint f(int a) {  // tail\n'
            '    const char *s = "// not a comment /* either */";\n    return a + 1;\n}\n')
    p = tmp_path / "k.cu"
    p.write_text(base)
    h0 = bench.code_hash(str(p))
    p.write_text(base.replace("// header", "// another header\n\n// more")
                     .replace("/* block\n comment */", "/* changed */"))
    assert bench.code_hash(str(p)) == h0
    p.write_text(base.replace('"// not a comment /* either */"', '"// not a comment"'))
    assert bench.code_hash(str(p)) != h0  # string literals are code
    p.write_text(base.replace("a + 1", "a + 2"))
    assert bench.code_hash(str(p)) != h0
