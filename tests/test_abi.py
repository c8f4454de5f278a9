"""Host-side checks of the C ABI (no GPU needed).

The library loads and exports every function that include/flashmask.h
declares.  Its host-only logic answers without touching a device: workspace
sizing, status strings, and argument validation that fails before any CUDA
call.
"""
import ctypes
import os
import re

import pytest

from sparse_masked_attention_gb300 import binding as B
from sparse_masked_attention_gb300 import build as build_mod

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build_mod.build()
    return B.load()


def _declared():
    text = open(os.path.join(ROOT, "include", "flashmask.h")).read()
    return sorted(set(re.findall(r"\b(flashmask_\w+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert len(names) >= 7
    for n in names:
        assert hasattr(lib, n), f"{n} declared in flashmask.h but not exported"
    assert set(names) == set(B.EXPORTS)


def test_error_strings(lib):
    for s in range(7):
        assert B.flashmask_error_string(s) != "unknown status"
    assert "bounds" in B.flashmask_error_string(B.FM_ERR_DEVICE_BOUNDS)
    assert B.flashmask_error_string(99) == "unknown status"


def _prob(**kw):
    p = dict(B=1, H=2, Hm=1, N=1000, d=128, dv=128, scale=0.0, causal=1)
    p.update(kw)
    return B.fm_problem(**p)


def test_workspace_size_host_only(lib):
    fwd = B.flashmask_workspace_size(_prob(), None, 0)
    bwd = B.flashmask_workspace_size(_prob(), None, 1)
    T = 8
    # normalised vectors + tile map + two lists + counts, each 256-byte aligned
    assert fwd >= 1024 * 16 + T * T + 2 * T * T * 4 + 2 * T * 4
    assert bwd >= fwd + 2 * 2 * 1024 * 4
    assert fwd % 256 == 0 and bwd % 256 == 0


@pytest.mark.parametrize("kw", [dict(N=0), dict(B=0), dict(Hm=3), dict(causal=2),
                                dict(d=96, dv=96), dict(d=128, dv=64), dict(scale=float("nan"))])
def test_invalid_problems_have_no_workspace(lib, kw):
    assert B.flashmask_workspace_size(_prob(**kw), None, 0) == 0


def test_invalid_args_rejected_before_cuda(lib):
    p = _prob()
    st = B.flashmask_fwd(p, None, None, None, None, None, None, None, None, None, None, None, 0,
                         None)
    assert st == B.FM_ERR_INVALID_ARG
    # misaligned pointer
    st = B.flashmask_fwd(p, None, 8, 16, 16, None, None, None, None, 16, 16, 256, 1 << 20, None)
    assert st == B.FM_ERR_INVALID_ARG
    st = B.flashmask_bwd(p, None, *([None] * 14), 0, None)
    assert st == B.FM_ERR_INVALID_ARG
    # unsupported head dims, all pointers plausible
    p2 = _prob(d=96, dv=96)
    st = B.flashmask_fwd(p2, None, 256, 256, 256, None, None, None, None, 256, 256, 256, 1 << 30,
                         None)
    assert st == B.FM_ERR_UNSUPPORTED
    # half-given interval pair
    st = B.flashmask_fwd(p, None, 256, 256, 256, 256, None, None, None, 256, 256, 256, 1 << 30,
                         None)
    assert st == B.FM_ERR_INVALID_ARG
    # workspace too small
    st = B.flashmask_fwd(p, None, 256, 256, 256, None, None, None, None, 256, 256, 256, 16, None)
    assert st == B.FM_ERR_WORKSPACE
    # debug_bounds is a flag: 0 or 1
    opt = B.fm_options(0, 2, 0, None, 0)
    st = B.flashmask_fwd(p, opt, 256, 256, 256, None, None, None, None, 256, 256, 256, 1 << 30,
                         None)
    assert st == B.FM_ERR_INVALID_ARG


def test_debug_bounds_is_a_flag(lib):
    p = _prob()
    base = B.flashmask_workspace_size(p, None, 1)
    assert B.flashmask_workspace_size(p, B.fm_options(0, 1, 0, None, 0), 1) == base
    assert B.flashmask_workspace_size(p, B.fm_options(0, 2, 0, None, 0), 1) == 0
    assert B.flashmask_workspace_size(p, B.fm_options(0, -1, 0, None, 0), 1) == 0


def test_chunk_entry_points_reject_bad_arguments_before_cuda(lib):
    p = _prob(N=1024)
    out = [256, 512, 768, 1024]
    # chunk length 0, chunks that overrun N, chunks not on a common grid
    for q0, k0, ln in ((0, 0, 0), (900, 0, 256), (0, 100, 256), (-256, 0, 256)):
        st, _ = B.flashmask_localize(p, None, None, None, None, q0, k0, ln, *out, None)
        assert st == B.FM_ERR_INVALID_ARG, (q0, k0, ln)
    st, _ = B.flashmask_localize(p, 256, None, None, None, 0, 0, 256, *out, None)  # half pair
    assert st == B.FM_ERR_INVALID_ARG
    # a causal key chunk after the query chunk: skipped, nothing enqueued
    st, flag = B.flashmask_localize(_prob(N=1024, causal=1), None, None, None, None, 0, 256, 256,
                                    *out, None)
    assert st == B.FM_OK and flag == -1
    assert B.flashmask_merge_init(0, 2, 64, 256, 512, None) == B.FM_ERR_INVALID_ARG
    assert B.flashmask_merge(16, 2, 12, 256, 512, 768, 1024, None) == B.FM_ERR_INVALID_ARG
    assert B.flashmask_merge(16, 2, 64, 8, 512, 768, 1024, None) == B.FM_ERR_INVALID_ARG
    assert B.flashmask_merge_finish(16, 2, 64, 256, 512, 768, 1024, 8, None) == \
        B.FM_ERR_INVALID_ARG  # LSE row stride below the chunk length
    assert B.flashmask_accumulate(12, 256, 512, None) == B.FM_ERR_INVALID_ARG
    assert B.flashmask_to_bf16(16, 8, 512, None) == B.FM_ERR_INVALID_ARG
    assert B.flashmask_accumulate(0, 256, 512, None) == B.FM_OK  # nothing to do


def test_sink_gradient_needs_its_logits(lib):
    opt = B.fm_options(0, 0, 0, None, 0, None, 256)
    assert B.flashmask_workspace_size(_prob(), opt, 1) == 0


def test_selftest_wait_limits_checked_before_cuda(lib):
    assert B.flashmask_selftest_wait(0, None) == B.FM_ERR_INVALID_ARG
    assert B.flashmask_selftest_wait(10_000_000_001, None) == B.FM_ERR_INVALID_ARG


def _header_struct(name):
    """Field names and C types of `typedef struct { ... } name;` in flashmask.h."""
    import re
    text = open(os.path.join(ROOT, "include", "flashmask.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    m = re.search(r"typedef struct\s*\{([^{}]*)\}\s*" + name + r"\s*;", text)
    assert m, name
    fields = []
    for decl in m.group(1).split(";"):
        decl = " ".join(decl.split())
        if not decl:
            continue
        ctype, names = re.match(r"((?:const )?(?:unsigned long long|[a-z_]+)\s*\**)\s*(.*)",
                                decl).groups()
        for n in names.split(","):
            n = n.strip()
            stars = n.count("*")
            fields.append((n.lstrip("*").strip(), ctype.replace(" ", "") + "*" * stars))
    return fields


_C_SIZES = {"int": 4, "float": 4, "unsignedlonglong": 8}


@pytest.mark.parametrize("name", ["fm_problem", "fm_options"])
def test_ctypes_structs_match_the_header(name):
    import ctypes
    fields = _header_struct(name)
    cls = getattr(B, name)
    assert [f[0] for f in fields] == [f[0] for f in cls._fields_]
    for (fname, ctype), (pname, ptype) in zip(fields, cls._fields_):
        size = 8 if ctype.endswith("*") else _C_SIZES[ctype.replace("const", "")]
        assert ctypes.sizeof(ptype) == size, (fname, ctype, ptype)


def _header_functions():
    """Parameter counts of the functions flashmask.h declares."""
    text = open(os.path.join(ROOT, "include", "flashmask.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    out = {}
    for m in re.finditer(r"\b(flashmask_[a-z0-9_]+)\s*\(([^;{]*?)\)\s*;", text):
        params = " ".join(m.group(2).split())
        out[m.group(1)] = 0 if params in ("", "void") else params.count(",") + 1
    return out


def test_ctypes_signatures_match_the_header(lib):
    decl = _header_functions()
    assert set(decl) == set(B.EXPORTS)
    for name, n in decl.items():
        assert len(getattr(lib, name).argtypes) == n, name
