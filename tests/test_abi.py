"""The C-ABI library loads and exports what include/lrm.h declares (no GPU).

Only host-side paths are exercised: the pure workspace query, the status
strings and argument validation that returns before any launch.
"""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "lrm.h")


def _declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(lrm_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    from demand_side_expert_gb300 import build as b

    if not os.path.exists(b.LIB):
        b.build()
    from demand_side_expert_gb300 import lrm

    return lrm


def test_every_declared_symbol_is_exported(lib):
    declared = _declared_functions()
    assert declared, "no declarations parsed"
    raw = ctypes.CDLL(lib.library_path())
    for name in declared:
        assert hasattr(raw, name), f"{name} missing from liblrm.so"
    assert sorted(lib.EXPORTS) == declared


def _declared_params():
    src = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    out = {}
    for m in re.finditer(r"\b(lrm_[a-z0-9_]+)\s*\(([^)]*)\)\s*;", src):
        params = [p.strip() for p in m.group(2).split(",") if p.strip()]
        out[m.group(1)] = [] if params == ["void"] else params
    return out


def test_binding_signatures_match_the_header(lib):
    """Every ctypes argtypes list has the header's arity and argument kinds."""
    decl = _declared_params()
    assert sorted(decl) == sorted(lib.EXPORTS)
    for name, params in decl.items():
        argtypes = getattr(lib._lib, name).argtypes
        assert len(argtypes) == len(params), (name, len(argtypes), len(params))
        for p, a in zip(params, argtypes):
            if "*" in p:
                assert a is ctypes.c_void_p or hasattr(a, "_type_") and a.__name__.startswith(
                    "LP_"), (name, p, a)
            elif p.startswith("size_t"):
                assert a is ctypes.c_size_t, (name, p, a)
            elif p.startswith("uint64_t"):
                assert a is ctypes.c_uint64, (name, p, a)
            elif p.startswith("int64_t"):
                assert a is ctypes.c_int64, (name, p, a)
            else:
                assert a is ctypes.c_int32, (name, p, a)


def test_workspace_query_is_pure_host(lib):
    s = lib.make_shape(4096, 2048, 768, 128, 8, lib.LRM_BF16)
    b = lib.lrm_workspace_bytes(s)
    assert b >= 256 and b % 256 == 0
    bad = lib.make_shape(4096, 2048, 768, 128, 0, lib.LRM_BF16)
    assert lib.lrm_workspace_bytes(bad) == 0
    odd = lib.make_shape(16, 30, 16, 4, 2, lib.LRM_F32)  # D not a multiple of 8
    assert lib.lrm_workspace_bytes(odd) == 0


def test_status_strings(lib):
    assert lib.status_string(0) == "LRM_OK"
    assert lib.status_string(lib.LRM_ERR_WORKSPACE) == "LRM_ERR_WORKSPACE"


def test_argument_errors_return_before_launch(lib):
    raw = lib._lib
    s = lib.make_shape(64, 32, 16, 8, 2, lib.LRM_F32)
    # no workspace
    assert raw.lrm_dispatch_permute(ctypes.byref(s), 8, 8, 8, 8, 8, None, 0, None) == \
        lib.LRM_ERR_WORKSPACE
    # null shape
    assert raw.lrm_score(None, 16, 16, 16, 16, 16, 256, 4096, None) == lib.LRM_ERR_INVALID_ARG
    # bad rate
    assert raw.lrm_quota_from_rate(16, 8, 3, 2, 0, 16, None) == lib.LRM_ERR_INVALID_ARG
    # row bytes not a multiple of 16
    assert raw.lrm_permute_rows(16, 4, 16, 32, 24, None) == lib.LRM_ERR_INVALID_ARG
    # misaligned activation pointer (checked before launch)
    ws = 256 * 1024
    assert raw.lrm_score(ctypes.byref(s), 18, 16, 16, 16, 16, ws, 1 << 20, None) == \
        lib.LRM_ERR_UNSUPPORTED
    # K too large for the backward's gather
    big = lib.make_shape(64, 64, 64, 64, 40, lib.LRM_BF16)
    args = [ctypes.byref(big)] + [256] * 16 + [ws, 1 << 24, None]
    assert raw.lrm_expert_bwd_grouped(*args) == lib.LRM_ERR_UNSUPPORTED
