"""C-ABI checks that need no GPU: the library loads, exports every function
declared in include/dattn.h, and rejects invalid arguments on the host before
any CUDA call (fake pointers are never dereferenced)."""
from __future__ import annotations

import ctypes
import os
import re

import pytest

from token_decode_attention_gb300 import _native, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dattn.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _native.load()


def declared_functions():
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dattn_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("dattn_decode_f16", "dattn_decode_f16_ex", "dattn_qk_f16", "dattn_pv_f16",
                     "dattn_decode_workspace_bytes", "dattn_status_string", "dattn_last_error"):
        assert required in names


def test_library_exports_every_declared_function(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in dattn.h but not exported"


def test_version_and_status_strings(lib):
    assert lib.dattn_version() >= 10000
    for code, name in [(0, "DATTN_OK"), (-1, "DATTN_ERR_INVALID_ARG"), (-2, "DATTN_ERR_UNSUPPORTED"),
                       (-3, "DATTN_ERR_MISALIGNED"), (-4, "DATTN_ERR_WORKSPACE"),
                       (-5, "DATTN_ERR_CUDA"), (-6, "DATTN_ERR_TIMEOUT"),
                       (-7, "DATTN_ERR_BAD_PAGE"), (-8, "DATTN_ERR_BAD_POSITION")]:
        assert lib.dattn_status_string(code).decode() == name


A = 0x10000  # 16-byte aligned fake device addresses; never dereferenced


def call_ex(lib, Q=A, K=A, V=A, out=A, B=1, H=2, D=64, S=16, cp=A, ws=A, wsb=1 << 20, ns=0):
    return lib.dattn_decode_f16_ex(Q, K, V, out, B, H, D, S, cp, ws, wsb, ns, None)


@pytest.mark.parametrize("kw,status", [
    (dict(Q=None), _native.ERR_INVALID_ARG),
    (dict(K=None), _native.ERR_INVALID_ARG),
    (dict(V=None), _native.ERR_INVALID_ARG),
    (dict(out=None), _native.ERR_INVALID_ARG),
    (dict(cp=None), _native.ERR_INVALID_ARG),
    (dict(Q=A + 8), _native.ERR_MISALIGNED),
    (dict(K=A + 2), _native.ERR_MISALIGNED),
    (dict(V=A + 4), _native.ERR_MISALIGNED),
    (dict(out=A + 1), _native.ERR_MISALIGNED),
    (dict(cp=A + 2), _native.ERR_MISALIGNED),
    (dict(B=0), _native.ERR_INVALID_ARG),
    (dict(H=-1), _native.ERR_INVALID_ARG),
    (dict(S=0), _native.ERR_INVALID_ARG),
    (dict(D=0), _native.ERR_INVALID_ARG),
    (dict(D=12), _native.ERR_UNSUPPORTED),
    (dict(D=264), _native.ERR_UNSUPPORTED),
    (dict(ns=-3), _native.ERR_INVALID_ARG),
])
def test_decode_ex_rejects_bad_arguments_on_host(lib, kw, status):
    assert call_ex(lib, **kw) == status
    assert lib.dattn_last_error().decode() != ""


def test_split_calls_reject_bad_arguments_on_host(lib):
    assert lib.dattn_qk_f16(None, A, A, 1, 2, 64, 16, A, None) == _native.ERR_INVALID_ARG
    assert lib.dattn_qk_f16(A, A, A + 6, 1, 2, 64, 16, A, None) == _native.ERR_MISALIGNED
    assert lib.dattn_qk_f16(A, A, A, 1, 2, 20, 16, A, None) == _native.ERR_UNSUPPORTED
    assert lib.dattn_pv_f16(A, None, A, 1, 2, 64, 16, None) == _native.ERR_INVALID_ARG
    assert lib.dattn_pv_f16(A, A, A, 1, 0, 64, 16, None) == _native.ERR_INVALID_ARG
    assert lib.dattn_decode_f16(A, A, A, None, 1, 2, 64, 16, A, None) == _native.ERR_INVALID_ARG


def test_paged_decode_rejects_bad_arguments_on_host(lib):
    def call(Q=A, K=A, V=A, out=A, B=1, H=2, D=64, ps=16, maxp=4, npages=8, table=A, cp=A):
        return lib.dattn_decode_paged_f16(Q, K, V, out, B, H, D, ps, maxp, npages, table, cp,
                                          A, 1 << 20, 0, None)
    assert call(table=None) == _native.ERR_INVALID_ARG
    assert call(table=A + 2) == _native.ERR_MISALIGNED
    assert call(K=A + 8) == _native.ERR_MISALIGNED
    assert call(ps=0) == _native.ERR_INVALID_ARG
    assert call(maxp=-1) == _native.ERR_INVALID_ARG
    assert call(npages=0) == _native.ERR_INVALID_ARG
    assert call(ps=1 << 20, maxp=1 << 12) == _native.ERR_UNSUPPORTED
    assert call(D=20) == _native.ERR_UNSUPPORTED


def test_plan_queries_reject_bad_arguments_on_host(lib):
    n = ctypes.c_size_t(0)
    assert lib.dattn_decode_workspace_bytes(1, 2, 64, 16, 0, None) == _native.ERR_INVALID_ARG
    assert lib.dattn_decode_workspace_bytes(1, 2, 63, 16, 0, ctypes.byref(n)) == \
        _native.ERR_UNSUPPORTED
    assert lib.dattn_decode_plan(1, 2, 64, 16, 0, None) == _native.ERR_INVALID_ARG
    plan = _native.Plan()
    assert lib.dattn_decode_paged_plan(1, 2, 64, 16, 4, 10, 0, None) == _native.ERR_INVALID_ARG
    assert lib.dattn_decode_paged_plan(1, 2, 64, 0, 4, 10, 0, ctypes.byref(plan)) == \
        _native.ERR_INVALID_ARG
    assert lib.dattn_decode_paged_plan(1, 2, 64, 16, 4, 0, 0, ctypes.byref(plan)) == \
        _native.ERR_INVALID_ARG
    assert lib.dattn_decode_paged_plan(1, 2, 64, 1 << 20, 1 << 12, 10, 0, ctypes.byref(plan)) == \
        _native.ERR_UNSUPPORTED
    assert lib.dattn_decode_paged_plan(1, 2, 63, 16, 4, 10, 0, ctypes.byref(plan)) == \
        _native.ERR_UNSUPPORTED


def test_python_binding_rejects_pageable_cpu_tensors():
    import torch
    q = torch.zeros(1, 2, 64, dtype=torch.float16)
    k = torch.zeros(1, 16, 2, 64, dtype=torch.float16)
    cp = torch.zeros(1, dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA"):
        _native.dattn_decode_f16_ex(q, k, k, q, cp)
    with pytest.raises(TypeError):
        _native.dattn_decode_f16_ex(q.float(), k, k, q, cp)


def test_batch_api_rejects_bad_arguments_on_host(lib):
    import ctypes as C
    assert lib.dattn_batch_begin(None) == _native.ERR_INVALID_ARG  # the legacy stream
    assert lib.dattn_batch_end(A, None) == _native.ERR_INVALID_ARG
    assert lib.dattn_batch_launch(None, None) == _native.ERR_INVALID_ARG
    assert lib.dattn_batch_nodes(None) == -1
    assert lib.dattn_batch_destroy(None) == _native.OK


def test_softmax_rejects_bad_arguments_on_host(lib):
    assert lib.dattn_softmax_f32(None, A, 4, 8, None) == _native.ERR_INVALID_ARG
    assert lib.dattn_softmax_f32(A + 2, A, 4, 8, None) == _native.ERR_MISALIGNED
    assert lib.dattn_softmax_f32(A, A, 0, 8, None) == _native.ERR_INVALID_ARG
    assert lib.dattn_softmax_f32(A, A, 4, -1, None) == _native.ERR_INVALID_ARG


def rope_call(lib, q=A, k=A, v=A, qo=A, K=A, V=A, B=2, H=4, D=64, S=32, rd=64, base=10000.0,
              cp=A):
    return lib.dattn_rope_append_f16(q, k, v, qo, K, V, B, H, D, S, rd, base, 0, cp, None)


@pytest.mark.parametrize("kw,status", [
    (dict(q=None), _native.ERR_INVALID_ARG),
    (dict(V=None), _native.ERR_INVALID_ARG),
    (dict(k=A + 8), _native.ERR_MISALIGNED),
    (dict(cp=None), _native.ERR_INVALID_ARG),
    (dict(cp=A + 2), _native.ERR_MISALIGNED),
    (dict(B=0), _native.ERR_INVALID_ARG),
    (dict(S=-1), _native.ERR_INVALID_ARG),
    (dict(D=20, rd=20), _native.ERR_UNSUPPORTED),
    (dict(rd=0), _native.ERR_INVALID_ARG),
    (dict(rd=31), _native.ERR_INVALID_ARG),
    (dict(rd=66), _native.ERR_INVALID_ARG),
    (dict(base=1.0), _native.ERR_INVALID_ARG),
    (dict(base=float("inf")), _native.ERR_INVALID_ARG),
    (dict(base=float("nan")), _native.ERR_INVALID_ARG),
])
def test_rope_append_rejects_bad_arguments_on_host(lib, kw, status):
    assert rope_call(lib, **kw) == status


def test_paged_rope_append_rejects_bad_arguments_on_host(lib):
    def call(table=A, ps=16, maxp=4, npages=8, rd=64):
        return lib.dattn_rope_append_paged_f16(A, A, A, A, A, A, 2, 4, 64, ps, maxp, npages,
                                               table, rd, 10000.0, 1, A, None)
    assert call(table=None) == _native.ERR_INVALID_ARG
    assert call(table=A + 2) == _native.ERR_MISALIGNED
    assert call(ps=0) == _native.ERR_INVALID_ARG
    assert call(npages=0) == _native.ERR_INVALID_ARG
    assert call(ps=1 << 20, maxp=1 << 12) == _native.ERR_UNSUPPORTED
    assert call(rd=3) == _native.ERR_INVALID_ARG
