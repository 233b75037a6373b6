"""dattn_decode_f16_noalloc: the fused decode for callers that cannot allocate.

Callers such as runtimes that own all device memory through their own pool, or
code running where a cudaMalloc is forbidden or would synchronise the device,
cannot hand the library a freshly allocated workspace.  This entry point uses a
static device array built into the library instead.  Here it is called
through the C ABI (ctypes, raw device pointers).  It runs the same plan and the
same kernels as the workspace-taking entry point dattn_decode_f16_ex with the
library-chosen partition count, so its output must be bit-identical to that
call's on the same inputs: that is checked on calls made back to back, among
them two calls of one shape on different inputs (the second finds the first
one's partial states left in the scratch and must not be affected by them).
One output is also compared with the fp64 oracle within the decode tolerance
of the other tests.

This file is named so that pytest collects it last; it passes alone in a fresh
process as well as after the other tests.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from token_decode_attention_gb300 import _native, build

from ._util import assert_decode_close, cur_pos_tensor, rand_f16, to_np

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 32 * 1024 * 1024  # DATTN_NOALLOC_SCRATCH_BYTES in include/dattn.h


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _native.load()


def _noalloc(lib, q, k, v, out, cp):
    B, H, D = q.shape
    S = k.shape[1]
    stream = torch.cuda.current_stream().cuda_stream
    return lib.dattn_decode_f16_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                        B, H, D, S, cp.data_ptr(), stream)


def _reference(q, k, v, cp):
    """The existing entry point, with a workspace allocated by the test and the
    library-chosen partition count (the plan the no-alloc call uses)."""
    B, H, D = q.shape
    S = k.shape[1]
    out = torch.empty((B, H, D), dtype=torch.float16, device="cuda")
    n = _native.dattn_decode_workspace_bytes(B, H, D, S, 0)
    ws = torch.empty((max(n, 16),), dtype=torch.uint8, device="cuda")
    _native.dattn_decode_f16_ex(q, k, v, out, cp, ws, 0)
    return out


def _inputs(g, B, H, D, S):
    return rand_f16(g, (B, H, D)), rand_f16(g, (B, S, H, D)), rand_f16(g, (B, S, H, D))


def test_calls_in_a_row_match_the_workspace_entry_point_bit_for_bit(lib):
    g = torch.Generator(device="cuda").manual_seed(20260123)
    cases = [
        # (B, H, D, S, current_pos): all take the split plan, whose partial
        # states go through the scratch.  The first two are one shape on
        # different inputs and current_pos.
        (2, 32, 128, 4096, [4095, 1000]),
        (2, 32, 128, 4096, [1777, 4095]),
        (6, 8, 64, 1500, [1499, 0, 700, 3, 1200, 999]),
    ]
    for i, (B, H, D, S, cp) in enumerate(cases):
        plan = _native.dattn_decode_plan(B, H, D, S, 0)
        assert plan["cluster_size"] == 0 and plan["workspace_bytes"] > 0
        q, k, v = _inputs(g, B, H, D, S)
        cpt = cur_pos_tensor(cp)
        out = torch.full((B, H, D), float("nan"), dtype=torch.float16, device="cuda")
        st = _noalloc(lib, q, k, v, out, cpt)
        assert st == 0, lib.dattn_last_error().decode()
        ref = _reference(q, k, v, cpt)
        torch.cuda.synchronize()
        assert torch.equal(out, ref), f"call {i + 1}: differs from dattn_decode_f16_ex"
        if i == 0:
            exact = oracle.decode_f64(to_np(q), to_np(k), to_np(v), np.asarray(cp, np.uint32))
            assert_decode_close(out, exact, f"call {i + 1} against the oracle")
    assert _native.dattn_device_error(clear=True) == 0


def test_single_sequence_on_the_cluster_plan_matches_bit_for_bit(lib):
    # one sequence takes the cluster plan, which needs no scratch at all: the
    # call must still match the workspace entry point exactly, twice in a row
    g = torch.Generator(device="cuda").manual_seed(20260124)
    B, H, D, S = 1, 32, 128, 4096
    plan = _native.dattn_decode_plan(B, H, D, S, 0)
    assert plan["cluster_size"] > 0 and plan["workspace_bytes"] == 0
    for i, cp in enumerate(([3000], [4095])):
        q, k, v = _inputs(g, B, H, D, S)
        cpt = cur_pos_tensor(cp)
        out = torch.full((B, H, D), float("nan"), dtype=torch.float16, device="cuda")
        assert _noalloc(lib, q, k, v, out, cpt) == 0, lib.dattn_last_error().decode()
        ref = _reference(q, k, v, cpt)
        torch.cuda.synchronize()
        assert torch.equal(out, ref), f"call {i + 1}: differs from dattn_decode_f16_ex"
    exact = oracle.decode_f64(to_np(q), to_np(k), to_np(v), np.asarray(cp, np.uint32))
    assert_decode_close(out, exact, "cluster plan against the oracle")
    assert _native.dattn_device_error(clear=True) == 0


def test_shape_beyond_static_scratch_is_rejected(lib):
    # 4096 short sequences x 64 heads need ~140 MB of partial states; the call
    # must fail on the host before launching anything
    B, H, D, S = 4096, 64, 128, 16
    need = _native.dattn_decode_workspace_bytes(B, H, D, S, 0)
    assert need > SCRATCH_BYTES  # guarantees the host-side rejection below
    fake = 1 << 20  # aligned, never dereferenced: nothing is launched on rejection
    st = lib.dattn_decode_f16_noalloc(fake, fake, fake, fake, B, H, D, S, fake, None)
    assert st == _native.ERR_WORKSPACE
    assert "scratch" in lib.dattn_last_error().decode()
