"""Failure detection on the GPU, without any fault.

Every pipeline wait in the library's kernels is bounded: a wait that runs out
records a code in the device error word and lets its kernel return, so the
context stays usable and the host reads the failure as DATTN_ERR_TIMEOUT.  The
self-test entry point makes one such wait run out on purpose (an mbarrier that
nothing arrives on); this test checks the status and that the next decode on
the same context is still correct.
"""
from __future__ import annotations

import time

import numpy as np
import pytest
import torch

import oracle
import token_decode_attention_gb300 as dattn
from token_decode_attention_gb300 import _native

from ._util import assert_decode_close, cur_pos_tensor, rand_f16, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from token_decode_attention_gb300 import build
    build.build()
    dattn.load()


def test_run_out_wait_becomes_a_host_status_and_context_stays_usable():
    assert dattn.dattn_device_error(clear=True) == _native.OK
    t0 = time.perf_counter()
    _native.dattn_selftest_wait_timeout()
    assert dattn.dattn_device_error(clear=True) == _native.ERR_TIMEOUT
    elapsed = time.perf_counter() - t0
    assert 0.5 < elapsed < 30.0  # the wait gave up after about its one-second limit
    assert dattn.dattn_device_error(clear=True) == _native.OK  # cleared

    # the context is intact: a decode right after is correct
    g = torch.Generator(device="cuda").manual_seed(31)
    B, H, D, S, cp = 2, 32, 128, 700, [699, 100]
    q, k, v = rand_f16(g, (B, H, D)), rand_f16(g, (B, S, H, D)), rand_f16(g, (B, S, H, D))
    out = dattn.decode(q, k, v, cur_pos_tensor(cp))
    torch.cuda.synchronize()
    ref = oracle.decode_f64(to_np(q), to_np(k), to_np(v), np.asarray(cp, np.uint32))
    assert_decode_close(out, ref, "decode after the self-test")
    assert dattn.dattn_device_error(clear=True) == _native.OK
