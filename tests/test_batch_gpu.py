"""Submission batching (dattn_batch_*): decode calls recorded once on a stream
and replayed as one submission, with new contents written into the same
buffers between replays -- how a decode loop reuses one recorded step."""
from __future__ import annotations

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


def _fill(g, *tensors):
    for t in tensors:
        t.normal_(0.0, 1.0, generator=g)


def test_recorded_decodes_replay_on_new_contents():
    g = torch.Generator(device="cuda").manual_seed(123)
    # call 1: dense decode with a caller workspace (merge kernel included)
    B1, H1, D1, S1 = 2, 32, 128, 3000
    q1, k1, v1 = rand_f16(g, (B1, H1, D1)), rand_f16(g, (B1, S1, H1, D1)), rand_f16(g, (B1, S1, H1, D1))
    cp1 = cur_pos_tensor([2999, 1200])
    out1 = torch.empty_like(q1)
    ws1 = torch.empty(max(16, dattn.dattn_decode_workspace_bytes(B1, H1, D1, S1)),
                      dtype=torch.uint8, device="cuda")
    # call 2: paged decode
    B2, H2, D2, ps, maxp = 3, 8, 64, 16, 10
    q2 = rand_f16(g, (B2, H2, D2))
    kp, vp = rand_f16(g, (B2 * maxp, ps, H2, D2)), rand_f16(g, (B2 * maxp, ps, H2, D2))
    table = torch.from_numpy(np.random.default_rng(5).permutation(B2 * maxp)
                             .reshape(B2, maxp).astype(np.int32)).cuda()
    cp2 = cur_pos_tensor([159, 20, 77])
    out2 = torch.empty_like(q2)
    ws2 = torch.empty(max(16, dattn.dattn_decode_workspace_bytes(B2, H2, D2, ps * maxp)),
                      dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    # call 3: the library-owned workspace of stream s, grown by one ordinary
    # call on s before recording
    out3 = torch.empty_like(q1)
    dattn.dattn_decode_f16(q1, k1, v1, out3, cp1, s)
    torch.cuda.synchronize()

    dattn.dattn_batch_begin(s)
    try:
        dattn.dattn_decode_f16_ex(q1, k1, v1, out1, cp1, ws1, 0, s)
        dattn.dattn_decode_paged_f16(q2, kp, vp, out2, table, cp2, ws2, 0, s)
        dattn.dattn_decode_f16(q1, k1, v1, out3, cp1, s)
    finally:
        batch = dattn.dattn_batch_end(s)
    assert batch.nodes >= 3
    torch.cuda.synchronize()

    for replay in range(3):
        _fill(g, q1, k1, v1, q2, kp, vp)
        cp1.copy_(cur_pos_tensor([2999 - replay, 600 + replay]))
        torch.cuda.synchronize()
        launch_stream = s if replay < 2 else torch.cuda.Stream()
        batch.launch(launch_stream)
        torch.cuda.synchronize()
        cph = cp1.cpu().numpy().astype(np.uint32)
        ref1 = oracle.decode_f64(to_np(q1), to_np(k1), to_np(v1), cph)
        assert_decode_close(out1, ref1, f"replay {replay}, dense")
        assert_decode_close(out3, ref1, f"replay {replay}, library workspace")
        ref2 = oracle.decode_paged_f64(to_np(q2), to_np(kp), to_np(vp), table.cpu().numpy(),
                                       np.array([159, 20, 77], np.uint32))
        assert_decode_close(out2, ref2, f"replay {replay}, paged")
    batch.close()
    assert dattn.dattn_device_error(clear=True) == _native.OK


def test_growing_the_library_workspace_while_recording_is_refused_cleanly():
    g = torch.Generator(device="cuda").manual_seed(9)
    # two sequences: the split plan, which needs a workspace (a single
    # sequence would take the cluster plan, which needs none)
    B, H, D, S = 2, 32, 128, 5000
    assert dattn.dattn_decode_plan(B, H, D, S)["workspace_bytes"] > 0
    q, k, v = rand_f16(g, (B, H, D)), rand_f16(g, (B, S, H, D)), rand_f16(g, (B, S, H, D))
    out = torch.empty_like(q)
    cp = cur_pos_tensor([4999, 1234])  # made before recording: no copies while recording
    s = torch.cuda.Stream()  # a fresh stream: its library workspace does not exist yet
    s.wait_stream(torch.cuda.current_stream())
    torch.cuda.synchronize()
    dattn.dattn_batch_begin(s)
    try:
        with pytest.raises(_native.DattnError) as ei:
            dattn.dattn_decode_f16(q, k, v, out, cp, s)
        assert ei.value.status == _native.ERR_WORKSPACE
    finally:
        batch = dattn.dattn_batch_end(s)
    batch.close()
    # outside recording the same call works
    dattn.dattn_decode_f16(q, k, v, out, cp, s)
    torch.cuda.synchronize()
    ref = oracle.decode_f64(to_np(q), to_np(k), to_np(v), np.array([4999, 1234], np.uint32))
    assert_decode_close(out, ref, "after the refused recording")


def test_recorded_decode_step_advances_one_token_per_replay():
    # one recorded step -- rotate and append the new token, then attend -- replayed
    # for three consecutive tokens with new q, k, v and current_pos written into
    # the same buffers between replays
    g = torch.Generator(device="cuda").manual_seed(321)
    B, H, D, S = 2, 16, 128, 64
    K, V = rand_f16(g, (B, S, H, D)), rand_f16(g, (B, S, H, D))
    K_host, V_host = to_np(K).copy(), to_np(V).copy()
    q, kn, vn = (torch.empty((B, H, D), dtype=torch.float16, device="cuda") for _ in range(3))
    cp = torch.empty((B,), dtype=torch.int32, device="cuda")
    q_rot, out = torch.empty_like(q), torch.empty_like(q)
    ws = torch.empty(max(16, dattn.dattn_decode_workspace_bytes(B, H, D, S)), dtype=torch.uint8,
                     device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    torch.cuda.synchronize()
    dattn.dattn_batch_begin(s)
    try:
        dattn.dattn_rope_append_f16(q, kn, vn, q_rot, K, V, cp, stream=s)
        dattn.dattn_decode_f16_ex(q_rot, K, V, out, cp, ws, 0, s)
    finally:
        batch = dattn.dattn_batch_end(s)
    try:
        for step, pos in enumerate(([40, 10], [41, 11], [42, 12])):
            _fill(g, q, kn, vn)
            cp.copy_(cur_pos_tensor(pos))
            torch.cuda.synchronize()
            batch.launch(s)
            s.synchronize()
            q_ref = oracle.rope_f64(to_np(q), pos).astype(np.float16)
            k_ref = oracle.rope_f64(to_np(kn), pos).astype(np.float16)
            for b in range(B):
                K_host[b, pos[b]] = k_ref[b]
                V_host[b, pos[b]] = to_np(vn[b])
            ref = oracle.decode_f64(q_ref, K_host, V_host, np.asarray(pos, np.uint32))
            assert_decode_close(out, ref, f"recorded step {step}")
    finally:
        batch.close()
    assert dattn.dattn_device_error(clear=True) == _native.OK
