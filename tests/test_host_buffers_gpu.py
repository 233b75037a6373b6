"""Calls whose small per-step buffers live in pinned host memory.

Under unified addressing a page-locked host allocation has the same address on
the device, so the kernels can read a new token's q, k, v and current_pos from
the host and write the decode output back there over the CPU-GPU link, with no
copy-engine transfer.  The results must be bit-identical to the same calls on
device buffers, for both decode plans, for the rotary-embedding append, and for
a recorded step replayed on new host contents.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import token_decode_attention_gb300 as dattn

from ._util import assert_decode_close, rand_f16, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from token_decode_attention_gb300 import build
    build.build()
    dattn.load()
    yield
    assert dattn.dattn_device_error(clear=True) == 0


def _pinned(t: torch.Tensor) -> torch.Tensor:
    return t.cpu().pin_memory()


@pytest.mark.parametrize("B,H,D,S,cp", [
    (1, 32, 128, 4096, [4095]),          # cluster plan
    (1, 8, 64, 256, [200]),              # cluster plan, one head group
    (3, 32, 128, 1000, [999, 10, 500]),  # split plan with its merge kernel
])
def test_decode_with_host_query_positions_and_output(B, H, D, S, cp):
    g = torch.Generator(device="cuda").manual_seed(B * 1000 + S)
    q, k, v = rand_f16(g, (B, H, D)), rand_f16(g, (B, S, H, D)), rand_f16(g, (B, S, H, D))
    cpt = torch.tensor(cp, dtype=torch.int32, device="cuda")
    ref = dattn.decode(q, k, v, cpt)
    q_h, cp_h = _pinned(q), _pinned(cpt)
    out_h = torch.full((B, H, D), float("nan"), dtype=torch.float16).pin_memory()
    ws = torch.empty((max(16, dattn.dattn_decode_workspace_bytes(B, H, D, S)),),
                     dtype=torch.uint8, device="cuda")
    dattn.dattn_decode_f16_ex(q_h, k, v, out_h, cp_h, ws)
    torch.cuda.synchronize()
    assert torch.equal(out_h, ref.cpu())


def test_rope_append_reads_the_new_token_from_host():
    B, H, D, S = 2, 16, 128, 64
    g = torch.Generator(device="cuda").manual_seed(31)
    new = [rand_f16(g, (B, H, D)) for _ in range(3)]
    cpt = torch.tensor([17, 63], dtype=torch.int32, device="cuda")
    K, V = rand_f16(g, (B, S, H, D)), rand_f16(g, (B, S, H, D))
    K2, V2 = K.clone(), V.clone()
    q_dev = torch.empty_like(new[0])
    dattn.dattn_rope_append_f16(*new, q_dev, K, V, cpt)
    q_host_in = torch.empty_like(new[0])
    hn = [_pinned(t) for t in new]
    dattn.dattn_rope_append_f16(*hn, q_host_in, K2, V2, _pinned(cpt))
    torch.cuda.synchronize()
    assert torch.equal(q_dev, q_host_in)
    assert torch.equal(K, K2) and torch.equal(V, V2)


def test_recorded_step_replayed_on_new_host_contents():
    # the end-to-end decode step: rotate and append the new token read from one
    # pinned host buffer, attend, write the output into pinned host memory
    B, H, D, S = 1, 32, 128, 512
    g = torch.Generator(device="cuda").manual_seed(47)
    K, V = rand_f16(g, (B, S, H, D)), rand_f16(g, (B, S, H, D))
    n = B * H * D
    pack = torch.empty((3 * n * 2 + 4 * B,), dtype=torch.uint8).pin_memory()
    halves = pack[:6 * n].view(torch.float16)
    q_h, k_h, v_h = (halves[i * n:(i + 1) * n].view(B, H, D) for i in range(3))
    cp_h = pack[6 * n:].view(torch.int32)
    out_h = torch.empty((B, H, D), dtype=torch.float16).pin_memory()
    q_rot = torch.empty((B, H, D), dtype=torch.float16, device="cuda")
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    hg = torch.Generator().manual_seed(5)
    halves.copy_(torch.randn(3 * n, generator=hg).half())
    cp_h.fill_(100)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        dattn.dattn_rope_append_f16(q_h, k_h, v_h, q_rot, K, V, cp_h, stream=stream)
        dattn.dattn_decode_f16(q_rot, K, V, out_h, cp_h, stream=stream)
        stream.synchronize()
        dattn.dattn_batch_begin(stream)
        dattn.dattn_rope_append_f16(q_h, k_h, v_h, q_rot, K, V, cp_h, stream=stream)
        dattn.dattn_decode_f16(q_rot, K, V, out_h, cp_h, stream=stream)
        batch = dattn.dattn_batch_end(stream)
    for step, pos in enumerate((101, 102, 103)):
        halves.copy_(torch.randn(3 * n, generator=hg).half())
        cp_h.fill_(pos)
        batch.launch(stream)
        stream.synchronize()
        # the decode, on the cache as it stands (the appended rows included)
        ref = oracle.decode_f64(to_np(q_rot), to_np(K), to_np(V), np.array([pos], np.uint32))
        assert_decode_close(out_h, ref, f"step {step}")
        # the rotation and the append equal those of the same call on device copies
        assert torch.equal(V[0, pos].cpu(), v_h[0])
        K_chk, V_chk, q_chk = K.clone(), V.clone(), torch.empty_like(q_rot)
        dattn.dattn_rope_append_f16(q_h.cuda(), k_h.cuda(), v_h.cuda(), q_chk, K_chk, V_chk,
                                    cp_h.cuda())
        torch.cuda.synchronize()
        assert torch.equal(q_chk, q_rot) and torch.equal(K_chk, K)
    batch.close()
