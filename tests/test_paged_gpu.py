"""Paged KV cache: dattn_decode_paged_f16 against the fp64 paged oracle.

The cache is a pool of pages [num_pages, page_size, H, D] reached through a
block table [B, max_pages]; the oracle's paged decode is pinned against the
dense oracle (tests/test_oracle_pins.py).
"""
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
    yield
    assert dattn.dattn_device_error(clear=True) == _native.OK


def make_paged(seed, B, H, D, ps, maxp, extra=5, share=True):
    g = torch.Generator(device="cuda").manual_seed(seed)
    num_pages = B * maxp + extra
    kp = rand_f16(g, (num_pages, ps, H, D))
    vp = rand_f16(g, (num_pages, ps, H, D))
    q = rand_f16(g, (B, H, D))
    rng = np.random.default_rng(seed)
    table = rng.permutation(num_pages)[: B * maxp].reshape(B, maxp).astype(np.int32)
    if share and B > 1:
        table[1, : maxp // 2] = table[0, : maxp // 2]  # shared prefix pages
    return q, kp, vp, table


CASES = [
    # B, H, D, page_size, max_pages, current_pos
    (3, 8, 64, 16, 8, [127, 40, 0]),
    (4, 32, 128, 16, 20, [319, 100, 5, 1000]),
    (2, 32, 128, 1, 300, [299, 150]),
    (3, 40, 128, 7, 30, [209, 13, 100]),
    (2, 4, 48, 64, 3, [191, 70]),
    (2, 64, 256, 8, 6, [47, 20]),   # two head groups: tensor boxes inside pages
    (2, 80, 256, 7, 9, [62, 30]),   # three groups, odd pages: boxes and per-position runs
]


@pytest.mark.parametrize("partitions", [0, 5])
@pytest.mark.parametrize("B,H,D,ps,maxp,cp", CASES,
                         ids=[f"B{c[0]}H{c[1]}D{c[2]}ps{c[3]}" for c in CASES])
def test_paged_decode_matches_oracle(B, H, D, ps, maxp, cp, partitions):
    q, kp, vp, table = make_paged(B * 100 + ps + D, B, H, D, ps, maxp)
    out = dattn.decode_paged(q, kp, vp, torch.from_numpy(table).cuda(), cur_pos_tensor(cp),
                             num_partitions=partitions)
    torch.cuda.synchronize()
    ref = oracle.decode_paged_f64(to_np(q), to_np(kp), to_np(vp), table,
                                  np.asarray(cp, np.uint32))
    assert_decode_close(out, ref, f"paged ps={ps} partitions={partitions}")


def test_identity_table_equals_dense_decode_bit_for_bit():
    g = torch.Generator(device="cuda").manual_seed(77)
    B, H, D, ps, maxp = 3, 32, 128, 16, 16
    S = ps * maxp
    q, k, v = rand_f16(g, (B, H, D)), rand_f16(g, (B, S, H, D)), rand_f16(g, (B, S, H, D))
    cp = cur_pos_tensor([255, 100, 7])
    table = torch.arange(B * maxp, dtype=torch.int32, device="cuda").view(B, maxp)
    dense = dattn.decode(q, k, v, cp)
    paged = dattn.decode_paged(q, k.view(B * maxp, ps, H, D), v.view(B * maxp, ps, H, D), table,
                               cp)
    torch.cuda.synchronize()
    assert torch.equal(dense.view(torch.int16), paged.view(torch.int16))


def test_unreferenced_pages_and_entries_past_live_length_have_no_effect():
    # K and V are never read through them (the kernel may read such entries as
    # bounds-checked L2 prefetch hints); NaN pages and invalid entries there
    # leave the output bit-identical and raise no error
    B, H, D, ps, maxp = 3, 32, 128, 8, 10
    q, kp, vp, table = make_paged(5, B, H, D, ps, maxp, extra=6, share=False)
    cp = [30, 7, 55]  # live pages: 4, 1, 7
    tab = torch.from_numpy(table).cuda()
    base = dattn.decode_paged(q, kp, vp, tab, cur_pos_tensor(cp)).clone()
    live = {int(table[b, j]) for b, n in enumerate([4, 1, 7]) for j in range(n)}
    kp2, vp2 = kp.clone(), vp.clone()
    for pg in range(kp.shape[0]):
        if pg not in live:
            kp2[pg] = float("nan")
            vp2[pg] = float("nan")
    table2 = table.copy()
    table2[0, 4:] = -1
    table2[1, 1:] = 1 << 30
    out = dattn.decode_paged(q, kp2, vp2, torch.from_numpy(table2).cuda(), cur_pos_tensor(cp))
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), base.view(torch.int16))
    assert dattn.dattn_device_error(clear=True) == _native.OK


def test_invalid_live_page_is_reported_not_dereferenced():
    B, H, D, ps, maxp = 2, 8, 64, 16, 4
    q, kp, vp, table = make_paged(9, B, H, D, ps, maxp)
    table[1, 2] = kp.shape[0] + 5  # a live page of sequence 1 points outside the pool
    assert dattn.dattn_device_error(clear=True) == _native.OK
    dattn.decode_paged(q, kp, vp, torch.from_numpy(table).cuda(), cur_pos_tensor([63, 63]))
    assert dattn.dattn_device_error(clear=True) == _native.ERR_BAD_PAGE
    # the context is fine: a valid call right after is correct
    table[1, 2] = 0
    out = dattn.decode_paged(q, kp, vp, torch.from_numpy(table).cuda(), cur_pos_tensor([63, 63]))
    torch.cuda.synchronize()
    ref = oracle.decode_paged_f64(to_np(q), to_np(kp), to_np(vp), table,
                                  np.array([63, 63], np.uint32))
    assert_decode_close(out, ref, "after a bad page")
    assert dattn.dattn_device_error(clear=True) == _native.OK


def test_paged_ragged_workload_shape():
    # the ragged workload's shape (B=64 H=32 D=128 S=2048) held in 16-position pages
    from token_decode_attention_gb300.workloads import WORKLOADS, make_inputs
    w = WORKLOADS["ragged"]
    x = make_inputs(w, "cuda")
    ps = 16
    maxp = w.seq_len // ps
    B, S, H, D = x["k"].shape
    rng = np.random.default_rng(w.seed)
    perm = rng.permutation(B * maxp)
    kp = torch.empty((B * maxp, ps, H, D), dtype=torch.float16, device="cuda")
    vp = torch.empty_like(kp)
    kp[torch.from_numpy(perm).cuda()] = x["k"].view(B * maxp, ps, H, D)
    vp[torch.from_numpy(perm).cuda()] = x["v"].view(B * maxp, ps, H, D)
    table = torch.from_numpy(perm.reshape(B, maxp).astype(np.int32)).cuda()
    out = dattn.decode_paged(x["q"], kp, vp, table, x["cur_pos"])
    dense = dattn.decode(x["q"], x["k"], x["v"], x["cur_pos"])
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), dense.view(torch.int16))
    ref = oracle.decode_f64(to_np(x["q"]), to_np(x["k"]), to_np(x["v"]), x["cur_pos_host"])
    assert_decode_close(out, ref, "paged ragged")


# few heads in small pages over long contexts: a page is a small copy, a
# stage spans many pages and the pre-wait prefetch window many table entries
# (read one lane per page); B, H, D, page_size, max_pages, current_pos
FEW_HEAD_CASES = [
    (1, 1, 128, 16, 8192, [100000]),
    (1, 2, 128, 16, 8192, [131071]),
    (4, 1, 128, 16, 4096, [65535, 30000, 1, 50000]),
    (2, 4, 64, 8, 4096, [32767, 20000]),
]


@pytest.mark.parametrize("B,H,D,ps,maxp,cp", FEW_HEAD_CASES,
                         ids=[f"B{c[0]}H{c[1]}D{c[2]}ps{c[3]}x{c[4]}" for c in FEW_HEAD_CASES])
def test_few_heads_small_pages_long_context(B, H, D, ps, maxp, cp):
    q, kp, vp, table = make_paged(B * 1000 + H * 10 + ps, B, H, D, ps, maxp, share=False)
    out = dattn.decode_paged(q, kp, vp, torch.from_numpy(table).cuda(), cur_pos_tensor(cp))
    torch.cuda.synchronize()
    ref = oracle.decode_paged_f64(to_np(q), to_np(kp), to_np(vp), table, np.asarray(cp, np.uint32))
    assert_decode_close(out, ref, f"B={B} H={H} ps={ps}")
