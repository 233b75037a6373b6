"""Parity of the cluster plan over a paged cache with the fp64 CPU oracle.

A single sequence held in pages of a pool (block table [1, max_pages]) is
decoded by one cluster of CTAs per head group, as for a dense cache, with the
CTAs' ranges cut at page boundaries so that the rows of a head group in each
whole page are copied as one tensor box.  Every comparison is element by
element with |out - ref| <= 2e-3 + 1e-2 |ref| (tests/_util.py), through the C
ABI; the oracle's paged decode is pinned against the dense oracle
(tests/test_oracle_pins.py).
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


def make_single(seed, H, D, ps, maxp, extra=3):
    """One sequence of maxp pages scattered over a pool of maxp + extra pages."""
    g = torch.Generator(device="cuda").manual_seed(seed)
    num_pages = maxp + extra
    kp = rand_f16(g, (num_pages, ps, H, D))
    vp = rand_f16(g, (num_pages, ps, H, D))
    q = rand_f16(g, (1, H, D))
    rng = np.random.default_rng(seed)
    table = rng.permutation(num_pages)[:maxp].reshape(1, maxp).astype(np.int32)
    return q, kp, vp, table


def run_and_check(q, kp, vp, table, cp, what):
    out = dattn.decode_paged(q, kp, vp, torch.from_numpy(table).cuda(), cur_pos_tensor([cp]))
    torch.cuda.synchronize()
    ref = oracle.decode_paged_f64(to_np(q), to_np(kp), to_np(vp), table,
                                  np.asarray([cp], np.uint32))
    assert_decode_close(out, ref, what)
    return out


def test_plan_choice():
    # the 7B-class step in 128-position pages takes the cluster plan, without
    # workspace, with stages of whole pages
    plan = dattn.dattn_decode_paged_plan(1, 32, 128, 128, 32, 40)
    assert plan["cluster_size"] > 0
    assert plan["workspace_bytes"] == 0
    assert plan["stage_positions"] % 128 == 0
    # 16-position pages (a head group's slice of a page would hold 32 KB of K
    # only with fewer CTAs), batches, forced partition counts and pools past
    # the 32-bit box row keep the split plan
    assert dattn.dattn_decode_paged_plan(1, 32, 128, 16, 256, 300)["cluster_size"] == 0
    assert dattn.dattn_decode_paged_plan(4, 32, 128, 128, 32, 140)["cluster_size"] == 0
    assert dattn.dattn_decode_paged_plan(1, 32, 128, 128, 32, 40, 37)["cluster_size"] == 0
    assert dattn.dattn_decode_paged_plan(1, 32, 128, 128, 32, 1 << 24)["cluster_size"] == 0


# (n_heads, head_dim, page_size, max_pages, current_pos, plan): the plan the
# call must take (True: cluster, False: split, None: either).  Pages of 128 and
# 256 positions, odd page sizes, live lengths ending inside a page, fewer live
# pages than CTAs, current_pos 0 and past the capacity, one head (whole-page
# spans instead of boxes)
CASES = [
    (32, 128, 128, 32, 4095, True),   # the 7B-class step in 128-position pages
    (32, 128, 128, 32, 0, True),
    (32, 128, 128, 32, 5, True),
    (32, 128, 128, 32, 130, True),    # the live length ends in the second page
    (32, 128, 128, 32, 1000, True),
    (32, 128, 128, 32, 9000, True),
    (32, 128, 256, 16, 4095, None),  # two 256-position stages do not fit one head per group
    (32, 128, 256, 16, 300, None),
    (40, 128, 128, 24, 3000, None),
    (64, 128, 128, 8, 1000, None),
    (16, 256, 128, 16, 2047, None),
    (8, 64, 256, 4, 1000, None),
    (32, 64, 256, 8, 2047, None),
    (32, 128, 200, 20, 3999, None),
    (1, 128, 256, 32, 8191, None),
    (2, 128, 128, 40, 5000, None),
    (32, 128, 16, 256, 4095, False),  # the 7B-class step in 16-position pages
    (32, 128, 1, 2048, 2047, False),
    (40, 128, 13, 100, 1234, None),
    (12, 64, 64, 2, 63, None),
    (8, 48, 5, 7, 34, None),
    (3, 8, 3, 40, 99, None),
    (20, 72, 9, 170, 1499, None),
]


@pytest.mark.parametrize("H,D,ps,maxp,cp,cluster", CASES,
                         ids=[f"H{c[0]}D{c[1]}ps{c[2]}x{c[3]}cp{c[4]}" for c in CASES])
def test_single_sequence(H, D, ps, maxp, cp, cluster):
    q, kp, vp, table = make_single(H * 7 + D + ps * 31 + cp, H, D, ps, maxp)
    plan = dattn.dattn_decode_paged_plan(1, H, D, ps, maxp, kp.shape[0])
    if cluster is not None:
        assert (plan["cluster_size"] > 0) == cluster, plan
    run_and_check(q, kp, vp, table, cp, f"H={H} D={D} ps={ps} cp={cp} plan={plan}")


def test_same_result_as_split_plan_within_tolerance_and_against_oracle():
    H, D, ps, maxp, cp = 32, 128, 128, 32, 4095
    q, kp, vp, table = make_single(3, H, D, ps, maxp)
    kp[..., :4] *= 20  # outlier channels: large scores
    tab = torch.from_numpy(table).cuda()
    a = dattn.decode_paged(q, kp, vp, tab, cur_pos_tensor([cp]))
    b = dattn.decode_paged(q, kp, vp, tab, cur_pos_tensor([cp]), num_partitions=152)
    torch.cuda.synchronize()
    ref = oracle.decode_paged_f64(to_np(q), to_np(kp), to_np(vp), table,
                                  np.asarray([cp], np.uint32))
    assert_decode_close(a, ref, "cluster plan")
    assert_decode_close(b, ref, "split plan")


def test_unreferenced_pages_and_entries_past_live_length_have_no_effect():
    H, D, ps, maxp, cp = 32, 128, 128, 16, 700  # live pages: 6
    q, kp, vp, table = make_single(11, H, D, ps, maxp, extra=8)
    assert dattn.dattn_decode_paged_plan(1, H, D, ps, maxp, kp.shape[0])["cluster_size"] > 0
    tab = torch.from_numpy(table).cuda()
    base = dattn.decode_paged(q, kp, vp, tab, cur_pos_tensor([cp])).clone()
    live = {int(table[0, j]) for j in range(cp // ps + 1)}
    kp2, vp2 = kp.clone(), vp.clone()
    for pg in range(kp.shape[0]):
        if pg not in live:
            kp2[pg] = float("nan")
            vp2[pg] = float("nan")
    table2 = table.copy()
    table2[0, cp // ps + 1:] = -1
    out = dattn.decode_paged(q, kp2, vp2, torch.from_numpy(table2).cuda(), cur_pos_tensor([cp]))
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), base.view(torch.int16))
    assert dattn.dattn_device_error(clear=True) == _native.OK


def test_invalid_live_page_is_reported_not_dereferenced():
    H, D, ps, maxp, cp = 32, 128, 128, 16, 1000
    q, kp, vp, table = make_single(12, H, D, ps, maxp)
    assert dattn.dattn_decode_paged_plan(1, H, D, ps, maxp, kp.shape[0])["cluster_size"] > 0
    bad = table.copy()
    bad[0, 5] = kp.shape[0] + 5  # a live page outside the pool
    assert dattn.dattn_device_error(clear=True) == _native.OK
    dattn.decode_paged(q, kp, vp, torch.from_numpy(bad).cuda(), cur_pos_tensor([cp]))
    assert dattn.dattn_device_error(clear=True) == _native.ERR_BAD_PAGE
    run_and_check(q, kp, vp, table, cp, "after a bad page")
    assert dattn.dattn_device_error(clear=True) == _native.OK


def test_identity_table_matches_dense_cluster_plan_within_tolerance():
    # the same cache seen densely and through an identity table: both plans
    # are cluster plans (their ranges differ, so the rounding may too)
    H, D, ps, maxp, cp = 32, 128, 128, 32, 3000
    S = ps * maxp
    g = torch.Generator(device="cuda").manual_seed(21)
    q, k, v = rand_f16(g, (1, H, D)), rand_f16(g, (1, S, H, D)), rand_f16(g, (1, S, H, D))
    table = torch.arange(maxp, dtype=torch.int32, device="cuda").view(1, maxp)
    cpt = cur_pos_tensor([cp])
    assert dattn.dattn_decode_paged_plan(1, H, D, ps, maxp, maxp)["cluster_size"] > 0
    dense = dattn.decode(q, k, v, cpt)
    paged = dattn.decode_paged(q, k.view(maxp, ps, H, D), v.view(maxp, ps, H, D), table, cpt)
    torch.cuda.synchronize()
    ref = oracle.decode_f64(to_np(q), to_np(k), to_np(v), np.asarray([cp], np.uint32))
    assert_decode_close(dense, ref, "dense")
    assert_decode_close(paged, ref, "paged")


def draw_paged_cases(n=80, seed=20261203):
    """Seeded single-sequence paged shapes: every head_dim class, page sizes 1
    to 256, head counts with few and many divisors, live lengths from 1 to past
    the capacity."""
    rng = np.random.default_rng(seed)
    cases = []
    while len(cases) < n:
        D = int(rng.integers(1, 33)) * 8
        H = int(rng.choice([1, 2, 4, 6, 8, 12, 16, 24, 32, 40, 64]))
        ps = int(rng.choice([1, 3, 5, 16, 16, 64, 100, 128, 128, 128, 200, 256, 256]))
        maxp = int(rng.integers(1, 4097 // ps + 2))
        S = ps * maxp
        if S * H * D > 1.6e7:
            continue
        cp = int(rng.integers(0, S + 5)) if rng.random() < 0.8 else int(rng.integers(0, 40))
        cases.append((H, D, ps, maxp, cp, len(cases)))
    return cases


RANDOM_CASES = draw_paged_cases()


@pytest.mark.parametrize("H,D,ps,maxp,cp,i", RANDOM_CASES,
                         ids=[f"{c[5]}-H{c[0]}D{c[1]}ps{c[2]}x{c[3]}cp{c[4]}" for c in RANDOM_CASES])
def test_random_single_sequence(H, D, ps, maxp, cp, i):
    q, kp, vp, table = make_single(9000 + i, H, D, ps, maxp)
    plan = dattn.dattn_decode_paged_plan(1, H, D, ps, maxp, kp.shape[0])
    run_and_check(q, kp, vp, table, cp, f"case {i}: plan {plan}")


def test_random_cases_cover_both_plans():
    plans = [dattn.dattn_decode_paged_plan(1, H, D, ps, maxp, maxp + 3)["cluster_size"] > 0
             for H, D, ps, maxp, _, _ in RANDOM_CASES]
    assert sum(plans) >= 12 and len(plans) - sum(plans) >= 12, sum(plans)


def test_append_and_decode_steps_back_to_back_across_a_page_boundary():
    # rope/append into a page and decode on the cluster plan, eight steps issued
    # back to back with no host synchronisation; the appended positions cross
    # from one page into the next.  Each step must see its own and every earlier
    # appended row.
    H, D, ps, maxp, steps, start = 32, 128, 128, 32, 8, 1020
    q0, kp, vp, table = make_single(31, H, D, ps, maxp)
    assert dattn.dattn_decode_paged_plan(1, H, D, ps, maxp, kp.shape[0])["cluster_size"] > 0
    g = torch.Generator(device="cuda").manual_seed(32)
    kp_host, vp_host = to_np(kp).copy(), to_np(vp).copy()
    tab = torch.from_numpy(table).cuda()
    toks = [tuple(rand_f16(g, (1, H, D)) for _ in range(3)) for _ in range(steps)]
    cpts = [cur_pos_tensor([start + t]) for t in range(steps)]
    q_rots = [torch.empty((1, H, D), dtype=torch.float16, device="cuda") for _ in range(steps)]
    outs = [torch.empty((1, H, D), dtype=torch.float16, device="cuda") for _ in range(steps)]
    n = _native.dattn_decode_workspace_bytes(1, H, D, ps * maxp, 0)
    ws = torch.empty((max(n, 16),), dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    for t in range(steps):
        q, kn, vn = toks[t]
        dattn.rope_append(q, kn, vn, kp, vp, cpts[t], block_table=tab, q_out=q_rots[t])
        dattn.decode_paged(q_rots[t], kp, vp, tab, cpts[t], out=outs[t], workspace=ws)
    torch.cuda.synchronize()
    for t in range(steps):
        q, kn, vn = toks[t]
        cp = [start + t]
        page, row = int(table[0, cp[0] // ps]), cp[0] % ps
        kp_host[page, row] = oracle.rope_f64(to_np(kn), cp).astype(np.float16)[0]
        vp_host[page, row] = to_np(vn)[0]
        q_ref = oracle.rope_f64(to_np(q), cp).astype(np.float16)
        ref = oracle.decode_paged_f64(q_ref, kp_host, vp_host, table, np.asarray(cp, np.uint32))
        assert_decode_close(outs[t], ref, f"step {t} (position {cp[0]})")


def test_recorded_batch_replays_on_new_pages_and_table():
    # a recorded submission keeps the pool's address (in the tensor maps) and
    # reads the block table, current_pos and the pages at replay
    H, D, ps, maxp = 32, 128, 128, 16
    q, kp, vp, table = make_single(41, H, D, ps, maxp, extra=8)
    assert dattn.dattn_decode_paged_plan(1, H, D, ps, maxp, kp.shape[0])["cluster_size"] > 0
    g = torch.Generator(device="cuda").manual_seed(42)
    tab = torch.from_numpy(table).cuda()
    cpt = cur_pos_tensor([2000])
    out = torch.empty_like(q)
    n = _native.dattn_decode_workspace_bytes(1, H, D, ps * maxp, 0)
    ws = torch.empty((max(n, 16),), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        dattn.dattn_decode_paged_f16(q, kp, vp, out, tab, cpt, ws, 0, stream=stream)
        torch.cuda.synchronize()
        dattn.dattn_batch_begin(stream)
        dattn.dattn_decode_paged_f16(q, kp, vp, out, tab, cpt, ws, 0, stream=stream)
        batch = dattn.dattn_batch_end(stream)
    rng = np.random.default_rng(43)
    for cp in (2000, 127, 128, 1500):
        q.normal_(generator=g)
        kp.normal_(generator=g)
        vp.normal_(generator=g)
        table = rng.permutation(kp.shape[0])[:maxp].reshape(1, maxp).astype(np.int32)
        tab.copy_(torch.from_numpy(table))
        cpt.fill_(cp)
        torch.cuda.synchronize()
        batch.launch(stream)
        stream.synchronize()
        ref = oracle.decode_paged_f64(to_np(q), to_np(kp), to_np(vp), table,
                                      np.asarray([cp], np.uint32))
        assert_decode_close(out, ref, f"replay cp={cp}")
    batch.close()


def test_rows_past_current_pos_in_the_last_page_have_no_effect():
    # the unit's last, partial page is copied whole (one tensor box); its rows
    # past current_pos land in shared memory but are never read
    H, D, ps, maxp = 32, 128, 128, 16
    q, kp, vp, table = make_single(51, H, D, ps, maxp)
    assert dattn.dattn_decode_paged_plan(1, H, D, ps, maxp, kp.shape[0])["cluster_size"] > 0
    tab = torch.from_numpy(table).cuda()
    for cp in (1000, 1023, 1024, 5):
        base = dattn.decode_paged(q, kp, vp, tab, cur_pos_tensor([cp])).clone()
        kp2, vp2 = kp.clone(), vp.clone()
        last = int(table[0, cp // ps])
        kp2[last, cp % ps + 1:] = float("nan")
        vp2[last, cp % ps + 1:] = float("inf")
        out = dattn.decode_paged(q, kp2, vp2, tab, cur_pos_tensor([cp]))
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), base.view(torch.int16)), cp
        ref = oracle.decode_paged_f64(to_np(q), to_np(kp), to_np(vp), table,
                                      np.asarray([cp], np.uint32))
        assert_decode_close(out, ref, f"cp={cp}")
