"""Parity of the cluster plan of the fused decode with the fp64 CPU oracle.

A dense cache of a single sequence is decoded by one cluster of CTAs per head
group: the CTAs of a cluster split the live positions, and their partial
softmax states (m, l, acc) are merged through distributed shared memory into
the f16 output by the same launch (no workspace, no merge kernel).  Head groups
smaller than n_heads are copied as tensor boxes.  Every comparison is element by
element with |out - ref| <= 2e-3 + 1e-2 |ref| (tests/_util.py), through the C ABI.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import token_decode_attention_gb300 as dattn
from token_decode_attention_gb300.workloads import WORKLOADS

from ._util import assert_decode_close, cur_pos_tensor, rand_f16, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from token_decode_attention_gb300 import build
    build.build()
    dattn.load()
    yield
    assert dattn.dattn_device_error(clear=True) == 0, "a kernel recorded a pipeline timeout"


def test_plan_choice():
    # the latency-bound single-sequence workloads take a cluster plan without
    # workspace ...
    for name in ("small", "7b"):
        w = WORKLOADS[name]
        plan = dattn.dattn_decode_plan(w.batch, w.n_heads, w.head_dim, w.seq_len)
        assert plan["cluster_size"] > 0, name
        assert plan["workspace_bytes"] == 0, name
        assert plan["partitions"] == plan["cluster_size"] * plan["head_groups"], name
    # ... a 2 GiB cache, batches and forced partition counts keep the split plan
    w = WORKLOADS["long"]
    assert dattn.dattn_decode_plan(w.batch, w.n_heads, w.head_dim, w.seq_len)["cluster_size"] == 0
    assert dattn.dattn_decode_plan(64, 32, 128, 2048)["cluster_size"] == 0
    assert dattn.dattn_decode_plan(1, 32, 128, 4096, 37)["cluster_size"] == 0
    # few heads leave too few CTAs for a cluster plan past the latency-bound sizes
    for H, S in ((1, 131072), (2, 131072), (4, 65536), (1, 16384)):
        assert dattn.dattn_decode_plan(1, H, 128, S)["cluster_size"] == 0, (H, S)
    assert dattn.dattn_decode_plan(1, 1, 128, 256)["cluster_size"] > 0


# (n_heads, head_dim, seq_len, current_pos): a single sequence; head counts with
# several divisors, every head_dim class, fewer live positions than CTAs,
# current_pos 0 and past seq_len, live lengths that end inside a stage
CASES = [
    (32, 128, 4096, 4095),   # the 7b workload's shape
    (32, 128, 4096, 0),
    (32, 128, 4096, 5),      # most CTAs of each cluster hold no position
    (32, 128, 4096, 17),
    (32, 128, 4096, 1000),
    (32, 128, 4096, 9000),   # beyond seq_len: nothing masked
    (8, 64, 256, 200),       # the small workload's shape
    (8, 64, 256, 3),
    (40, 128, 3000, 2999),
    (40, 128, 3000, 1234),
    (12, 64, 64, 63),        # the page's test shape
    (8, 48, 35, 34),         # the page's awkward dimensions
    (16, 256, 2048, 2047),
    (64, 128, 1024, 1000),
    (6, 96, 500, 499),
    (3, 8, 100, 99),
    (1, 128, 8192, 8191),
    (2, 16, 777, 700),
    (20, 72, 1500, 1499),
]


@pytest.mark.parametrize("H,D,S,cp", CASES)
def test_single_sequence(H, D, S, cp):
    g = torch.Generator(device="cuda").manual_seed(H * 100003 + D * 1009 + S + cp)
    q, k, v = rand_f16(g, (1, H, D)), rand_f16(g, (1, S, H, D)), rand_f16(g, (1, S, H, D))
    out = dattn.decode(q, k, v, cur_pos_tensor([cp]))
    torch.cuda.synchronize()
    ref = oracle.decode_f64(to_np(q), to_np(k), to_np(v), np.asarray([cp], np.uint32))
    plan = dattn.dattn_decode_plan(1, H, D, S)
    assert_decode_close(out, ref, f"H={H} D={D} S={S} cp={cp} plan={plan}")


@pytest.mark.parametrize("cp", [2500, 4000, 130, 5])
def test_positions_past_current_pos_are_never_read(cp):
    # live lengths whose CTA ranges end inside a stage: each range's last stage
    # is copied as a whole tensor box ending where the range ends (its first
    # rows are rows before the range, or the fill value below position 0)
    H, D, S = 32, 128, 4096
    g = torch.Generator(device="cuda").manual_seed(77)
    q, k, v = rand_f16(g, (1, H, D)), rand_f16(g, (1, S, H, D)), rand_f16(g, (1, S, H, D))
    cpt = cur_pos_tensor([cp])
    clean = dattn.decode(q, k, v, cpt)
    k2, v2 = k.clone(), v.clone()
    k2[:, cp + 1:] = float("nan")
    v2[:, cp + 1:] = float("inf")
    poisoned = dattn.decode(q, k2, v2, cpt)
    torch.cuda.synchronize()
    assert dattn.dattn_decode_plan(1, H, D, S)["cluster_size"] > 0
    assert torch.equal(clean, poisoned)
    ref = oracle.decode_f64(to_np(q), to_np(k), to_np(v), np.asarray([cp], np.uint32))
    assert_decode_close(clean, ref, f"cp={cp}")


def test_against_split_plan_and_oracle_outlier_channels():
    # K with 20x outlier channels (large scores); the cluster plan and a forced
    # split plan both match the oracle
    H, D, S, cp = 32, 128, 4096, 4095
    g = torch.Generator(device="cuda").manual_seed(5)
    q, k, v = rand_f16(g, (1, H, D)), rand_f16(g, (1, S, H, D)), rand_f16(g, (1, S, H, D))
    k[..., :4] *= 20
    cpt = cur_pos_tensor([cp])
    a = dattn.decode(q, k, v, cpt)
    b = dattn.decode(q, k, v, cpt, num_partitions=152)
    torch.cuda.synchronize()
    ref = oracle.decode_f64(to_np(q), to_np(k), to_np(v), np.asarray([cp], np.uint32))
    assert_decode_close(a, ref, "cluster plan")
    assert_decode_close(b, ref, "split plan")


def test_back_to_back_calls_without_host_sync():
    # consecutive launches overlap their prologues (programmatic dependent
    # launch); each call must still see only its own inputs
    H, D, S = 32, 128, 4096
    g = torch.Generator(device="cuda").manual_seed(9)
    sets = []
    for cp in (4095, 100, 2048, 7):
        q, k, v = rand_f16(g, (1, H, D)), rand_f16(g, (1, S, H, D)), rand_f16(g, (1, S, H, D))
        sets.append((q, k, v, cp, cur_pos_tensor([cp])))
    outs = [dattn.decode(q, k, v, cpt) for q, k, v, _, cpt in sets]
    torch.cuda.synchronize()
    for (q, k, v, cp, _), out in zip(sets, outs):
        ref = oracle.decode_f64(to_np(q), to_np(k), to_np(v), np.asarray([cp], np.uint32))
        assert_decode_close(out, ref, f"cp={cp}")


def test_recorded_batch_replays_on_new_contents():
    H, D, S = 8, 64, 256
    g = torch.Generator(device="cuda").manual_seed(13)
    q, k, v = rand_f16(g, (1, H, D)), rand_f16(g, (1, S, H, D)), rand_f16(g, (1, S, H, D))
    cpt = cur_pos_tensor([200])
    out = torch.empty_like(q)
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        dattn.dattn_decode_f16(q, k, v, out, cpt)  # first call outside the recording
        torch.cuda.synchronize()
        dattn.dattn_batch_begin(stream)
        dattn.dattn_decode_f16(q, k, v, out, cpt, stream=stream)
        batch = dattn.dattn_batch_end(stream)
    for cp in (200, 31, 255):
        q.normal_(generator=g)
        k.normal_(generator=g)
        v.normal_(generator=g)
        cpt.fill_(cp)
        torch.cuda.synchronize()
        batch.launch(stream)
        stream.synchronize()
        ref = oracle.decode_f64(to_np(q), to_np(k), to_np(v), np.asarray([cp], np.uint32))
        assert_decode_close(out, ref, f"replay cp={cp}")
    batch.close()


def draw_single_sequence_cases(n=120, seed=20261202):
    """Seeded single-sequence shapes for the cluster plan: every head_dim class,
    head counts with few and many divisors, live lengths from 1 to past seq_len."""
    rng = np.random.default_rng(seed)
    cases = []
    while len(cases) < n:
        D = int(rng.integers(1, 33)) * 8
        H = int(rng.choice([1, 2, 3, 4, 6, 7, 8, 12, 16, 24, 32, 40, 48, 64]))
        S = int(rng.integers(1, 5000))
        if S * H * D > 1.6e7:
            continue
        cp = int(rng.integers(0, S + 5)) if rng.random() < 0.8 else int(rng.integers(0, 40))
        cases.append((H, D, S, cp, len(cases)))
    return cases


RANDOM_CASES = draw_single_sequence_cases()


@pytest.mark.parametrize("H,D,S,cp,i", RANDOM_CASES,
                         ids=[f"{c[4]}-H{c[0]}D{c[1]}S{c[2]}cp{c[3]}" for c in RANDOM_CASES])
def test_random_single_sequence(H, D, S, cp, i):
    g = torch.Generator(device="cuda").manual_seed(5000 + i)
    q, k, v = rand_f16(g, (1, H, D)), rand_f16(g, (1, S, H, D)), rand_f16(g, (1, S, H, D))
    out = dattn.decode(q, k, v, cur_pos_tensor([cp]))
    torch.cuda.synchronize()
    ref = oracle.decode_f64(to_np(q), to_np(k), to_np(v), np.asarray([cp], np.uint32))
    assert_decode_close(out, ref, f"case {i}: plan {dattn.dattn_decode_plan(1, H, D, S)}")
