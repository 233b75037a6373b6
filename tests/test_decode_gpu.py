"""Parity of the fused decode path (C ABI, CUDA) with the fp64 CPU oracle.

Every comparison is element by element with |out - ref| <= 2e-3 + 1e-2 |ref|
(see tests/_util.py), on seeded synthetic inputs, through the C ABI.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import token_decode_attention_gb300 as dattn
from token_decode_attention_gb300 import _native
from token_decode_attention_gb300.workloads import WORKLOADS, make_inputs

from ._util import assert_decode_close, cur_pos_tensor, rand_f16, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from token_decode_attention_gb300 import build
    build.build()
    dattn.load()
    yield
    assert dattn.dattn_device_error(clear=True) == 0, "a kernel recorded a pipeline timeout"


def run_case(B, H, D, S, cp, seed, num_partitions=0, scale=1.0):
    g = torch.Generator(device="cuda").manual_seed(seed)
    q = rand_f16(g, (B, H, D), scale=scale)
    k = rand_f16(g, (B, S, H, D), scale=scale)
    v = rand_f16(g, (B, S, H, D))
    cpt = cur_pos_tensor(cp)
    out = dattn.decode(q, k, v, cpt, num_partitions=num_partitions)
    torch.cuda.synchronize()
    ref = oracle.decode_f64(to_np(q), to_np(k), to_np(v), np.asarray(cp, np.uint32))
    return q, k, v, cpt, out, ref


# shapes spanning several CTAs, stages and a ragged tail; every head_dim class
SHAPES = [
    # B, H, D, S, current_pos per sequence
    (1, 12, 64, 64, [63]),            # the page's test shape
    (1, 12, 64, 64, [31]),            # the page's causal-mask test
    (1, 8, 48, 35, [34]),             # the page's awkward dimensions
    (1, 8, 64, 256, [200]),           # the small workload
    (3, 5, 8, 97, [0, 50, 96]),
    (2, 3, 16, 300, [299, 17]),
    (2, 7, 32, 513, [512, 100]),
    (4, 32, 128, 1000, [999, 0, 517, 5000]),
    (2, 40, 128, 777, [776, 300]),
    (2, 4, 96, 130, [129, 64]),
    (2, 6, 192, 70, [69, 3]),
    (2, 16, 256, 150, [149, 88]),
    (1, 64, 256, 40, [39]),            # two head groups
    (2, 64, 256, 600, [599, 300]),     # head groups over many full stages (tensor boxes)
    (2, 80, 256, 301, [300, 41]),      # three groups, the last one smaller (per-position copies)
    (1, 128, 128, 500, [499]),         # 128 heads at head_dim 128: two groups of 64
    (1, 200, 64, 20, [19]),            # two head groups at head_dim 64
    (3, 1, 8, 1000, [999, 1, 400]),    # one head, many phases
    (5, 2, 128, 1, [0, 0, 7, 0, 0]),   # seq_len 1
]


@pytest.mark.parametrize("B,H,D,S,cp", SHAPES, ids=[f"B{s[0]}H{s[1]}D{s[2]}S{s[3]}" for s in SHAPES])
def test_decode_matches_oracle(B, H, D, S, cp):
    *_, out, ref = run_case(B, H, D, S, cp, seed=B * 7919 + H * 31 + D * 7 + S)
    assert_decode_close(out, ref, f"B={B} H={H} D={D} S={S}")


@pytest.mark.parametrize("num_partitions", [1, 2, 3, 7, 64, 10_000])
def test_forced_split_counts_agree(num_partitions):
    B, H, D, S, cp = 3, 32, 128, 1200, [1199, 333, 0]
    *_, out, ref = run_case(B, H, D, S, cp, seed=99, num_partitions=num_partitions)
    assert_decode_close(out, ref, f"num_partitions={num_partitions}")
    base = run_case(B, H, D, S, cp, seed=99, num_partitions=1)[4]
    # any two split counts differ only by fp32 rounding order: at most one f16 step
    diff = (out.float() - base.float()).abs()
    ulp = torch.clamp(base.float().abs(), min=2.0**-14) * 2.0**-10
    assert bool((diff <= ulp * 1.01).all())


PIECE_SHAPES = [
    (5, 8, 64, 300, [299, 0, 150, 17, 260]),       # several lane groups per head
    (3, 64, 256, 100, [99, 5, 50]),                # two head groups per sequence
    (6, 40, 128, 200, [199, 3, 77, 150, 0, 120]),  # two heads per lane group
    (40, 4, 32, 30, list(range(0, 40))),           # many short units per partition
]


@pytest.mark.parametrize("partitions", [1, 3, 13, 100])
@pytest.mark.parametrize("B,H,D,S,cp", PIECE_SHAPES,
                         ids=[f"B{s[0]}H{s[1]}D{s[2]}S{s[3]}" for s in PIECE_SHAPES])
def test_partitions_cut_units_anywhere(B, H, D, S, cp, partitions):
    # ranges that start and end inside units, span several units, or hold
    # nothing at all, all merge to the same result
    *_, out, ref = run_case(B, H, D, S, cp, seed=B + H + D + S + partitions,
                            num_partitions=partitions)
    assert_decode_close(out, ref, f"partitions={partitions}")


def test_large_scores_outlier_channels():
    # scores of ~15 and beyond: exp overflows f16, so nothing may be kept in f16
    B, H, D, S, cp = 2, 8, 128, 600, [599, 250]
    g = torch.Generator(device="cuda").manual_seed(5)
    q = rand_f16(g, (B, H, D))
    k = rand_f16(g, (B, S, H, D))
    v = rand_f16(g, (B, S, H, D))
    k[..., :4] *= 20
    q[..., :4] *= 3
    cpt = cur_pos_tensor(cp)
    out = dattn.decode(q, k, v, cpt)
    ref = oracle.decode_f64(to_np(q), to_np(k), to_np(v), np.asarray(cp, np.uint32))
    assert_decode_close(out, ref, "outlier channels")


def test_single_live_position_is_v0_bit_exact():
    B, H, D, S = 4, 6, 64, 50
    g = torch.Generator(device="cuda").manual_seed(3)
    q, k, v = rand_f16(g, (B, H, D), scale=4.0), rand_f16(g, (B, S, H, D)), rand_f16(g, (B, S, H, D))
    for ns in (0, 1, 5):
        out = dattn.decode(q, k, v, cur_pos_tensor([0] * B), num_partitions=ns)
        torch.cuda.synchronize()
        assert torch.equal(out, v[:, 0]), f"num_partitions={ns}"


def test_zero_query_gives_mean_of_live_v():
    B, H, D, S, cp = 3, 4, 128, 333, [332, 10, 0]
    g = torch.Generator(device="cuda").manual_seed(4)
    q = torch.zeros((B, H, D), dtype=torch.float16, device="cuda")
    k, v = rand_f16(g, (B, S, H, D)), rand_f16(g, (B, S, H, D))
    out = dattn.decode(q, k, v, cur_pos_tensor(cp))
    vn = to_np(v).astype(np.float64)
    ref = np.stack([vn[b, : cp[b] + 1].mean(axis=0) for b in range(B)])
    assert_decode_close(out, ref, "Q = 0")


@pytest.mark.parametrize("poison", ["nan", "inf", "huge"])
def test_masked_positions_are_never_read(poison):
    # positions past current_pos carry zero weight: poisoning them (even with
    # NaN, which 0 * NaN would propagate) leaves the output bit-identical
    B, H, D, S, cp = 3, 32, 128, 900, [899, 400, 13]
    g = torch.Generator(device="cuda").manual_seed(6)
    q, k, v = rand_f16(g, (B, H, D)), rand_f16(g, (B, S, H, D)), rand_f16(g, (B, S, H, D))
    cpt = cur_pos_tensor(cp)
    for ns in (0, 1, 9):
        base = dattn.decode(q, k, v, cpt, num_partitions=ns).clone()
        k2, v2 = k.clone(), v.clone()
        fill = {"nan": float("nan"), "inf": float("inf"), "huge": 60000.0}[poison]
        for b in range(B):
            k2[b, cp[b] + 1:] = fill
            v2[b, cp[b] + 1:] = fill
        out = dattn.decode(q, k2, v2, cpt, num_partitions=ns)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), base.view(torch.int16)), f"num_partitions={ns}"


def test_current_pos_beyond_seq_len_masks_nothing():
    B, H, D, S = 2, 4, 64, 77
    cp = [76, 2**32 - 1]
    g = torch.Generator(device="cuda").manual_seed(8)
    q, k, v = rand_f16(g, (B, H, D)), rand_f16(g, (B, S, H, D)), rand_f16(g, (B, S, H, D))
    cpt = torch.tensor(np.array(cp, dtype=np.uint32).view(np.int32), device="cuda")
    out = dattn.decode(q, k, v, cpt)
    ref = oracle.decode_f64(to_np(q), to_np(k), to_np(v), np.array(cp, np.uint32))
    assert_decode_close(out, ref, "cp >= S")


def test_output_and_workspace_guard_bands():
    # out and workspace sit inside larger buffers filled with a sentinel; the
    # call may write only its own elements
    B, H, D, S, cp = 2, 32, 128, 2000, [1999, 700]
    g = torch.Generator(device="cuda").manual_seed(9)
    q, k, v = rand_f16(g, (B, H, D)), rand_f16(g, (B, S, H, D)), rand_f16(g, (B, S, H, D))
    cpt = cur_pos_tensor(cp)
    n_out = B * H * D
    pad = 4096
    big = torch.full((pad + n_out + pad,), 1234.0, dtype=torch.float16, device="cuda")
    out = big[pad:pad + n_out].view(B, H, D)
    ws_bytes = dattn.dattn_decode_workspace_bytes(B, H, D, S, 16)
    assert ws_bytes > 0
    ws_big = torch.full(((1 << 16) + ws_bytes + (1 << 16),), 0x5A, dtype=torch.uint8, device="cuda")
    ws = ws_big[1 << 16:(1 << 16) + ws_bytes]
    dattn.dattn_decode_f16_ex(q, k, v, out, cpt, ws, 16)
    torch.cuda.synchronize()
    assert bool((big[:pad] == 1234.0).all()) and bool((big[pad + n_out:] == 1234.0).all())
    assert bool((ws_big[: 1 << 16] == 0x5A).all())
    assert bool((ws_big[(1 << 16) + ws_bytes:] == 0x5A).all())
    ref = oracle.decode_f64(to_np(q), to_np(k), to_np(v), np.asarray(cp, np.uint32))
    assert_decode_close(out, ref, "guarded out")


def test_library_workspace_entry_point_matches_ex():
    B, H, D, S, cp = 4, 32, 128, 3000, [2999, 1000, 5, 2500]
    g = torch.Generator(device="cuda").manual_seed(10)
    q, k, v = rand_f16(g, (B, H, D)), rand_f16(g, (B, S, H, D)), rand_f16(g, (B, S, H, D))
    cpt = cur_pos_tensor(cp)
    ref = dattn.decode(q, k, v, cpt)
    out = torch.empty_like(ref)
    dattn.dattn_decode_f16(q, k, v, out, cpt)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)


def test_workspace_too_small_is_rejected_and_nothing_written():
    B, H, D, S, cp = 1, 32, 128, 4096, [4095]
    g = torch.Generator(device="cuda").manual_seed(11)
    q, k, v = rand_f16(g, (B, H, D)), rand_f16(g, (B, S, H, D)), rand_f16(g, (B, S, H, D))
    n = dattn.dattn_decode_workspace_bytes(B, H, D, S, 32)
    out = torch.full((B, H, D), 7.0, dtype=torch.float16, device="cuda")
    ws = torch.empty(n - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(_native.DattnError) as ei:
        dattn.dattn_decode_f16_ex(q, k, v, out, cur_pos_tensor([4095]), ws, 32)
    assert ei.value.status == _native.ERR_WORKSPACE
    torch.cuda.synchronize()
    assert bool((out == 7.0).all())


def test_non_contiguous_input_is_rejected():
    g = torch.Generator(device="cuda").manual_seed(12)
    k = rand_f16(g, (1, 16, 2, 64))
    q = rand_f16(g, (1, 64, 2)).transpose(1, 2)
    with pytest.raises(ValueError, match="contiguous"):
        dattn.decode(q, k, k, cur_pos_tensor([15]))


# -------------------------------------------------- the five seeded workloads

@pytest.mark.parametrize("name", ["small", "7b", "ragged"])
def test_workload_full_parity(name):
    w = WORKLOADS[name]
    x = make_inputs(w, "cuda")
    out = dattn.decode(x["q"], x["k"], x["v"], x["cur_pos"])
    torch.cuda.synchronize()
    ref = oracle.decode_f64(to_np(x["q"]), to_np(x["k"]), to_np(x["v"]), x["cur_pos_host"])
    assert_decode_close(out, ref, w.description)


@pytest.mark.slow
def test_workload_long_context_full_parity():
    w = WORKLOADS["long"]
    x = make_inputs(w, "cuda")
    out = dattn.decode(x["q"], x["k"], x["v"], x["cur_pos"])
    torch.cuda.synchronize()
    ref = oracle.decode_f64(to_np(x["q"]), to_np(x["k"]), to_np(x["v"]), x["cur_pos_host"])
    del x
    torch.cuda.empty_cache()
    assert_decode_close(out, ref, w.description)


@pytest.mark.slow
def test_workload_outlier_full_parity():
    # The whole 40 GiB workload (256 sequences x 40 heads) in the launch
    # configuration the benchmark uses, every output element against the fp64
    # oracle.  The inputs stay on the device; the oracle takes them a few
    # sequences at a time, so the host holds ~1.3 GB at once.
    w = WORKLOADS["outlier"]
    x = make_inputs(w, "cuda")
    out = dattn.decode(x["q"], x["k"], x["v"], x["cur_pos"])
    torch.cuda.synchronize()
    got = to_np(out)
    q = to_np(x["q"])
    step = 8
    for b0 in range(0, w.batch, step):
        sl = slice(b0, min(w.batch, b0 + step))
        ref = oracle.decode_f64(q[sl], to_np(x["k"][sl]), to_np(x["v"][sl]),
                                x["cur_pos_host"][sl])
        assert_decode_close(torch.from_numpy(got[sl]), ref,
                            f"{w.description}, sequences {sl.start}..{sl.stop - 1}")
    del x
    torch.cuda.empty_cache()


@pytest.mark.parametrize("partitions", [0, 7])
@pytest.mark.parametrize("B", [300, 5000])
def test_large_batches_take_every_prefix_path(B, partitions):
    # More sequences than threads per CTA: each prologue thread scans several
    # sequences.  Above 4096 sequences the merge kernel reads the prefix sums
    # the decode kernel wrote instead of summing current_pos itself.
    rng = np.random.default_rng(B + partitions)
    H, D, S = 2, 16, 24
    cp = rng.integers(0, S + 3, B).tolist()  # some beyond seq_len: nothing masked
    *_, out, ref = run_case(B, H, D, S, cp, seed=B * 7 + partitions, num_partitions=partitions)
    assert_decode_close(out, ref, f"B={B} partitions={partitions}")


@pytest.mark.parametrize("B,H,D,S,cp,partitions", [
    (2, 1, 112, 478, [89, 178], 288),     # W = 269 live positions < 288 partitions
    (4, 8, 64, 64, [0, 3, 1, 10], 40),    # W = 19 < 40
    (6, 4, 128, 512, [0, 0, 2, 0, 7, 1], 0),  # W = 16: fewer live positions than the plan's CTAs
    (2, 1, 112, 478, [89, 178], 100),     # W > G: every range holds positions
])
def test_empty_partitions_are_skipped_whatever_the_workspace_holds(B, H, D, S, cp, partitions):
    # With fewer live positions than partitions some ranges are empty, and an
    # empty one can lie between a sequence's first and last partition.  Its
    # workspace slot is not written by this call, so the merge must skip it:
    # the workspace is poisoned with NaN bytes first, and the result must still
    # match the oracle.
    g = torch.Generator(device="cuda").manual_seed(B * 31 + partitions)
    q, k, v = rand_f16(g, (B, H, D)), rand_f16(g, (B, S, H, D)), rand_f16(g, (B, S, H, D))
    n = max(16, dattn.dattn_decode_workspace_bytes(B, H, D, S, partitions))
    ws = torch.full((n,), 0xFF, dtype=torch.uint8, device="cuda")  # every float NaN
    out = dattn.decode(q, k, v, cur_pos_tensor(cp), num_partitions=partitions, workspace=ws)
    torch.cuda.synchronize()
    ref = oracle.decode_f64(to_np(q), to_np(k), to_np(v), np.asarray(cp, np.uint32))
    assert_decode_close(out, ref, f"W={sum(min(c, S - 1) + 1 for c in cp)} G={partitions}")


# few heads (rows of at most 4 KB per position): the split plan's larger
# stages, and the shapes where it keeps the smaller ones; B, H, D, S, current_pos
# (None: drawn uniformly per sequence)
FEW_HEAD_SHAPES = [
    (1, 1, 128, 131072, [100000]),
    (1, 4, 128, 65536, [50000]),
    (4, 1, 128, 65536, [65535, 65535, 65535, 65535]),
    (64, 8, 128, 2048, None),
    (4, 8, 256, 2048, None),
    (16, 8, 64, 1024, None),
]


@pytest.mark.parametrize("B,H,D,S,cp", FEW_HEAD_SHAPES,
                         ids=[f"B{c[0]}H{c[1]}D{c[2]}S{c[3]}" for c in FEW_HEAD_SHAPES])
def test_few_head_shapes(B, H, D, S, cp):
    g = torch.Generator(device="cuda").manual_seed(B * 7919 + H * 31 + D + S)
    if cp is None:
        cp = [int(x) for x in np.random.default_rng(B + S).integers(0, S, B)]
    q, k, v = rand_f16(g, (B, H, D)), rand_f16(g, (B, S, H, D)), rand_f16(g, (B, S, H, D))
    out = dattn.decode(q, k, v, cur_pos_tensor(cp))
    torch.cuda.synchronize()
    ref = oracle.decode_f64(to_np(q), to_np(k), to_np(v), np.asarray(cp, np.uint32))
    plan = dattn.dattn_decode_plan(B, H, D, S)
    assert_decode_close(out, ref, f"B={B} H={H} D={D} S={S} plan={plan}")
