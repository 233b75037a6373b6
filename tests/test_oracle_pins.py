"""Pins for the CPU oracle: checks against things other than the oracle itself.

The oracle (``oracle/``) restates single-query decode attention from "Developing
Apple Metal Kernels in Rust - A Deep Dive Through Attention", section "The MSL,
briefly".  Here it is held to:
  * library routines: torch's scaled_dot_product_attention and softmax in fp64,
    numpy's IEEE float16 conversions;
  * exact rational arithmetic (fractions) on the page's own test inputs
    (section "Testing");
  * closed forms: one live position, two live positions (a sigmoid), constant V,
    identical K rows, Q = 0;
  * invariants: masked positions carry zero weight (even NaN there changes
    nothing), convex combination, permutation of live positions, independence of
    heads and sequences.
Every test here runs on the CPU.
"""
from __future__ import annotations

import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rand_f16(rng, shape, scale=1.0):
    return (rng.standard_normal(shape) * scale).astype(np.float16)


def sdpa_f64(Q, K, V, cp):
    """torch SDPA in fp64 with a boolean mask p <= cp (library routine)."""
    S = K.shape[1]
    q = torch.from_numpy(Q.astype(np.float64)).unsqueeze(2)
    k = torch.from_numpy(K.astype(np.float64)).permute(0, 2, 1, 3)
    v = torch.from_numpy(V.astype(np.float64)).permute(0, 2, 1, 3)
    pos = torch.arange(S)
    cpt = torch.from_numpy(np.asarray(cp, dtype=np.int64))
    mask = (pos[None, :] <= cpt[:, None])[:, None, None, :]
    return F.scaled_dot_product_attention(q, k, v, attn_mask=mask).squeeze(2).numpy()


# ---------------------------------------------------------------- conversions

def test_f16_decode_every_bit_pattern():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.f16_bits_to_f64(bits)
    ref = bits.view(np.float16).astype(np.float64)
    assert np.array_equal(got, ref, equal_nan=True)
    assert np.array_equal(np.signbit(got), np.signbit(ref))


def test_f32_to_f16_round_to_nearest_even():
    rng = np.random.default_rng(1)
    raw = rng.integers(0, 2**32, size=400_000, dtype=np.uint64).astype(np.uint32)
    vals = raw.view(np.float32)
    # values concentrated in and around binary16's range, plus exact ties
    near = (rng.standard_normal(200_000) * np.exp2(rng.uniform(-30, 18, 200_000)))
    ties = []
    for e in range(-24, 16):
        ulp = 2.0 ** max(e - 10, -24)
        base = 2.0 ** e
        ties += [base + ulp / 2, base + 1.5 * ulp, base + ulp / 2 * 1.0000001,
                 base + ulp / 2 * 0.9999999]
    special = [0.0, -0.0, 65504.0, 65519.99, 65520.0, 65536.0, 1e10, 2**-24, 2**-25,
               2**-25 * 1.0000001, 3 * 2**-26, 2**-14, 2**-14 - 2**-25, np.inf, -np.inf,
               np.nan]
    x = np.concatenate([vals, near.astype(np.float32), np.array(ties, np.float32),
                        np.array(special, np.float32), -np.array(ties, np.float32)])
    got = oracle.f32_to_f16_bits(x)
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    nan = np.isnan(x)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.isnan(got[nan].view(np.float16)).all()


# ------------------------------------------------------------ library routine

@pytest.mark.parametrize("D,S,H", [(1, 1, 1), (8, 7, 3), (48, 35, 8), (64, 64, 12),
                                   (64, 17, 2), (128, 40, 4)])
def test_decode_matches_torch_sdpa_every_current_pos(D, S, H):
    rng = np.random.default_rng(D * 1000 + S * 10 + H)
    B = S + 2                      # one sequence per current_pos 0..S+1
    cp = np.arange(B, dtype=np.uint32)
    Q, K, V = rand_f16(rng, (B, H, D)), rand_f16(rng, (B, S, H, D)), rand_f16(rng, (B, S, H, D))
    got = oracle.decode_f64(Q, K, V, cp)
    ref = sdpa_f64(Q, K, V, cp)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_decode_matches_sdpa_large_scores():
    # scores of size ~15 and more, the regime where max subtraction matters
    rng = np.random.default_rng(7)
    B, S, H, D = 4, 50, 3, 64
    Q = rand_f16(rng, (B, H, D), 3.0)
    K = rand_f16(rng, (B, S, H, D), 3.0)
    V = rand_f16(rng, (B, S, H, D))
    cp = np.array([0, 10, 49, 1000], np.uint32)
    np.testing.assert_allclose(oracle.decode_f64(Q, K, V, cp), sdpa_f64(Q, K, V, cp),
                               rtol=1e-11, atol=1e-12)


def test_pv_matches_torch_softmax():
    rng = np.random.default_rng(11)
    B, H, S, D = 3, 4, 37, 24
    scores = rand_f16(rng, (B, H, S), 2.0)
    scores[0, 1, 5:] = -np.inf
    scores[2, :, ::3] = -np.inf
    V = rand_f16(rng, (B, S, H, D))
    got = oracle.pv_f64(scores, V)
    w = torch.softmax(torch.from_numpy(scores.astype(np.float64)), dim=-1)     # B,H,S
    ref = torch.einsum("bhs,bshd->bhd", w, torch.from_numpy(V.astype(np.float64))).numpy()
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-13)


# ------------------------------------------------------------- closed forms

def test_single_live_position_returns_v0_exactly():
    rng = np.random.default_rng(2)
    B, S, H, D = 3, 9, 5, 32
    Q, K, V = rand_f16(rng, (B, H, D), 4.0), rand_f16(rng, (B, S, H, D)), rand_f16(rng, (B, S, H, D))
    out = oracle.decode_f64(Q, K, V, np.zeros(B, np.uint32))
    assert np.array_equal(out, V[:, 0].astype(np.float64))


def test_zero_query_gives_mean_of_live_v():
    rng = np.random.default_rng(3)
    B, S, H, D = 5, 33, 4, 16
    Q = np.zeros((B, H, D), np.float16)
    K, V = rand_f16(rng, (B, S, H, D)), rand_f16(rng, (B, S, H, D))
    cp = np.array([0, 1, 16, 32, 99], np.uint32)
    out = oracle.decode_f64(Q, K, V, cp)
    for b in range(B):
        L = min(int(cp[b]), S - 1) + 1
        ref = V[b, :L].astype(np.float64).mean(axis=0)
        np.testing.assert_allclose(out[b], ref, rtol=1e-12, atol=1e-15)


def test_two_live_positions_sigmoid_exact_scores():
    rng = np.random.default_rng(4)
    H, D, S = 3, 16, 6
    Q, K, V = rand_f16(rng, (1, H, D), 2.0), rand_f16(rng, (1, S, H, D), 2.0), rand_f16(rng, (1, S, H, D))
    out = oracle.decode_f64(Q, K, V, np.array([1], np.uint32))
    for h in range(H):
        # exact rational scores; sqrt(16) = 4
        s = [sum(Fraction(float(Q[0, h, i])) * Fraction(float(K[0, p, h, i])) for i in range(D)) / 4
             for p in range(2)]
        d01 = float(s[0] - s[1])
        w0 = 1.0 / (1.0 + math.exp(-d01))
        w1 = 1.0 / (1.0 + math.exp(d01))
        ref = w0 * V[0, 0, h].astype(np.float64) + w1 * V[0, 1, h].astype(np.float64)
        np.testing.assert_allclose(out[0, h], ref, rtol=1e-13, atol=1e-15)


def test_constant_v_and_identical_k_rows():
    rng = np.random.default_rng(5)
    B, S, H, D = 2, 21, 3, 8
    Q, K = rand_f16(rng, (B, H, D), 3.0), rand_f16(rng, (B, S, H, D), 3.0)
    vrow = rand_f16(rng, (B, 1, H, D))
    V = np.repeat(vrow, S, axis=1)
    cp = np.array([20, 7], np.uint32)
    out = oracle.decode_f64(Q, K, V, cp)
    np.testing.assert_allclose(out, vrow[:, 0].astype(np.float64), rtol=1e-14, atol=1e-15)
    # identical K rows: uniform weights, out = mean of live V
    K2 = np.repeat(rand_f16(rng, (B, 1, H, D), 3.0), S, axis=1)
    V2 = rand_f16(rng, (B, S, H, D))
    out2 = oracle.decode_f64(Q, K2, V2, cp)
    for b in range(B):
        L = int(cp[b]) + 1
        np.testing.assert_allclose(out2[b], V2[b, :L].astype(np.float64).mean(axis=0),
                                   rtol=1e-12, atol=1e-15)


# --------------------------------------------------------------- invariants

@pytest.mark.parametrize("poison", ["random", "huge", "nan", "inf"])
def test_masked_positions_have_zero_weight(poison):
    rng = np.random.default_rng(6)
    B, S, H, D = 3, 40, 4, 32
    Q, K, V = rand_f16(rng, (B, H, D)), rand_f16(rng, (B, S, H, D)), rand_f16(rng, (B, S, H, D))
    cp = np.array([0, 17, 38], np.uint32)
    base = oracle.decode_f64(Q, K, V, cp)
    K2, V2 = K.copy(), V.copy()
    for b in range(B):
        L = int(cp[b]) + 1
        fill = {"random": rand_f16(rng, (S - L, H, D), 10.0),
                "huge": np.full((S - L, H, D), 60000.0, np.float16),
                "nan": np.full((S - L, H, D), np.nan, np.float16),
                "inf": np.full((S - L, H, D), np.inf, np.float16)}[poison]
        K2[b, L:] = fill
        V2[b, L:] = fill
    assert np.array_equal(oracle.decode_f64(Q, K2, V2, cp), base)


def test_output_is_convex_combination_of_live_v():
    rng = np.random.default_rng(8)
    B, S, H, D = 4, 30, 5, 16
    Q, K, V = rand_f16(rng, (B, H, D), 2.0), rand_f16(rng, (B, S, H, D), 2.0), rand_f16(rng, (B, S, H, D))
    cp = np.array([3, 29, 12, 0], np.uint32)
    out = oracle.decode_f64(Q, K, V, cp)
    for b in range(B):
        L = int(cp[b]) + 1
        lo = V[b, :L].astype(np.float64).min(axis=0)
        hi = V[b, :L].astype(np.float64).max(axis=0)
        assert (out[b] >= lo - 1e-12).all() and (out[b] <= hi + 1e-12).all()


def test_joint_permutation_of_live_positions():
    rng = np.random.default_rng(9)
    B, S, H, D = 2, 25, 3, 24
    Q, K, V = rand_f16(rng, (B, H, D), 2.0), rand_f16(rng, (B, S, H, D)), rand_f16(rng, (B, S, H, D))
    cp = np.array([24, 13], np.uint32)
    base = oracle.decode_f64(Q, K, V, cp)
    K2, V2 = K.copy(), V.copy()
    for b in range(B):
        L = int(cp[b]) + 1
        perm = rng.permutation(L)
        K2[b, :L] = K[b, perm]
        V2[b, :L] = V[b, perm]
    np.testing.assert_allclose(oracle.decode_f64(Q, K2, V2, cp), base, rtol=1e-13, atol=1e-15)


def test_heads_and_sequences_are_independent():
    rng = np.random.default_rng(10)
    B, S, H, D = 3, 12, 4, 8
    Q, K, V = rand_f16(rng, (B, H, D)), rand_f16(rng, (B, S, H, D)), rand_f16(rng, (B, S, H, D))
    cp = np.array([11, 5, 8], np.uint32)
    base = oracle.decode_f64(Q, K, V, cp)
    Q2, K2, V2 = Q.copy(), K.copy(), V.copy()
    Q2[1, 2] = rand_f16(rng, (D,))
    K2[1, :, 2] = rand_f16(rng, (S, D))
    V2[1, :, 2] = rand_f16(rng, (S, D))
    out = oracle.decode_f64(Q2, K2, V2, cp)
    keep = np.ones((B, H), bool)
    keep[1, 2] = False
    assert np.array_equal(out[keep], base[keep])
    assert not np.array_equal(out[1, 2], base[1, 2])


# ------------------------------------------------ the page's own test inputs

def _page_values(n):
    # f16::from_f32((i % 10) as f32 * 0.1): an fp32 product, then a half rounding
    i = np.arange(n)
    return (np.float32(0.1) * (i % 10).astype(np.float32)).astype(np.float16)


def _page_cases():
    with open(os.path.join(GOLDEN, "pages_qk_tests.json")) as f:
        return json.load(f)


@pytest.mark.parametrize("case", _page_cases()["cases"], ids=lambda c: c["name"])
def test_page_qk_inputs_exact_scores(case):
    spec = _page_cases()
    H, D, S, cp = case["n_heads"], case["head_dim"], case["seq_len"], case["current_pos"]
    Q = _page_values(H * D).reshape(1, H, D)
    K = _page_values(S * H * D).reshape(1, S, H, D)
    cpa = np.array([cp], np.uint32)
    s64 = oracle.qk_f64(Q, K, cpa)
    s16 = oracle.qk_pages_f16(Q, K, cpa).astype(np.float64)
    qf = [Fraction(float(x)) for x in Q.reshape(-1)]
    kf = [Fraction(float(x)) for x in K.reshape(-1)]
    sqrt_d = math.sqrt(D)
    for h in range(H):
        for p in range(S):
            if p > cp:
                assert s64[0, h, p] == -np.inf and s16[0, h, p] == -np.inf
                continue
            dot = sum(qf[h * D + i] * kf[(p * H + h) * D + i] for i in range(D))
            exact = float(dot) / sqrt_d
            assert abs(s64[0, h, p] - exact) <= 1e-13 * max(1.0, abs(exact))
            # page precision: one f16 rounding (half an ulp) plus fp32 rounding
            ulp16 = 2.0 ** (math.floor(math.log2(abs(exact))) - 10) if exact else 2.0**-24
            assert abs(s16[0, h, p] - exact) <= 0.5 * ulp16 + 1e-5 * abs(exact) + 2.0**-24
            assert abs(s16[0, h, p] - exact) < spec["abs_tolerance"]


def test_page_qk_single_channel_is_one_rounded_product():
    # head_dim = 1: scale is exactly 1 and the fp32 product of two halves is
    # exact, so the score is numpy's float16 rounding of that product
    rng = np.random.default_rng(12)
    B, S, H = 2, 50, 3
    Q, K = rand_f16(rng, (B, H, 1), 50.0), rand_f16(rng, (B, S, H, 1), 50.0)
    cp = np.array([49, 20], np.uint32)
    got = oracle.qk_pages_f16(Q, K, cp)
    prod = Q[:, None, :, 0].astype(np.float32) * K[..., 0].astype(np.float32)  # B,S,H
    ref = prod.transpose(0, 2, 1).astype(np.float16)
    for b in range(B):
        ref[b, :, int(cp[b]) + 1:] = -np.inf
    assert np.array_equal(got.view(np.uint16), ref.view(np.uint16))


def test_page_qk_within_half_ulp_of_fp64():
    rng = np.random.default_rng(13)
    B, S, H, D = 2, 33, 5, 64
    Q, K = rand_f16(rng, (B, H, D)), rand_f16(rng, (B, S, H, D))
    cp = np.array([32, 9], np.uint32)
    s16 = oracle.qk_pages_f16(Q, K, cp).astype(np.float64)
    s64 = oracle.qk_f64(Q, K, cp)
    live = np.isfinite(s64)
    assert (s16[~live] == -np.inf).all() and (s64[~live] == -np.inf).all()
    mag = np.abs(s64[live])
    ulp16 = np.exp2(np.floor(np.log2(np.maximum(mag, 2.0**-14))) - 10)
    bound = np.abs(Q).max() * np.abs(K).max() * D * 2.0**-23 / 8 + 0.5 * ulp16 + 2.0**-24
    assert (np.abs(s16[live] - s64[live]) <= bound).all()


def test_pv_closed_forms():
    rng = np.random.default_rng(14)
    B, H, S, D = 2, 3, 19, 8
    V = rand_f16(rng, (B, S, H, D))
    # equal scores everywhere: the mean over all S positions
    out = oracle.pv_f64(np.zeros((B, H, S), np.float16), V)
    np.testing.assert_allclose(out, V.astype(np.float64).mean(axis=1), rtol=1e-12, atol=1e-15)
    # one finite score, the rest -inf: exactly that row of V
    sc = np.full((B, H, S), -np.inf, np.float16)
    sc[:, :, 7] = 3.0
    assert np.array_equal(oracle.pv_f64(sc, V), V[:, 7].astype(np.float64))


def test_qk_f64_square_head_dims_exact():
    rng = np.random.default_rng(15)
    for D in (1, 4, 16, 64):
        B, S, H = 1, 6, 2
        Q, K = rand_f16(rng, (B, H, D), 2.0), rand_f16(rng, (B, S, H, D), 2.0)
        got = oracle.qk_f64(Q, K, np.array([4], np.uint32))
        r = int(math.isqrt(D))
        for h in range(H):
            for p in range(S):
                if p > 4:
                    assert got[0, h, p] == -np.inf
                    continue
                exact = sum(Fraction(float(Q[0, h, i])) * Fraction(float(K[0, p, h, i]))
                            for i in range(D)) / r
                assert abs(got[0, h, p] - float(exact)) <= 1e-14 * max(1.0, abs(float(exact)))


# --------------------------------------------------------- paged KV cache

def _paged_case(rng, B, H, D, ps, maxp, extra_pages=3, share=False):
    num_pages = B * maxp + extra_pages
    Kp = rand_f16(rng, (num_pages, ps, H, D))
    Vp = rand_f16(rng, (num_pages, ps, H, D))
    table = rng.permutation(num_pages)[: B * maxp].reshape(B, maxp).astype(np.int32)
    if share and B > 1:
        table[1, :2] = table[0, :2]  # a shared prefix: two sequences read the same pages
    return Kp, Vp, table


def _gather_dense(pages, table, ps):
    # the logical cache K[b, p] = pages[table[b, p // ps], p % ps] (numpy indexing)
    B, maxp = table.shape
    p = np.arange(maxp * ps)
    return pages[table[:, p // ps], p % ps]          # [B, S, H, D]


def test_paged_identity_table_equals_dense():
    rng = np.random.default_rng(40)
    B, H, D, ps, maxp = 3, 4, 32, 8, 6
    S = ps * maxp
    Q, K, V = rand_f16(rng, (B, H, D)), rand_f16(rng, (B, S, H, D)), rand_f16(rng, (B, S, H, D))
    Kp = K.reshape(B * maxp, ps, H, D)
    Vp = V.reshape(B * maxp, ps, H, D)
    table = np.arange(B * maxp, dtype=np.int32).reshape(B, maxp)
    cp = np.array([47, 9, 0], np.uint32)
    assert np.array_equal(oracle.decode_paged_f64(Q, Kp, Vp, table, cp),
                          oracle.decode_f64(Q, K, V, cp))


@pytest.mark.parametrize("ps", [1, 5, 16])
def test_paged_random_and_shared_tables_equal_dense_gather(ps):
    rng = np.random.default_rng(41 + ps)
    B, H, D, maxp = 4, 3, 16, 7
    Kp, Vp, table = _paged_case(rng, B, H, D, ps, maxp, share=True)
    Q = rand_f16(rng, (B, H, D))
    cp = np.array([ps * maxp - 1, 3, ps * maxp + 100, 0], np.uint32)
    dense = oracle.decode_f64(Q, _gather_dense(Kp, table, ps), _gather_dense(Vp, table, ps), cp)
    assert np.array_equal(oracle.decode_paged_f64(Q, Kp, Vp, table, cp), dense)


def test_paged_unreferenced_and_past_live_pages_do_not_matter():
    rng = np.random.default_rng(45)
    B, H, D, ps, maxp = 2, 2, 8, 4, 5
    Kp, Vp, table = _paged_case(rng, B, H, D, ps, maxp, extra_pages=4)
    Q = rand_f16(rng, (B, H, D))
    cp = np.array([5, 10], np.uint32)  # live pages: 0..1 and 0..2
    base = oracle.decode_paged_f64(Q, Kp, Vp, table, cp)
    used = set(table[0, :2].tolist()) | set(table[1, :3].tolist())
    Kp2, Vp2 = Kp.copy(), Vp.copy()
    for pg in range(Kp.shape[0]):
        if pg not in used:
            Kp2[pg] = np.nan
            Vp2[pg] = np.nan
    table2 = table.copy()
    table2[0, 2:] = -7          # invalid entries past the live pages are never looked at
    table2[1, 3:] = 10**6
    assert np.array_equal(oracle.decode_paged_f64(Q, Kp2, Vp2, table2, cp), base)


def test_paged_invalid_live_page_gives_nan_row_only_for_that_sequence():
    rng = np.random.default_rng(46)
    B, H, D, ps, maxp = 3, 2, 8, 4, 3
    Kp, Vp, table = _paged_case(rng, B, H, D, ps, maxp)
    Q = rand_f16(rng, (B, H, D))
    cp = np.array([11, 11, 11], np.uint32)
    good = oracle.decode_paged_f64(Q, Kp, Vp, table, cp)
    table[1, 1] = Kp.shape[0]  # out of range
    got = oracle.decode_paged_f64(Q, Kp, Vp, table, cp)
    assert np.isnan(got[1]).all()
    assert np.array_equal(got[[0, 2]], good[[0, 2]])


# ---------------------------------------------------------- row softmax

def test_softmax_matches_torch_fp64():
    rng = np.random.default_rng(50)
    x = (rng.standard_normal((37, 129)) * 6).astype(np.float32)
    x[3, ::2] = -np.inf
    x[5, :] = -np.inf
    x[5, 7] = 2.0
    ref = torch.softmax(torch.from_numpy(x.astype(np.float64)), dim=-1).numpy()
    np.testing.assert_allclose(oracle.softmax_f64(x), ref, rtol=1e-13, atol=1e-300)


def test_softmax_closed_forms_and_invariants():
    rng = np.random.default_rng(51)
    # constant row: uniform weights
    assert np.array_equal(oracle.softmax_f64(np.full((2, 8), 3.5, np.float32)),
                          np.full((2, 8), 1 / 8))
    # shifting a row changes nothing (up to rounding); rows sum to one
    x = rng.standard_normal((6, 50)).astype(np.float32)
    a = oracle.softmax_f64(x)
    b = oracle.softmax_f64(x + np.float32(1000.0))
    np.testing.assert_allclose(a, b, rtol=1e-4, atol=0)  # x + 1000 rounds in float32
    np.testing.assert_allclose(a.sum(axis=1), 1.0, rtol=1e-14)
    # two entries: a sigmoid of their difference
    y = np.array([[0.25, -1.5]], np.float32)
    d = float(y[0, 0]) - float(y[0, 1])
    np.testing.assert_allclose(oracle.softmax_f64(y)[0],
                               [1 / (1 + math.exp(-d)), 1 / (1 + math.exp(d))], rtol=1e-15)
    # -inf entries get weight exactly 0; a row far above the rest is one-hot
    w = np.array([[0.5, -np.inf, 1.0, -np.inf], [1000.0, 0.0, -3.0, 2.0]], np.float32)
    ow = oracle.softmax_f64(w)
    assert ow[0, 1] == 0.0 and ow[0, 3] == 0.0
    np.testing.assert_allclose(ow[0, [0, 2]], [1 / (1 + math.exp(0.5)), 1 / (1 + math.exp(-0.5))],
                               rtol=1e-15)
    assert np.array_equal(ow[1], [1.0, 0.0, 0.0, 0.0])
    # all -inf or a NaN gives NaN for that row only
    z = rng.standard_normal((3, 4)).astype(np.float32)
    z[0] = -np.inf
    z[2, 1] = np.nan
    o = oracle.softmax_f64(z)
    assert np.isnan(o[0]).all() and np.isnan(o[2]).all() and np.isfinite(o[1]).all()


# ------------------------------------------------------- rotary embedding

def _rope_complex(x64, pos, rd, base, traditional):
    # the same rotation as complex multiplication by exp(i a), with numpy
    B, H, D = x64.shape
    half = rd // 2
    # theta_i from C's pow (math.pow), not numpy's vectorised power: at positions
    # near 2^31 a one-ulp difference in theta moves the angle by ~2e-7 rad
    theta = np.array([math.pow(base, -2.0 * i / rd) for i in range(half)])
    a = np.asarray(pos, np.float64)[:, None, None] * theta[None, None, :]
    if traditional:
        z = x64[..., 0:rd:2] + 1j * x64[..., 1:rd:2]
    else:
        z = x64[..., :half] + 1j * x64[..., half:rd]
    z = z * np.exp(1j * a)
    out = x64.copy()
    if traditional:
        out[..., 0:rd:2], out[..., 1:rd:2] = z.real, z.imag
    else:
        out[..., :half], out[..., half:rd] = z.real, z.imag
    return out


@pytest.mark.parametrize("traditional", [False, True])
@pytest.mark.parametrize("rd", [8, 64, 128])
def test_rope_equals_complex_rotation(traditional, rd):
    rng = np.random.default_rng(60 + rd)
    x = rand_f16(rng, (4, 4, 128))
    pos = np.array([0, 17, 131071, 2**31 - 1], np.uint32)
    got = oracle.rope_f64(x, pos, rd, 10000.0, traditional)
    ref = _rope_complex(x.astype(np.float64), pos, rd, 10000.0, traditional)
    np.testing.assert_allclose(got, ref, rtol=1e-9, atol=1e-9)


def test_rope_position_zero_is_identity_and_norms_are_kept():
    # the page-1 engine's RoPE tests: position zero is the identity, and
    # different positions differ; a rotation keeps each pair's norm
    rng = np.random.default_rng(61)
    x = rand_f16(rng, (2, 3, 64))
    assert np.array_equal(oracle.rope_f64(x, [0, 0]), x.astype(np.float64))
    r = oracle.rope_f64(x, [5, 900])
    assert not np.allclose(r, x.astype(np.float64))
    x64 = x.astype(np.float64)
    np.testing.assert_allclose(r[..., :32] ** 2 + r[..., 32:] ** 2,
                               x64[..., :32] ** 2 + x64[..., 32:] ** 2, rtol=1e-12)


def test_rope_scores_depend_on_relative_position_only():
    rng = np.random.default_rng(62)
    q, k = rand_f16(rng, (1, 1, 64)), rand_f16(rng, (1, 1, 64))
    s1 = float((oracle.rope_f64(q, [100]) * oracle.rope_f64(k, [40])).sum())
    s2 = float((oracle.rope_f64(q, [1060]) * oracle.rope_f64(k, [1000])).sum())
    assert abs(s1 - s2) <= 1e-9 * max(1.0, abs(s1))


def test_rope_leaves_channels_past_rope_dims_unchanged():
    rng = np.random.default_rng(63)
    x = rand_f16(rng, (2, 2, 96))
    r = oracle.rope_f64(x, [7, 3000], rope_dims=32)
    assert np.array_equal(r[..., 32:], x[..., 32:].astype(np.float64))
