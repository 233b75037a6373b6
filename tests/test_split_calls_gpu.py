"""The page-faithful split calls (dattn_qk_f16, dattn_pv_f16) against the oracle.

dattn_qk_f16 restates attention_qk_f16 at the page's precision (sequential fp32
products and sums, fp32 scale, half rounding), so it must equal the oracle's
page-precision emulator bit for bit, with exactly -infinity at masked
positions.  dattn_pv_f16 is compared with the fp64 PV of the same f16 scores.
"""
from __future__ import annotations

import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import token_decode_attention_gb300 as dattn

from ._util import assert_decode_close, cur_pos_tensor, rand_f16, to_np

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module", autouse=True)
def _built():
    from token_decode_attention_gb300 import build
    build.build()
    dattn.load()


QK_SHAPES = [(1, 12, 64, 64, [63]), (1, 12, 64, 64, [31]), (1, 8, 48, 35, [34]),
             (3, 5, 8, 97, [0, 50, 96]), (2, 32, 128, 300, [299, 17]),
             (2, 4, 256, 40, [39, 1000])]


@pytest.mark.parametrize("B,H,D,S,cp", QK_SHAPES)
def test_qk_bit_exact_with_page_precision(B, H, D, S, cp):
    g = torch.Generator(device="cuda").manual_seed(B + H + D + S)
    q, k = rand_f16(g, (B, H, D)), rand_f16(g, (B, S, H, D))
    scores = dattn.qk(q, k, cur_pos_tensor(cp))
    torch.cuda.synchronize()
    ref = oracle.qk_pages_f16(to_np(q), to_np(k), np.asarray(cp, np.uint32))
    got = to_np(scores)
    assert np.array_equal(got.view(np.uint16), ref.view(np.uint16))
    pos = np.arange(S)
    for b in range(B):
        masked = pos > cp[b]
        assert (got[b][:, masked] == -np.inf).all()
        assert np.isfinite(got[b][:, ~masked]).all()


def _page_values(n):
    i = np.arange(n)
    return (np.float32(0.1) * (i % 10).astype(np.float32)).astype(np.float16)


def test_qk_page_test_inputs():
    spec = json.load(open(os.path.join(GOLDEN, "pages_qk_tests.json")))
    for case in spec["cases"]:
        H, D, S, cp = case["n_heads"], case["head_dim"], case["seq_len"], case["current_pos"]
        Q = _page_values(H * D).reshape(1, H, D)
        K = _page_values(S * H * D).reshape(1, S, H, D)
        scores = to_np(dattn.qk(torch.from_numpy(Q).cuda(), torch.from_numpy(K).cuda(),
                                cur_pos_tensor([cp])))
        qf = [Fraction(float(x)) for x in Q.reshape(-1)]
        kf = [Fraction(float(x)) for x in K.reshape(-1)]
        for h in range(H):
            for p in range(S):
                s = float(scores[0, h, p])
                if p > cp:
                    assert s == -math.inf, (case["name"], h, p)
                    continue
                exact = float(sum(qf[h * D + i] * kf[(p * H + h) * D + i] for i in range(D))) \
                    / math.sqrt(D)
                assert abs(s - exact) < spec["abs_tolerance"]
                assert abs(s - exact) <= 2.0 ** (math.floor(math.log2(max(abs(exact), 2**-14)))
                                                 - 11) + 1e-5 * abs(exact)


PV_SHAPES = [(1, 12, 64, 64, [63]), (1, 8, 48, 35, [20]), (2, 32, 128, 500, [499, 3]),
             (2, 4, 256, 3000, [2999, 1500])]


@pytest.mark.parametrize("B,H,D,S,cp", PV_SHAPES)
def test_pv_matches_fp64_on_same_scores(B, H, D, S, cp):
    g = torch.Generator(device="cuda").manual_seed(7 * B + H + D + S)
    q, k, v = rand_f16(g, (B, H, D)), rand_f16(g, (B, S, H, D)), rand_f16(g, (B, S, H, D))
    scores = dattn.qk(q, k, cur_pos_tensor(cp))
    out = dattn.pv(scores, v)
    torch.cuda.synchronize()
    ref = oracle.pv_f64(to_np(scores), to_np(v))
    assert_decode_close(out, ref, "pv")


def test_split_path_agrees_with_fused_path():
    # the two-dispatch form differs from the fused one only by the f16 rounding
    # of the scores; both stay within the decode tolerance of the fp64 oracle
    B, H, D, S, cp = 2, 8, 128, 700, [699, 123]
    g = torch.Generator(device="cuda").manual_seed(21)
    q, k, v = rand_f16(g, (B, H, D)), rand_f16(g, (B, S, H, D)), rand_f16(g, (B, S, H, D))
    cpt = cur_pos_tensor(cp)
    split = dattn.pv(dattn.qk(q, k, cpt), v)
    fused = dattn.decode(q, k, v, cpt)
    ref = oracle.decode_f64(to_np(q), to_np(k), to_np(v), np.asarray(cp, np.uint32))
    assert_decode_close(fused, ref, "fused")
    assert_decode_close(split, ref, "split")
