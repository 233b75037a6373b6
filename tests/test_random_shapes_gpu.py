"""Seeded random shapes, dense and paged, against the fp64 oracle.

Three hundred cases drawn from one seed: every head_dim class (multiples of 8 up
to 256), head counts up to 80 (head groups included), ragged current_pos (some
beyond seq_len), the library's partition count or a forced one (often more
partitions than live positions, so some ranges are empty), and half of them
through a paged cache with a shuffled block table.  Sizes stay small enough for
the oracle (B*S*H*D <= 1.2e7).
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


def draw_cases(n=300, seed=20260101):
    rng = np.random.default_rng(seed)
    cases = []
    while len(cases) < n:
        D = int(rng.integers(1, 33)) * 8
        H = int(rng.choice([1, 2, 3, 5, 8, 12, 32, 40, 64, 80]))
        B = int(rng.integers(1, 7))
        S = int(rng.integers(1, 1500))
        if B * S * H * D > 1.2e7:
            continue
        cp = rng.integers(0, S + 3, B).tolist()
        live = sum(min(c, S - 1) + 1 for c in cp)
        r = rng.random()
        if r < 0.4:
            partitions = 0
        elif r < 0.7:  # more partitions than live positions: empty ranges
            partitions = int(rng.integers(live + 1, live + 300))
        else:
            partitions = int(rng.integers(1, 301))
        ps = int(rng.choice([1, 3, 8, 16, 64])) if rng.random() < 0.5 else 0
        cases.append((B, H, D, S, cp, partitions, ps, len(cases)))
    return cases


CASES = draw_cases()


@pytest.fixture(scope="module", autouse=True)
def _built():
    from token_decode_attention_gb300 import build
    build.build()
    dattn.load()
    yield
    assert dattn.dattn_device_error(clear=True) == _native.OK


@pytest.mark.parametrize("B,H,D,S,cp,partitions,ps,i", CASES,
                         ids=[f"{c[7]}-B{c[0]}H{c[1]}D{c[2]}S{c[3]}G{c[5]}ps{c[6]}" for c in CASES])
def test_random_shape_matches_oracle(B, H, D, S, cp, partitions, ps, i):
    g = torch.Generator(device="cuda").manual_seed(1000 + i)
    q = rand_f16(g, (B, H, D))
    cpn = np.asarray(cp, np.uint32)
    if not ps:
        k, v = rand_f16(g, (B, S, H, D)), rand_f16(g, (B, S, H, D))
        out = dattn.decode(q, k, v, cur_pos_tensor(cp), num_partitions=partitions)
        torch.cuda.synchronize()
        ref = oracle.decode_f64(to_np(q), to_np(k), to_np(v), cpn)
    else:
        maxp = (S + ps - 1) // ps
        num_pages = B * maxp + 3
        kp, vp = rand_f16(g, (num_pages, ps, H, D)), rand_f16(g, (num_pages, ps, H, D))
        table = np.random.default_rng(i).permutation(num_pages)[: B * maxp]
        table = table.reshape(B, maxp).astype(np.int32)
        out = dattn.decode_paged(q, kp, vp, torch.from_numpy(table).cuda(), cur_pos_tensor(cp),
                                 num_partitions=partitions)
        torch.cuda.synchronize()
        ref = oracle.decode_paged_f64(to_np(q), to_np(kp), to_np(vp), table, cpn)
    assert_decode_close(out, ref, f"case {i}")
