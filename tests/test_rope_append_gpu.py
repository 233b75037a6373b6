"""Fused rotary embedding + KV append against the fp64 oracle.

dattn_rope_append_f16 rotates the new token's q and k at position
current_pos[b] ("Tutorial 16: Writing Custom Metal Kernels", section 5,
FastRoPE) and writes the rotated k and the new v into the cache row at that
position.  The oracle's rotation is pinned against a complex-exponential
rotation and the position invariants in tests/test_oracle_pins.py.

Bound, per element: one f16 ulp of the fp64 value (the single rounding to
f16) plus 1e-6 (|u| + |w|) for the element's pair (u, w).  The kernel reduces
p * theta modulo 2 pi exactly, as a wrapping integer product with theta / 2 pi
held as a 64-bit binary fraction, and takes fp32 cos/sin of the reduced angle
(angle error below 4e-7 rad), then rotates in fp32 (about 2e-7 relative to
|u| + |w|).  Channels past rope_dims are copied, so their bound is zero.
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


def f16_ulp(ref: np.ndarray) -> np.ndarray:
    """Spacing of float16 values at |ref| (2^-24 in the subnormal range)."""
    a = np.abs(ref)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a >= 2.0 ** -14, 2.0 ** (e - 10), 2.0 ** -24)


def pair_magnitude(x: np.ndarray, rope_dims: int, traditional: bool) -> np.ndarray:
    """|u| + |w| of the rotated pair each channel belongs to; 0 past rope_dims."""
    a = np.abs(x.astype(np.float64))
    m = np.zeros_like(a)
    half = rope_dims // 2
    if traditional:
        s = a[..., 0:rope_dims:2] + a[..., 1:rope_dims:2]
        m[..., 0:rope_dims:2] = s
        m[..., 1:rope_dims:2] = s
    else:
        s = a[..., :half] + a[..., half:rope_dims]
        m[..., :half] = s
        m[..., half:rope_dims] = s
    return m


def assert_rotated(got: torch.Tensor, ref: np.ndarray, x: np.ndarray, rope_dims: int,
                   traditional: bool, what: str):
    g = to_np(got).astype(np.float64)
    assert g.shape == ref.shape, what
    err = np.abs(g - ref)
    rd = rope_dims or ref.shape[-1]
    bound = f16_ulp(ref) * (np.arange(ref.shape[-1]) < rd) + \
        1e-6 * pair_magnitude(x, rd, traditional)
    bad = ~(err <= bound)
    if bad.any():
        i = tuple(np.argwhere(bad)[0])
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} out of bound; first at "
                             f"{i}: got {g[i]!r} ref {ref[i]!r} bound {bound[i]:.3g}")


def check_append(q, k_new, v_new, q_out, K0, V0, K, V, cp, rope_dims, base, traditional,
                 rows_of):
    """rows_of(b) -> (cache index tuple of sequence b's new row) or None if not written."""
    rd = rope_dims or q.shape[2]
    ref_q = oracle.rope_f64(to_np(q), cp, rd, base, traditional)
    ref_k = oracle.rope_f64(to_np(k_new), cp, rd, base, traditional)
    assert_rotated(q_out, ref_q, to_np(q), rd, traditional, "rotated q")
    Kc, Vc, K0c, V0c = (to_np(t).view(np.uint16) for t in (K, V, K0, V0))
    expect_k, expect_v = K0c.copy(), V0c.copy()
    for b in range(q.shape[0]):
        r = rows_of(b)
        if r is None:
            continue
        assert_rotated(K[r], ref_k[b], to_np(k_new[b]), rd, traditional,
                       f"appended k of sequence {b}")
        expect_k[r] = Kc[r]  # checked above
        expect_v[r] = to_np(v_new[b]).view(np.uint16)
    assert np.array_equal(Kc, expect_k), "a K cache row other than the appended ones changed"
    assert np.array_equal(Vc, expect_v), "V cache rows differ from the old cache + appended v"


CASES = [
    # B, H, D, S, rope_dims (0: all), traditional, base, current_pos
    (2, 8, 64, 32, 0, False, 10000.0, [0, 31]),
    (3, 32, 128, 300, 0, True, 10000.0, [5, 299, 100]),
    (4, 40, 128, 50, 64, False, 500000.0, [1, 2, 3, 49]),
    (2, 4, 256, 40, 0, True, 10000.0, [39, 17]),
    (3, 12, 96, 20, 32, True, 10000.0, [0, 10, 19]),
    (1, 2, 64, 131072, 0, False, 10000.0, [131071]),
    (2, 3, 64, 70000, 16, False, 1e6, [65537, 69999]),
    # rope_dims not a multiple of 8: one pair per work item, scalar pass-through
    (2, 5, 64, 24, 20, False, 10000.0, [23, 1]),
    (2, 5, 64, 24, 36, True, 10000.0, [12, 0]),
    (3, 9, 32, 8, 2, False, 10000.0, [7, 6, 5]),
    (2, 4, 48, 10, 0, True, 10000.0, [9, 4]),
]


@pytest.mark.parametrize("B,H,D,S,rd,trad,base,cp", CASES,
                         ids=[f"B{c[0]}H{c[1]}D{c[2]}S{c[3]}rd{c[4]}{'t' if c[5] else 'n'}"
                              for c in CASES])
def test_rope_append_matches_oracle(B, H, D, S, rd, trad, base, cp):
    g = torch.Generator(device="cuda").manual_seed(B * 1000 + H + D + S)
    q, kn, vn = (rand_f16(g, (B, H, D), scale=2.0) for _ in range(3))
    K0, V0 = rand_f16(g, (B, S, H, D)), rand_f16(g, (B, S, H, D))
    K, V = K0.clone(), V0.clone()
    qo = dattn.rope_append(q, kn, vn, K, V, cur_pos_tensor(cp), rd, base, trad)
    torch.cuda.synchronize()
    check_append(q, kn, vn, qo, K0, V0, K, V, cp, rd, base, trad, lambda b: (b, cp[b]))


def test_rotation_in_place_on_q():
    g = torch.Generator(device="cuda").manual_seed(3)
    B, H, D, S, cp = 3, 16, 128, 64, [7, 63, 0]
    q, kn, vn = (rand_f16(g, (B, H, D)) for _ in range(3))
    q0 = q.clone()
    K, V = rand_f16(g, (B, S, H, D)), rand_f16(g, (B, S, H, D))
    out = dattn.rope_append(q, kn, vn, K, V, cur_pos_tensor(cp), q_out=q)
    torch.cuda.synchronize()
    assert out is q
    assert_rotated(q, oracle.rope_f64(to_np(q0), cp), to_np(q0), 0, False, "in-place q")


@pytest.mark.parametrize("ps,trad", [(16, False), (1, True), (7, False)])
def test_paged_append_writes_the_page_row(ps, trad):
    g = torch.Generator(device="cuda").manual_seed(ps)
    B, H, D, maxp = 3, 8, 128, 6
    num_pages = B * maxp + 4
    q, kn, vn = (rand_f16(g, (B, H, D)) for _ in range(3))
    K0, V0 = rand_f16(g, (num_pages, ps, H, D)), rand_f16(g, (num_pages, ps, H, D))
    K, V = K0.clone(), V0.clone()
    table = np.random.default_rng(ps).permutation(num_pages)[: B * maxp].reshape(B, maxp)
    table = table.astype(np.int32)
    cp = [ps * maxp - 1, ps * 2 + ps // 2, 0]
    qo = dattn.rope_append(q, kn, vn, K, V, cur_pos_tensor(cp), traditional=trad,
                           block_table=torch.from_numpy(table).cuda())
    torch.cuda.synchronize()
    check_append(q, kn, vn, qo, K0, V0, K, V, cp, 0, 10000.0, trad,
                 lambda b: (int(table[b, cp[b] // ps]), cp[b] % ps))


def test_position_outside_cache_is_reported_and_not_written():
    g = torch.Generator(device="cuda").manual_seed(11)
    B, H, D, S = 2, 8, 64, 16
    q, kn, vn = (rand_f16(g, (B, H, D)) for _ in range(3))
    K0, V0 = rand_f16(g, (B, S, H, D)), rand_f16(g, (B, S, H, D))
    K, V = K0.clone(), V0.clone()
    cp = [3, S]  # sequence 1 is full
    assert dattn.dattn_device_error(clear=True) == _native.OK
    qo = dattn.rope_append(q, kn, vn, K, V, cur_pos_tensor(cp))
    assert dattn.dattn_device_error(clear=True) == _native.ERR_BAD_POSITION
    check_append(q, kn, vn, qo, K0, V0, K, V, cp, 0, 10000.0, False,
                 lambda b: (b, cp[b]) if cp[b] < S else None)


def test_invalid_page_is_reported_and_not_written():
    g = torch.Generator(device="cuda").manual_seed(12)
    B, H, D, ps, maxp = 2, 8, 64, 16, 4
    num_pages = B * maxp
    q, kn, vn = (rand_f16(g, (B, H, D)) for _ in range(3))
    K0, V0 = rand_f16(g, (num_pages, ps, H, D)), rand_f16(g, (num_pages, ps, H, D))
    K, V = K0.clone(), V0.clone()
    table = np.arange(num_pages, dtype=np.int32).reshape(B, maxp)
    table[0, 2] = -1
    cp = [40, 40]
    assert dattn.dattn_device_error(clear=True) == _native.OK
    qo = dattn.rope_append(q, kn, vn, K, V, cur_pos_tensor(cp),
                           block_table=torch.from_numpy(table).cuda())
    assert dattn.dattn_device_error(clear=True) == _native.ERR_BAD_PAGE
    check_append(q, kn, vn, qo, K0, V0, K, V, cp, 0, 10000.0, False,
                 lambda b: None if b == 0 else (int(table[b, cp[b] // ps]), cp[b] % ps))


def test_append_then_decode_is_one_decode_step():
    # the step a decoder runs per token: rotate and append, then attend over
    # positions 0..current_pos including the new one
    g = torch.Generator(device="cuda").manual_seed(21)
    B, H, D, S, cp = 4, 32, 128, 512, [511, 0, 200, 33]
    q, kn, vn = (rand_f16(g, (B, H, D)) for _ in range(3))
    K, V = rand_f16(g, (B, S, H, D)), rand_f16(g, (B, S, H, D))
    K_host, V_host = to_np(K).copy(), to_np(V).copy()
    cpt = cur_pos_tensor(cp)
    q_rot = dattn.rope_append(q, kn, vn, K, V, cpt)
    out = dattn.decode(q_rot, K, V, cpt)
    torch.cuda.synchronize()
    # oracle inputs: its own rotation, rounded to the cache's f16
    q_ref = oracle.rope_f64(to_np(q), cp).astype(np.float16)
    k_ref = oracle.rope_f64(to_np(kn), cp).astype(np.float16)
    for b in range(B):
        K_host[b, cp[b]] = k_ref[b]
        V_host[b, cp[b]] = to_np(vn[b])
    ref = oracle.decode_f64(q_ref, K_host, V_host, np.asarray(cp, np.uint32))
    assert_decode_close(out, ref, "rope + append + decode")


def test_decode_steps_back_to_back_without_host_sync():
    # rope/append and decode (with its merge) are launched with programmatic
    # dependent launch: each kernel may begin launching before the one before it
    # ends and waits for it before reading.  Several decode steps issued back to
    # back on one stream, with every input staged beforehand and no host
    # synchronisation in between, must each see the rows appended by its own and
    # every earlier step.
    g = torch.Generator(device="cuda").manual_seed(33)
    B, H, D, S, steps = 2, 32, 128, 2048, 4
    start = [1500, 700]
    K, V = rand_f16(g, (B, S, H, D)), rand_f16(g, (B, S, H, D))
    K_host, V_host = to_np(K).copy(), to_np(V).copy()
    toks = [tuple(rand_f16(g, (B, H, D)) for _ in range(3)) for _ in range(steps)]
    cps = [[s + t for s in start] for t in range(steps)]
    cpts = [cur_pos_tensor(cp) for cp in cps]
    q_rots = [torch.empty((B, H, D), dtype=torch.float16, device="cuda") for _ in range(steps)]
    outs = [torch.empty((B, H, D), dtype=torch.float16, device="cuda") for _ in range(steps)]
    torch.cuda.synchronize()
    for t in range(steps):
        q, kn, vn = toks[t]
        dattn.rope_append(q, kn, vn, K, V, cpts[t], q_out=q_rots[t])
        dattn.decode(q_rots[t], K, V, cpts[t], out=outs[t])
    torch.cuda.synchronize()
    for t in range(steps):
        q, kn, vn = toks[t]
        cp = cps[t]
        k_ref = oracle.rope_f64(to_np(kn), cp).astype(np.float16)
        for b in range(B):
            K_host[b, cp[b]] = k_ref[b]
            V_host[b, cp[b]] = to_np(vn[b])
        q_ref = oracle.rope_f64(to_np(q), cp).astype(np.float16)
        ref = oracle.decode_f64(q_ref, K_host, V_host, np.asarray(cp, np.uint32))
        assert_decode_close(outs[t], ref, f"step {t}")
