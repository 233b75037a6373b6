"""Standalone row softmax (dattn_softmax_f32) against the fp64 oracle."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import token_decode_attention_gb300 as dattn

pytestmark = pytest.mark.gpu

# fp32 with expf: per element about 1e-6 relative; the row sum adds at most a
# few 1e-6 for the widths below.  Bound: |out - ref| <= 1e-7 + 2e-5 |ref|.
ATOL, RTOL = 1e-7, 2e-5


@pytest.fixture(scope="module", autouse=True)
def _built():
    from token_decode_attention_gb300 import build
    build.build()
    dattn.load()


def check(x: torch.Tensor, out: torch.Tensor):
    ref = oracle.softmax_f64(x.cpu().numpy())
    got = out.cpu().numpy().astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    err = np.abs(got[~nan] - ref[~nan])
    assert (err <= ATOL + RTOL * np.abs(ref[~nan])).all(), f"max err {err.max():.3g}"


# widths cover: one warp per row (<= 1024); one CTA per row held in registers
# (<= 8192) as float4 slots (cols % 4 == 0: 2, 4, 8 per thread) or scalar slots
# (8, 16, 32 per thread), and up to 16384 aligned columns with 512 threads;
# longer aligned rows: persistent CTAs (two per SM up to 65536 columns, one
# beyond); other long rows: two passes
@pytest.mark.parametrize("rows,cols", [(1, 1), (7, 5), (64, 32), (33, 1000), (5, 1024),
                                       (9, 1025), (6, 2052), (4, 4096), (2, 6000), (3, 8192),
                                       (5, 3001), (3, 8191), (2, 8193), (2, 8196),
                                       (3, 16384), (2, 16388), (3, 24580), (5, 32768),
                                       (3, 50000), (400, 65536), (3, 65540), (2, 131072),
                                       (2, 128256), (2, 196612), (2, 200001)])
def test_softmax_matches_oracle(rows, cols):
    g = torch.Generator(device="cuda").manual_seed(rows * 100003 + cols)
    x = torch.empty((rows, cols), dtype=torch.float32, device="cuda")
    x.normal_(0.0, 4.0, generator=g)
    out = dattn.softmax(x)
    torch.cuda.synchronize()
    check(x, out)


def test_softmax_masked_and_degenerate_rows():
    g = torch.Generator(device="cuda").manual_seed(3)
    for cols in (300, 5000, 5001, 9000, 9001, 60000):  # warp; CTA: float4, scalar; persistent; 2 passes
        x = torch.empty((6, cols), dtype=torch.float32, device="cuda")
        x.normal_(0.0, 3.0, generator=g)
        x[0, ::3] = float("-inf")          # masked entries: weight 0
        x[1] = float("-inf")               # all masked: NaN row
        x[2, 5] = float("nan")             # a NaN: NaN row
        x[3, 0] = float("-inf")
        x[3, 1:] = float("-inf")
        x[3, 7] = float("nan")             # -inf first, then a NaN: NaN row
        x[4] = 7.0                         # constant: uniform
        x[5] += 1000.0                     # large values: max subtraction
        out = dattn.softmax(x)
        torch.cuda.synchronize()
        check(x, out)
        assert float(out[0, 0]) == 0.0


def test_softmax_in_place_and_row_sums():
    g = torch.Generator(device="cuda").manual_seed(4)
    x = torch.empty((100, 2048), dtype=torch.float32, device="cuda")
    x.normal_(0.0, 2.0, generator=g)
    ref = x.clone()
    dattn.dattn_softmax_f32(x, x)  # out may equal x
    torch.cuda.synchronize()
    check(ref, x)
    assert torch.allclose(x.double().sum(dim=1).cpu(), torch.ones(100, dtype=torch.float64),
                          atol=1e-5)


def test_softmax_long_rows_with_masked_spans_and_nan():
    # 60000 columns (the persistent long-row kernel): a span of -infinity gets
    # weight exactly 0; a NaN inside such a span still turns its row into NaN;
    # a single live entry takes all the weight.
    g = torch.Generator(device="cuda").manual_seed(6)
    x = torch.empty((4, 60000), dtype=torch.float32, device="cuda")
    x.normal_(0.0, 3.0, generator=g)
    x[0, 20000:40000] = float("-inf")      # the middle slice masked
    x[1, 40000:] = float("-inf")           # the last slice masked
    x[2, 20000:40000] = float("-inf")
    x[2, 31000] = float("nan")             # ... with a NaN in it
    x[3, :] = float("-inf")
    x[3, 59999] = 5.0                      # one live entry in the last slice
    out = dattn.softmax(x)
    torch.cuda.synchronize()
    check(x, out)
    assert (out[0, 20000:40000] == 0).all() and (out[1, 40000:] == 0).all()
    assert torch.isnan(out[2]).all()
    assert abs(float(out[3, 59999]) - 1.0) <= 1e-6 and float(out[3, :59999].abs().max()) == 0.0


def _random_softmax_cases(n=40, seed=20260202):
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        cols = int(rng.choice([int(rng.integers(1, 1100)), int(rng.integers(1000, 20000)),
                               int(rng.integers(16000, 70000))]))
        rows = int(max(1, min(int(rng.integers(1, 300)), 4e6 // cols)))
        cases.append((rows, cols, bool(rng.random() < 0.3), i))  # 30 %: not 16-byte aligned
    return cases


@pytest.mark.parametrize("rows,cols,shifted,i", _random_softmax_cases(),
                         ids=[f"{c[3]}-{c[0]}x{c[1]}{'-shift' if c[2] else ''}"
                              for c in _random_softmax_cases()])
def test_softmax_random_shapes(rows, cols, shifted, i):
    # seeded widths across every path; "shifted" matrices start one float past a
    # 16-byte boundary, which takes the scalar forms
    g = torch.Generator(device="cuda").manual_seed(4000 + i)
    n = rows * cols
    buf = torch.empty((n + 1,), dtype=torch.float32, device="cuda")
    buf.normal_(0.0, 5.0, generator=g)
    x = buf[1:].view(rows, cols) if shifted else buf[:n].view(rows, cols)
    obuf = torch.empty_like(buf)
    out = obuf[1:].view(rows, cols) if shifted else obuf[:n].view(rows, cols)
    dattn.dattn_softmax_f32(x, out)
    torch.cuda.synchronize()
    check(x, out)


def test_softmax_very_long_rows_with_masked_halves_and_nan():
    # 160000 aligned columns (past 256 KB: one persistent 1024-thread CTA per
    # SM, the row re-read from L2): a masked span across the middle, a whole
    # half masked either side, a NaN in the second half only, and a single
    # live entry in the first half.
    g = torch.Generator(device="cuda").manual_seed(7)
    x = torch.empty((5, 160000), dtype=torch.float32, device="cuda")
    x.normal_(0.0, 3.0, generator=g)
    x[0, 60000:100000] = float("-inf")     # across the middle
    x[1, 80000:] = float("-inf")           # the second half masked
    x[2, 120000] = float("nan")            # a NaN in the second half only
    x[3, :] = float("-inf")
    x[3, 12345] = 2.0                      # one live entry, first half
    x[4, :80000] = float("-inf")           # the first half masked
    out = dattn.softmax(x)
    torch.cuda.synchronize()
    check(x, out)
    assert (out[0, 60000:100000] == 0).all() and (out[1, 80000:] == 0).all()
    assert torch.isnan(out[2]).all() and not torch.isnan(out[4]).any()
    assert abs(float(out[3, 12345]) - 1.0) <= 1e-6 and float(out[3].abs().sum()) - float(out[3, 12345]) == 0.0
    assert torch.allclose(out[[0, 1, 4]].double().sum(dim=1).cpu(), torch.ones(3, dtype=torch.float64), atol=1e-5)


@pytest.mark.parametrize("rows,cols", [(37, 65540), (9, 100004), (300, 128256), (5, 262144),
                                       (3, 400000), (2, 600000)])
def test_softmax_rows_held_by_a_cluster(rows, cols):
    # aligned rows above 256 KB: a cluster of CTAs per row holds the row in
    # shared memory (slices double-buffered, partial states merged through
    # distributed shared memory); 600000 columns need more shared memory than
    # a cluster offers and take the L2 path.  Row counts are not multiples of
    # the resident clusters.  Row 0 has a masked slice, row 1 is masked but for
    # one entry, the last row has a NaN near its end.
    g = torch.Generator(device="cuda").manual_seed(rows + cols)
    x = torch.empty((rows, cols), dtype=torch.float32, device="cuda")
    x.normal_(0.0, 3.0, generator=g)
    x[0, cols // 3: cols // 3 + cols // 4] = float("-inf")
    if rows > 2:
        x[1, :] = float("-inf")
        x[1, cols - 5] = -3.0
    x[rows - 1, cols - 7] = float("nan")
    out = dattn.softmax(x)
    torch.cuda.synchronize()
    check(x, out)
    assert (out[0, cols // 3: cols // 3 + cols // 4] == 0).all()
    assert torch.isnan(out[rows - 1]).all()
    if rows > 2:
        assert abs(float(out[1, cols - 5]) - 1.0) <= 1e-6
        assert float(out[1].abs().sum()) == float(out[1, cols - 5])  # every other entry is 0


def test_softmax_cluster_rows_all_masked_row_is_nan():
    x = torch.full((4, 131072), float("-inf"), dtype=torch.float32, device="cuda")
    x[1:].normal_()
    out = dattn.softmax(x)
    torch.cuda.synchronize()
    assert torch.isnan(out[0]).all() and not torch.isnan(out[1:]).any()
    check(x, out)
