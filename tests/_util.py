"""Shared helpers for the GPU parity tests (tolerance, conversions)."""
from __future__ import annotations

import numpy as np
import torch

# Per-element bound on the fused decode output against the fp64 oracle:
# |out - ref| <= ATOL + RTOL * |ref|.  f16 output rounding alone contributes
# at most 2^-11 |ref| (~4.9e-4 |ref|); fp32 accumulation over <= 131072 terms
# is ~1e-6 relative; the bound leaves a margin of more than 10x.
ATOL = 2e-3
RTOL = 1e-2


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()


def assert_decode_close(got: torch.Tensor, ref: np.ndarray, what: str = "") -> float:
    g = to_np(got).astype(np.float64)
    assert g.shape == ref.shape, f"{what}: shape {g.shape} vs {ref.shape}"
    err = np.abs(g - ref)
    bound = ATOL + RTOL * np.abs(ref)
    bad = ~(err <= bound)
    if bad.any():
        idx = np.argwhere(bad)[0]
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} elements out of tolerance; first at "
            f"{tuple(idx)}: got {g[tuple(idx)]!r} ref {ref[tuple(idx)]!r}; max err "
            f"{np.nanmax(err):.3g}")
    return float(err.max()) if err.size else 0.0


def rand_f16(gen: torch.Generator, shape, device="cuda", scale: float = 1.0) -> torch.Tensor:
    t = torch.empty(shape, dtype=torch.float16, device=device)
    t.normal_(0.0, scale, generator=gen)
    return t


def cur_pos_tensor(cp, device="cuda") -> torch.Tensor:
    a = np.asarray(cp, dtype=np.int64)
    return torch.from_numpy(a).to(torch.int32).to(device)
