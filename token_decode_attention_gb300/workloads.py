"""Seeded synthetic workloads for decode-step attention.

This module holds only shapes and random-number recipes: no attention
arithmetic.  It is the one module that both the CUDA path's tests/benchmark and
the CPU oracle's callers use to make inputs.

The five workloads are decode steps against an f16 KV cache with layout
Q [batch, n_heads, head_dim], K/V [batch, seq_len, n_heads, head_dim]:

  small    B=1,   H=8,  D=64,  S=256,    current_pos=200
  7b       B=1,   H=32, D=128, S=4096,   current_pos=4095 (a 7B-class decode step)
  ragged   B=64,  H=32, D=128, S=2048,   current_pos ~ U{0..2047} per sequence
  long     B=1,   H=32, D=128, S=131072, current_pos=131071 (~2 GiB of K+V)
  outlier  B=256, H=40, D=128, S=8192,   current_pos=8191, K with 4 channels per
           head scaled x20 (40 GiB of K+V)

Recipe: Q, K, V are i.i.d. N(0,1) drawn directly in float16 with a
``torch.Generator`` on the target device seeded with ``seed``, in the order Q, K,
V.  ``current_pos`` is drawn with a CPU generator seeded with ``seed + 1``.  The
outlier channels are ``randperm(head_dim)[:4]`` per head from a CPU generator
seeded with ``seed + 2``; K is multiplied by 20 in those channels for every
sequence and position, rounded back to float16.  Default seeds are
20260000 + workload index.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    index: int
    batch: int
    n_heads: int
    head_dim: int
    seq_len: int
    current_pos: int | None  # None: uniform per sequence over [0, seq_len-1]
    outlier_channels: int = 0
    outlier_scale: float = 1.0
    description: str = ""

    @property
    def seed(self) -> int:
        return 20260000 + self.index

    def kv_bytes(self) -> int:
        """Bytes of the whole K and V allocation (capacity, not live)."""
        return 2 * self.batch * self.seq_len * self.n_heads * self.head_dim * 2


WORKLOADS: dict[str, Workload] = {
    w.name: w
    for w in [
        Workload("small", 0, 1, 8, 64, 256, 200,
                 description="B=1 H=8 D=64 S=256 cp=200"),
        Workload("7b", 1, 1, 32, 128, 4096, 4095,
                 description="B=1 H=32 D=128 S=4096 cp=4095 (7B-class decode step)"),
        Workload("ragged", 2, 64, 32, 128, 2048, None,
                 description="B=64 H=32 D=128 S=2048 cp~U{0..2047} (ragged batch)"),
        Workload("long", 3, 1, 32, 128, 131072, 131071,
                 description="B=1 H=32 D=128 S=131072 cp=131071 (long context, 2 GiB K+V)"),
        Workload("outlier", 4, 256, 40, 128, 8192, 8191, outlier_channels=4,
                 outlier_scale=20.0,
                 description="B=256 H=40 D=128 S=8192 cp=8191, K with 4 outlier "
                             "channels per head x20 (40 GiB K+V)"),
    ]
}


def draw_current_pos(w: Workload, seed: int | None = None) -> np.ndarray:
    """current_pos per sequence, uint32 [batch]."""
    seed = w.seed if seed is None else seed
    if w.current_pos is not None:
        return np.full((w.batch,), w.current_pos, dtype=np.uint32)
    g = torch.Generator(device="cpu").manual_seed(seed + 1)
    cp = torch.randint(0, w.seq_len, (w.batch,), generator=g, dtype=torch.int64)
    return cp.numpy().astype(np.uint32)


def draw_outlier_channels(w: Workload, seed: int | None = None) -> np.ndarray:
    """[n_heads, outlier_channels] distinct channel indices per head (int64)."""
    seed = w.seed if seed is None else seed
    g = torch.Generator(device="cpu").manual_seed(seed + 2)
    rows = [torch.randperm(w.head_dim, generator=g)[: w.outlier_channels]
            for _ in range(w.n_heads)]
    return torch.stack(rows).numpy()


def _randn_f16(shape, gen, device) -> torch.Tensor:
    t = torch.empty(shape, dtype=torch.float16, device=device)
    t.normal_(0.0, 1.0, generator=gen)
    return t


def make_inputs(w: Workload, device: str | torch.device = "cuda", seed: int | None = None,
                batch: int | None = None) -> dict:
    """Draw Q, K, V (float16) and current_pos for a workload.

    ``batch`` overrides the batch size (same per-sequence recipe), which the
    tests use to draw a subset of a large workload.  Returns a dict with torch
    tensors ``q, k, v`` on ``device``, ``cur_pos`` (int32 tensor on ``device``,
    same bits as uint32) and ``cur_pos_host`` (numpy uint32).
    """
    seed = w.seed if seed is None else seed
    B = w.batch if batch is None else batch
    device = torch.device(device)
    gen = torch.Generator(device=device).manual_seed(seed)
    q = _randn_f16((B, w.n_heads, w.head_dim), gen, device)
    k = _randn_f16((B, w.seq_len, w.n_heads, w.head_dim), gen, device)
    v = _randn_f16((B, w.seq_len, w.n_heads, w.head_dim), gen, device)
    if w.outlier_channels:
        ch = torch.from_numpy(draw_outlier_channels(w, seed)).to(device)
        heads = torch.arange(w.n_heads, device=device).unsqueeze(1).expand_as(ch)
        kv = k.view(B * w.seq_len, w.n_heads, w.head_dim)
        kv[:, heads.reshape(-1), ch.reshape(-1)] *= w.outlier_scale
    cp = draw_current_pos(w, seed)
    if batch is not None:
        cp = np.resize(cp, B).astype(np.uint32)
    cp_dev = torch.from_numpy(cp.astype(np.int64)).to(torch.int32).to(device)
    return {"q": q, "k": k, "v": v, "cur_pos": cp_dev, "cur_pos_host": cp}


def live_lengths(cur_pos: np.ndarray, seq_len: int) -> np.ndarray:
    """Live positions per sequence: positions 0..current_pos, capped at seq_len."""
    return np.minimum(cur_pos.astype(np.int64), seq_len - 1) + 1


def algorithmic_bytes(batch: int, n_heads: int, head_dim: int, seq_len: int,
                      cur_pos: np.ndarray) -> int:
    """Bytes a decode step must move: Q + live K rows + live V rows + out (f16)."""
    live = int(live_lengths(cur_pos, seq_len).sum())
    qo = 2 * batch * n_heads * head_dim * 2
    return qo + 2 * live * n_heads * head_dim * 2
