"""CPU oracle for single-query (decode-step) attention against an f16 KV cache.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this package.  The
CUDA library never calls it and shares no code with it.

What it computes follows "Developing Apple Metal Kernels in Rust - A Deep Dive
Through Attention", section "The MSL, briefly" (kernels ``attention_qk_f16`` and
``attention_pv_f16``), with a leading batch dimension and one ``current_pos`` per
sequence.  The arithmetic lives in ``oracle.c`` (fp64, plain loops, OpenMP over
(batch, head)); this module only marshals numpy arrays through ctypes.

Every function here is pinned by ``tests/test_oracle_pins.py`` against closed
forms, invariants, exact rational arithmetic and library routines.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

_LIB = None


def _load(path: str):
    """Open a compiled oracle library and declare its signatures."""
    lib = ctypes.CDLL(path)
    i64, u16p, u32p, f64p = (ctypes.c_int64, ctypes.POINTER(ctypes.c_uint16),
                             ctypes.POINTER(ctypes.c_uint32),
                             ctypes.POINTER(ctypes.c_double))
    lib.oracle_decode_f64.argtypes = [u16p, u16p, u16p, i64, i64, i64, i64, u32p, f64p,
                                      ctypes.c_int]
    lib.oracle_qk_f64.argtypes = [u16p, u16p, i64, i64, i64, i64, u32p, f64p, ctypes.c_int]
    lib.oracle_pv_f64.argtypes = [u16p, u16p, i64, i64, i64, i64, f64p, ctypes.c_int]
    lib.oracle_qk_pages_f16.argtypes = [u16p, u16p, i64, i64, i64, i64, u32p, u16p,
                                        ctypes.c_int]
    lib.oracle_f16_to_f64_array.argtypes = [u16p, f64p, i64]
    lib.oracle_f32_to_f16_array.argtypes = [ctypes.POINTER(ctypes.c_float), u16p, i64]
    lib.oracle_max_threads.restype = ctypes.c_int
    lib.oracle_rope_f64.argtypes = [u16p, i64, i64, i64, i64, ctypes.c_double, ctypes.c_int,
                                    u32p, f64p]
    lib.oracle_softmax_f64.argtypes = [ctypes.POINTER(ctypes.c_float), i64, i64, f64p,
                                       ctypes.c_int]
    lib.oracle_decode_paged_f64.argtypes = [u16p, u16p, u16p, i64, i64, i64, i64, i64,
                                            ctypes.POINTER(ctypes.c_int32), i64, u32p, f64p,
                                            ctypes.c_int]
    return lib


def _lib():
    global _LIB
    if _LIB is None:
        path = _build.LIB
        if not os.path.exists(path) or os.path.getmtime(path) < os.path.getmtime(_build.SRC):
            _build.build()
        _LIB = _load(path)
    return _LIB


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _f16_bits(x, ndim: int, name: str) -> np.ndarray:
    a = np.ascontiguousarray(x)
    if a.dtype != np.float16:
        raise TypeError(f"{name} must be float16, got {a.dtype}")
    if a.ndim != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got shape {a.shape}")
    return a.view(np.uint16)


def _cur_pos(cp, B: int) -> np.ndarray:
    a = np.ascontiguousarray(np.asarray(cp, dtype=np.int64).reshape(-1))
    if a.shape[0] != B:
        raise ValueError(f"current_pos must have {B} entries, got {a.shape[0]}")
    if (a < 0).any() or (a > 0xFFFFFFFF).any():
        raise ValueError("current_pos must fit uint32")
    return a.astype(np.uint32)


def max_threads() -> int:
    """Number of OpenMP threads the oracle uses by default."""
    return int(_lib().oracle_max_threads())


def decode_f64(Q, K, V, current_pos, threads: int = 0) -> np.ndarray:
    """Fused decode attention in fp64.

    Q [B,H,D], K/V [B,S,H,D] float16, current_pos [B] -> out [B,H,D] float64.
    """
    q = _f16_bits(Q, 3, "Q")
    k = _f16_bits(K, 4, "K")
    v = _f16_bits(V, 4, "V")
    B, H, D = q.shape
    S = k.shape[1]
    if k.shape != (B, S, H, D) or v.shape != (B, S, H, D):
        raise ValueError(f"K/V shape {k.shape}/{v.shape} does not match Q {q.shape}")
    cp = _cur_pos(current_pos, B)
    out = np.empty((B, H, D), dtype=np.float64)
    _lib().oracle_decode_f64(_ptr(q, ctypes.c_uint16), _ptr(k, ctypes.c_uint16),
                             _ptr(v, ctypes.c_uint16), B, H, D, S,
                             _ptr(cp, ctypes.c_uint32), _ptr(out, ctypes.c_double), threads)
    return out


def decode_paged_f64(Q, K_pages, V_pages, block_table, current_pos,
                     threads: int = 0) -> np.ndarray:
    """Fused decode attention over a paged cache, fp64.

    Q [B,H,D], K/V pages [num_pages, page_size, H, D] float16, block_table
    [B, max_pages] int32, current_pos [B] -> out [B,H,D] float64 (NaN rows for
    sequences whose live pages are not valid indices).
    """
    q = _f16_bits(Q, 3, "Q")
    kp = _f16_bits(K_pages, 4, "K_pages")
    vp = _f16_bits(V_pages, 4, "V_pages")
    B, H, D = q.shape
    num_pages, page_size = kp.shape[0], kp.shape[1]
    if kp.shape != (num_pages, page_size, H, D) or vp.shape != kp.shape:
        raise ValueError(f"page shapes {kp.shape}/{vp.shape} do not match Q {q.shape}")
    table = np.ascontiguousarray(np.asarray(block_table, dtype=np.int32))
    if table.ndim != 2 or table.shape[0] != B:
        raise ValueError(f"block_table must be [{B}, max_pages], got {table.shape}")
    cp = _cur_pos(current_pos, B)
    out = np.empty((B, H, D), dtype=np.float64)
    _lib().oracle_decode_paged_f64(_ptr(q, ctypes.c_uint16), _ptr(kp, ctypes.c_uint16),
                                   _ptr(vp, ctypes.c_uint16), B, H, D, page_size,
                                   table.shape[1], _ptr(table, ctypes.c_int32), num_pages,
                                   _ptr(cp, ctypes.c_uint32), _ptr(out, ctypes.c_double),
                                   threads)
    return out


def qk_f64(Q, K, current_pos, threads: int = 0) -> np.ndarray:
    """QK step in fp64: scores [B,H,S], exactly -inf where p > current_pos."""
    q = _f16_bits(Q, 3, "Q")
    k = _f16_bits(K, 4, "K")
    B, H, D = q.shape
    S = k.shape[1]
    if k.shape != (B, S, H, D):
        raise ValueError(f"K shape {k.shape} does not match Q {q.shape}")
    cp = _cur_pos(current_pos, B)
    out = np.empty((B, H, S), dtype=np.float64)
    _lib().oracle_qk_f64(_ptr(q, ctypes.c_uint16), _ptr(k, ctypes.c_uint16), B, H, D, S,
                         _ptr(cp, ctypes.c_uint32), _ptr(out, ctypes.c_double), threads)
    return out


def pv_f64(scores, V, threads: int = 0) -> np.ndarray:
    """PV step in fp64 on f16 scores [B,H,S] and V [B,S,H,D] -> out [B,H,D]."""
    s = _f16_bits(scores, 3, "scores")
    v = _f16_bits(V, 4, "V")
    B, H, S = s.shape
    D = v.shape[3]
    if v.shape != (B, S, H, D):
        raise ValueError(f"V shape {v.shape} does not match scores {s.shape}")
    out = np.empty((B, H, D), dtype=np.float64)
    _lib().oracle_pv_f64(_ptr(s, ctypes.c_uint16), _ptr(v, ctypes.c_uint16), B, H, D, S,
                         _ptr(out, ctypes.c_double), threads)
    return out


def qk_pages_f16(Q, K, current_pos, threads: int = 0) -> np.ndarray:
    """QK step at the page's precision (fp32 in index order, f16 scores)."""
    q = _f16_bits(Q, 3, "Q")
    k = _f16_bits(K, 4, "K")
    B, H, D = q.shape
    S = k.shape[1]
    if k.shape != (B, S, H, D):
        raise ValueError(f"K shape {k.shape} does not match Q {q.shape}")
    cp = _cur_pos(current_pos, B)
    out = np.empty((B, H, S), dtype=np.uint16)
    _lib().oracle_qk_pages_f16(_ptr(q, ctypes.c_uint16), _ptr(k, ctypes.c_uint16), B, H, D,
                               S, _ptr(cp, ctypes.c_uint32), _ptr(out, ctypes.c_uint16),
                               threads)
    return out.view(np.float16)


def rope_f64(x, position, rope_dims: int | None = None, base: float = 10000.0,
             traditional: bool = False) -> np.ndarray:
    """Rotary embedding of x [B,H,D] float16 at per-sequence positions, fp64."""
    a = _f16_bits(x, 3, "x")
    B, H, D = a.shape
    rd = D if rope_dims is None else int(rope_dims)
    if rd < 2 or rd > D or rd % 2:
        raise ValueError(f"rope_dims must be even and in [2, {D}], got {rd}")
    pos = _cur_pos(position, B)
    out = np.empty((B, H, D), dtype=np.float64)
    _lib().oracle_rope_f64(_ptr(a, ctypes.c_uint16), B, H, D, rd, float(base),
                           1 if traditional else 0, _ptr(pos, ctypes.c_uint32),
                           _ptr(out, ctypes.c_double))
    return out


def softmax_f64(x, threads: int = 0) -> np.ndarray:
    """Row softmax over the last dimension of a float32 [rows, cols] array, fp64."""
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    if a.ndim != 2:
        raise ValueError(f"x must be [rows, cols], got {a.shape}")
    out = np.empty(a.shape, dtype=np.float64)
    _lib().oracle_softmax_f64(_ptr(a, ctypes.c_float), a.shape[0], a.shape[1],
                              _ptr(out, ctypes.c_double), threads)
    return out


def f16_bits_to_f64(bits) -> np.ndarray:
    """binary16 bit patterns -> float64, decoded from the format's definition."""
    a = np.ascontiguousarray(np.asarray(bits, dtype=np.uint16))
    out = np.empty(a.shape, dtype=np.float64)
    _lib().oracle_f16_to_f64_array(_ptr(a, ctypes.c_uint16), _ptr(out, ctypes.c_double),
                                   a.size)
    return out


def f32_to_f16_bits(x) -> np.ndarray:
    """float32 -> binary16 bit patterns, round to nearest, ties to even."""
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    out = np.empty(a.shape, dtype=np.uint16)
    _lib().oracle_f32_to_f16_array(_ptr(a, ctypes.c_float), _ptr(out, ctypes.c_uint16),
                                   a.size)
    return out
