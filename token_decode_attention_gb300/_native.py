"""ctypes binding of libdattn (include/dattn.h).

Argument marshalling only: every function here checks dtypes, devices, shapes
and contiguity of torch tensors, passes raw device pointers and the current
CUDA stream to the C ABI, and turns a non-zero status into ``DattnError``.
All arithmetic runs in the library's CUDA kernels.  There is no fallback: if
``libdattn.so`` is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

_LIB = None


class DattnError(RuntimeError):
    """A libdattn entry point returned a non-zero status."""

    def __init__(self, status: int, where: str, message: str):
        self.status = status
        super().__init__(f"{where}: {status_name(status)}: {message}")


class Plan(ctypes.Structure):
    _fields_ = [("partitions", ctypes.c_int), ("heads_per_cta", ctypes.c_int),
                ("head_groups", ctypes.c_int), ("stage_positions", ctypes.c_int),
                ("stages", ctypes.c_int), ("threads_per_cta", ctypes.c_int),
                ("smem_bytes", ctypes.c_int), ("ctas_per_sm", ctypes.c_int),
                ("sm_count", ctypes.c_int), ("workspace_bytes", ctypes.c_size_t),
                ("cluster_size", ctypes.c_int)]

    def as_dict(self) -> dict:
        return {name: getattr(self, name) for name, _ in self._fields_}


# status codes (enum dattn_status)
(OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_MISALIGNED, ERR_WORKSPACE, ERR_CUDA, ERR_TIMEOUT,
 ERR_BAD_PAGE, ERR_BAD_POSITION) = (0, -1, -2, -3, -4, -5, -6, -7, -8)

_P = ctypes.c_void_p
_I = ctypes.c_int
_SIGNATURES = {
    "dattn_version": ([], _I),
    "dattn_status_string": ([_I], ctypes.c_char_p),
    "dattn_last_error": ([], ctypes.c_char_p),
    "dattn_decode_plan": ([_I, _I, _I, _I, _I, ctypes.POINTER(Plan)], _I),
    "dattn_decode_paged_plan": ([_I, _I, _I, _I, _I, ctypes.c_longlong, _I, ctypes.POINTER(Plan)],
                                _I),
    "dattn_decode_workspace_bytes": ([_I, _I, _I, _I, _I, ctypes.POINTER(ctypes.c_size_t)], _I),
    "dattn_decode_f16_ex": ([_P, _P, _P, _P, _I, _I, _I, _I, _P, _P, ctypes.c_size_t, _I, _P],
                            _I),
    "dattn_decode_f16": ([_P, _P, _P, _P, _I, _I, _I, _I, _P, _P], _I),
    "dattn_decode_paged_f16": ([_P, _P, _P, _P, _I, _I, _I, _I, _I, ctypes.c_longlong, _P, _P, _P,
                                ctypes.c_size_t, _I, _P], _I),
    "dattn_decode_f16_noalloc": ([_P, _P, _P, _P, _I, _I, _I, _I, _P, _P], _I),
    "dattn_qk_f16": ([_P, _P, _P, _I, _I, _I, _I, _P, _P], _I),
    "dattn_pv_f16": ([_P, _P, _P, _I, _I, _I, _I, _P], _I),
    "dattn_device_error": ([_I], _I),
    "dattn_selftest_wait_timeout": ([_P], _I),
    "dattn_softmax_f32": ([_P, _P, ctypes.c_longlong, _I, _P], _I),
    "dattn_rope_append_f16": ([_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, ctypes.c_double, _I,
                               _P, _P], _I),
    "dattn_rope_append_paged_f16": ([_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I,
                                     ctypes.c_longlong, _P, _I, ctypes.c_double, _I, _P, _P], _I),
    "dattn_batch_begin": ([_P], _I),
    "dattn_batch_end": ([_P, ctypes.POINTER(ctypes.c_void_p)], _I),
    "dattn_batch_launch": ([_P, _P], _I),
    "dattn_batch_nodes": ([_P], ctypes.c_longlong),
    "dattn_batch_destroy": ([_P], _I),
}


def library_path() -> str:
    return _build.LIB


def load(path: str | None = None):
    """Open libdattn and declare every exported signature."""
    global _LIB
    if _LIB is not None and path is None:
        return _LIB
    p = path or _build.LIB
    if not os.path.exists(p):
        raise RuntimeError(f"libdattn is not built ({p} missing); run "
                           "__graft_entry__.build() or python -m "
                           "token_decode_attention_gb300.build")
    lib = ctypes.CDLL(p)
    for name, (args, res) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    if path is None:
        _LIB = lib
    return lib


def status_name(status: int) -> str:
    return load().dattn_status_string(status).decode()


def _check(status: int, where: str) -> None:
    if status != OK:
        raise DattnError(status, where, load().dattn_last_error().decode())


def _stream_handle(stream) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return int(s.cuda_stream)


def _tensor(t: torch.Tensor, name: str, shape=None, dtype=torch.float16) -> int:
    """Raw pointer of a CUDA tensor, or of a pinned (page-locked) CPU tensor: with
    unified addressing pinned host memory has the same address on the device, and
    the kernels read or write it over the CPU-GPU link."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not (t.is_cuda or t.is_pinned()):
        raise ValueError(f"{name} must be a CUDA tensor or a pinned CPU tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous (call .contiguous() first)")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    return t.data_ptr()


def _cur_pos(t: torch.Tensor, B: int) -> int:
    if t.dtype not in (torch.int32, getattr(torch, "uint32", torch.int32)):
        raise TypeError(f"current_pos must be int32 or uint32, got {t.dtype}")
    return _tensor(t, "current_pos", (B,), t.dtype)


def _qkv_dims(q, k):
    if q.dim() != 3 or k.dim() != 4:
        raise ValueError("Q must be [batch, n_heads, head_dim] and K/V "
                         "[batch, seq_len, n_heads, head_dim]")
    B, H, D = q.shape
    S = k.shape[1]
    return int(B), int(H), int(D), int(S)


# ----------------------------------------------------------- C-ABI mirrors

def dattn_version() -> int:
    return int(load().dattn_version())


def dattn_decode_plan(batch: int, n_heads: int, head_dim: int, seq_len: int,
                      num_partitions: int = 0) -> dict:
    plan = Plan()
    _check(load().dattn_decode_plan(batch, n_heads, head_dim, seq_len, num_partitions,
                                    ctypes.byref(plan)), "dattn_decode_plan")
    return plan.as_dict()


def dattn_decode_paged_plan(batch: int, n_heads: int, head_dim: int, page_size: int,
                            max_pages: int, num_pages: int, num_partitions: int = 0) -> dict:
    plan = Plan()
    _check(load().dattn_decode_paged_plan(batch, n_heads, head_dim, page_size, max_pages,
                                          num_pages, num_partitions, ctypes.byref(plan)),
           "dattn_decode_paged_plan")
    return plan.as_dict()


def dattn_decode_workspace_bytes(batch: int, n_heads: int, head_dim: int, seq_len: int,
                                 num_partitions: int = 0) -> int:
    n = ctypes.c_size_t(0)
    _check(load().dattn_decode_workspace_bytes(batch, n_heads, head_dim, seq_len, num_partitions,
                                               ctypes.byref(n)),
           "dattn_decode_workspace_bytes")
    return int(n.value)


def dattn_decode_f16_ex(q, k, v, out, current_pos, workspace=None, num_partitions: int = 0,
                        stream=None) -> None:
    B, H, D, S = _qkv_dims(q, k)
    args = (_tensor(q, "Q", (B, H, D)), _tensor(k, "K_cache", (B, S, H, D)),
            _tensor(v, "V_cache", (B, S, H, D)), _tensor(out, "out", (B, H, D)))
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr = _tensor(workspace, "workspace", None, workspace.dtype)
        ws_bytes = workspace.numel() * workspace.element_size()
    _check(load().dattn_decode_f16_ex(*args, B, H, D, S, _cur_pos(current_pos, B), ws_ptr,
                                      ws_bytes, num_partitions, _stream_handle(stream)),
           "dattn_decode_f16_ex")


def dattn_decode_paged_f16(q, k_pages, v_pages, out, block_table, current_pos, workspace=None,
                           num_partitions: int = 0, stream=None) -> None:
    if q.dim() != 3 or k_pages.dim() != 4 or block_table.dim() != 2:
        raise ValueError("Q must be [batch, n_heads, head_dim], pages [num_pages, page_size, "
                         "n_heads, head_dim], block_table [batch, max_pages]")
    B, H, D = (int(x) for x in q.shape)
    num_pages, page_size = int(k_pages.shape[0]), int(k_pages.shape[1])
    max_pages = int(block_table.shape[1])
    args = (_tensor(q, "Q", (B, H, D)), _tensor(k_pages, "K_pages", (num_pages, page_size, H, D)),
            _tensor(v_pages, "V_pages", (num_pages, page_size, H, D)),
            _tensor(out, "out", (B, H, D)))
    table = _tensor(block_table, "block_table", (B, max_pages), torch.int32)
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr = _tensor(workspace, "workspace", None, workspace.dtype)
        ws_bytes = workspace.numel() * workspace.element_size()
    _check(load().dattn_decode_paged_f16(*args, B, H, D, page_size, max_pages, num_pages, table,
                                         _cur_pos(current_pos, B), ws_ptr, ws_bytes,
                                         num_partitions, _stream_handle(stream)),
           "dattn_decode_paged_f16")


def dattn_decode_f16(q, k, v, out, current_pos, stream=None) -> None:
    B, H, D, S = _qkv_dims(q, k)
    _check(load().dattn_decode_f16(_tensor(q, "Q", (B, H, D)), _tensor(k, "K_cache", (B, S, H, D)),
                                   _tensor(v, "V_cache", (B, S, H, D)),
                                   _tensor(out, "out", (B, H, D)), B, H, D, S,
                                   _cur_pos(current_pos, B), _stream_handle(stream)),
           "dattn_decode_f16")


def dattn_qk_f16(q, k, scores, current_pos, stream=None) -> None:
    B, H, D, S = _qkv_dims(q, k)
    _check(load().dattn_qk_f16(_tensor(q, "Q", (B, H, D)), _tensor(k, "K_cache", (B, S, H, D)),
                               _tensor(scores, "scores", (B, H, S)), B, H, D, S,
                               _cur_pos(current_pos, B), _stream_handle(stream)),
           "dattn_qk_f16")


def dattn_pv_f16(scores, v, out, stream=None) -> None:
    if scores.dim() != 3 or v.dim() != 4:
        raise ValueError("scores must be [batch, n_heads, seq_len], V [batch, seq_len, n_heads, "
                         "head_dim]")
    B, H, S = (int(x) for x in scores.shape)
    D = int(v.shape[3])
    _check(load().dattn_pv_f16(_tensor(scores, "scores", (B, H, S)),
                               _tensor(v, "V_cache", (B, S, H, D)),
                               _tensor(out, "out", (B, H, D)), B, H, D, S,
                               _stream_handle(stream)), "dattn_pv_f16")


def dattn_device_error(clear: bool = True) -> int:
    """Status of the device error word (DATTN_OK, or the TIMEOUT, BAD_PAGE or
    BAD_POSITION it records); never raises on those, so callers can assert on it."""
    st = int(load().dattn_device_error(1 if clear else 0))
    if st not in (OK, ERR_TIMEOUT, ERR_BAD_PAGE, ERR_BAD_POSITION):
        _check(st, "dattn_device_error")
    return st


def dattn_softmax_f32(x, out, stream=None) -> None:
    if x.dim() != 2:
        raise ValueError("x must be [rows, cols]")
    rows, cols = (int(v) for v in x.shape)
    _check(load().dattn_softmax_f32(_tensor(x, "x", (rows, cols), torch.float32),
                                    _tensor(out, "out", (rows, cols), torch.float32), rows, cols,
                                    _stream_handle(stream)), "dattn_softmax_f32")


def softmax(x, out=None, stream=None):
    """Row softmax over the last dimension of a float32 [rows, cols] tensor."""
    if out is None:
        out = torch.empty_like(x)
    dattn_softmax_f32(x, out, stream)
    return out


def dattn_rope_append_f16(q_new, k_new, v_new, q_out, k_cache, v_cache, current_pos,
                          rope_dims: int = 0, rope_base: float = 10000.0,
                          traditional: bool = False, stream=None) -> None:
    if q_new.dim() != 3 or k_cache.dim() != 4:
        raise ValueError("q_new must be [batch, n_heads, head_dim], the cache [batch, seq_len, "
                         "n_heads, head_dim]")
    B, H, D = (int(x) for x in q_new.shape)
    S = int(k_cache.shape[1])
    new = [_tensor(t, n, (B, H, D)) for t, n in ((q_new, "q_new"), (k_new, "k_new"),
                                                 (v_new, "v_new"), (q_out, "q_out"))]
    _check(load().dattn_rope_append_f16(*new, _tensor(k_cache, "K_cache", (B, S, H, D)),
                                        _tensor(v_cache, "V_cache", (B, S, H, D)), B, H, D, S,
                                        rope_dims or D, float(rope_base), int(bool(traditional)),
                                        _cur_pos(current_pos, B), _stream_handle(stream)),
           "dattn_rope_append_f16")


def dattn_rope_append_paged_f16(q_new, k_new, v_new, q_out, k_pages, v_pages, block_table,
                                current_pos, rope_dims: int = 0, rope_base: float = 10000.0,
                                traditional: bool = False, stream=None) -> None:
    if q_new.dim() != 3 or k_pages.dim() != 4 or block_table.dim() != 2:
        raise ValueError("q_new must be [batch, n_heads, head_dim], pages [num_pages, page_size, "
                         "n_heads, head_dim], block_table [batch, max_pages]")
    B, H, D = (int(x) for x in q_new.shape)
    num_pages, page_size = int(k_pages.shape[0]), int(k_pages.shape[1])
    max_pages = int(block_table.shape[1])
    new = [_tensor(t, n, (B, H, D)) for t, n in ((q_new, "q_new"), (k_new, "k_new"),
                                                 (v_new, "v_new"), (q_out, "q_out"))]
    _check(load().dattn_rope_append_paged_f16(
        *new, _tensor(k_pages, "K_pages", (num_pages, page_size, H, D)),
        _tensor(v_pages, "V_pages", (num_pages, page_size, H, D)), B, H, D, page_size, max_pages,
        num_pages, _tensor(block_table, "block_table", (B, max_pages), torch.int32),
        rope_dims or D, float(rope_base), int(bool(traditional)), _cur_pos(current_pos, B),
        _stream_handle(stream)), "dattn_rope_append_paged_f16")


def rope_append(q_new, k_new, v_new, k_cache, v_cache, current_pos, rope_dims: int = 0,
                rope_base: float = 10000.0, traditional: bool = False, block_table=None,
                q_out=None, stream=None):
    """Rotate the new token's q and k at current_pos[b] and append k, v to the cache
    (dense, or paged when ``block_table`` is given); returns the rotated q."""
    if q_out is None:
        q_out = torch.empty_like(q_new)
    if block_table is None:
        dattn_rope_append_f16(q_new, k_new, v_new, q_out, k_cache, v_cache, current_pos,
                              rope_dims, rope_base, traditional, stream)
    else:
        dattn_rope_append_paged_f16(q_new, k_new, v_new, q_out, k_cache, v_cache, block_table,
                                    current_pos, rope_dims, rope_base, traditional, stream)
    return q_out


def dattn_selftest_wait_timeout(stream=None) -> None:
    _check(load().dattn_selftest_wait_timeout(_stream_handle(stream)),
           "dattn_selftest_wait_timeout")


class Batch:
    """Calls recorded between dattn_batch_begin and dattn_batch_end on a stream,
    replayed as one submission (see include/dattn.h)."""

    def __init__(self, handle: int):
        self.handle = handle

    def launch(self, stream=None) -> None:
        _check(load().dattn_batch_launch(self.handle, _stream_handle(stream)),
               "dattn_batch_launch")

    @property
    def nodes(self) -> int:
        return int(load().dattn_batch_nodes(self.handle))

    def close(self) -> None:
        if self.handle:
            _check(load().dattn_batch_destroy(self.handle), "dattn_batch_destroy")
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def dattn_batch_begin(stream) -> None:
    _check(load().dattn_batch_begin(_stream_handle(stream)), "dattn_batch_begin")


def dattn_batch_end(stream) -> Batch:
    h = ctypes.c_void_p(0)
    _check(load().dattn_batch_end(_stream_handle(stream), ctypes.byref(h)), "dattn_batch_end")
    return Batch(h.value)


# ------------------------------------------------------- convenience forms

def decode(q, k, v, current_pos, num_partitions: int = 0, out=None, workspace=None, stream=None):
    """Fused decode attention; allocates ``out`` and the workspace with torch if not given."""
    B, H, D, S = _qkv_dims(q, k)
    if out is None:
        out = torch.empty((B, H, D), dtype=torch.float16, device=q.device)
    if workspace is None:
        n = dattn_decode_workspace_bytes(B, H, D, S, num_partitions)
        workspace = torch.empty((max(n, 16),), dtype=torch.uint8, device=q.device)
    dattn_decode_f16_ex(q, k, v, out, current_pos, workspace, num_partitions, stream)
    return out


def decode_paged(q, k_pages, v_pages, block_table, current_pos, num_partitions: int = 0,
                 out=None, workspace=None, stream=None):
    """Fused decode over a paged cache; allocates ``out`` and the workspace if not given."""
    B, H, D = (int(x) for x in q.shape)
    S = int(k_pages.shape[1]) * int(block_table.shape[1])
    if out is None:
        out = torch.empty((B, H, D), dtype=torch.float16, device=q.device)
    if workspace is None:
        n = dattn_decode_workspace_bytes(B, H, D, S, num_partitions)
        workspace = torch.empty((max(n, 16),), dtype=torch.uint8, device=q.device)
    dattn_decode_paged_f16(q, k_pages, v_pages, out, block_table, current_pos, workspace,
                           num_partitions, stream)
    return out


def qk(q, k, current_pos, scores=None, stream=None):
    B, H, D, S = _qkv_dims(q, k)
    if scores is None:
        scores = torch.empty((B, H, S), dtype=torch.float16, device=q.device)
    dattn_qk_f16(q, k, scores, current_pos, stream)
    return scores


def pv(scores, v, out=None, stream=None):
    B, H, S = (int(x) for x in scores.shape)
    if out is None:
        out = torch.empty((B, H, int(v.shape[3])), dtype=torch.float16, device=v.device)
    dattn_pv_f16(scores, v, out, stream)
    return out
