"""Decode-step attention against an f16 KV cache, for NVIDIA GB300 (sm_103a).

The compute path is the C-ABI library ``libdattn.so`` (``include/dattn.h``),
built from the CUDA sources in ``csrc/``.  This package holds its build script,
its ctypes binding and the seeded synthetic workloads; the binding is loaded on
first use and raises if the library has not been built.
"""
from ._native import (  # noqa: F401
    Batch,
    DattnError,
    dattn_batch_begin,
    dattn_batch_end,
    dattn_decode_f16,
    dattn_decode_f16_ex,
    dattn_decode_paged_f16,
    dattn_decode_paged_plan,
    dattn_decode_plan,
    dattn_decode_workspace_bytes,
    dattn_device_error,
    dattn_pv_f16,
    dattn_qk_f16,
    dattn_rope_append_f16,
    dattn_rope_append_paged_f16,
    dattn_softmax_f32,
    dattn_version,
    decode,
    decode_paged,
    load,
    pv,
    qk,
    rope_append,
    softmax,
)
