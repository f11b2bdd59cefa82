"""UltraQuant 4-bit KV cache for NVIDIA GB300 (sm_103a).

Public API (ctypes binding of the C ABI in include/uq.h, same names):
``uq_store``, ``uq_store_rotated_f32``, ``uq_decode``, ``uq_decode_ex``, ``uq_decode_multi_query``,
``uq_full_dequant``,
``uq_decode_workspace_bytes``, ``uq_slot_bytes``, ``uq_check_device_error``,
``uq_last_error``, ``uq_version``.  Build the CUDA library with
``bit_quantized_kv_gb300.build.build()``.

Attributes are resolved lazily so that ``bit_quantized_kv_gb300.workloads``
(seeded synthetic inputs) can be imported without loading the library.
"""
from __future__ import annotations

_API = ("uq_store", "uq_store_rotated_f32", "uq_decode", "uq_decode_ex", "uq_decode_multi_query",
        "uq_full_dequant",
        "uq_decode_workspace_bytes",
        "uq_slot_bytes", "uq_check_device_error", "uq_last_error", "uq_version",
        "uq_set_timing_events", "uq_decode_static_scratch", "UQError")

__all__ = list(_API)


def __getattr__(name):
    if name in _API:
        from . import binding
        return getattr(binding, name)
    raise AttributeError(name)
