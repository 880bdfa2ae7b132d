"""Paged single-query decode attention for GB300 (sm_103a).

The compute path is the C-ABI library ``libpaged_decode.so`` built from
``csrc/``; ``paged_kv_decode_21_gb300.ops`` is a thin ctypes binding over it.
"""
__all__ = ["workloads", "traffic"]
