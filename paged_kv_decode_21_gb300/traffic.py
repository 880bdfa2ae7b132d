"""Byte accounting for paged decode attention (host-side helpers).

* ``algorithmic_bytes``: the bytes one call must move at minimum -- every used
  K and V row once, Q once, out once.  Block tables, context lengths and the
  split-K workspace are overhead and are reported separately.
* ``decode_step_kv_bytes``: the per-decode-step KV volume of a whole model,
  2 (K and V) x layers x kv_heads x head_dim x context x bytes; the blog post
  "KV Cache Prefetching：三层预取如何隐藏 KV 访问延迟" (section 1.1) works it
  out for an 80-layer, 8-kv-head, 128-dim model at 32K context as about 10 GB.
* ``m_block`` / ``m_total`` / ``l2_resident_batches``: the L2 capacity model of
  the review "Accelerating LLM Inference Throughput via Asynchronous KV Cache
  Prefetching", section 4.2: M_block = b * d_h * T_block bytes per (block,
  head) tile, M_total = M_block * (N_thread / 32) * H * B bytes touched by one
  loop iteration of all warps over the batch, and the batch count whose
  per-iteration tiles fit in an L2 of a given size.
"""
from __future__ import annotations

from typing import Iterable


def algorithmic_bytes(context_lens: Iterable[int], num_q_heads: int, num_kv_heads: int,
                      head_dim: int, elem_bytes: int = 2) -> int:
    """K+V rows of every used token and kv head, plus Q and out."""
    lens = [int(x) for x in context_lens]
    kv = 2 * sum(lens) * num_kv_heads * head_dim * elem_bytes
    qo = 2 * len(lens) * num_q_heads * head_dim * elem_bytes
    return kv + qo


def kv_bytes(context_lens: Iterable[int], num_kv_heads: int, head_dim: int, elem_bytes: int = 2) -> int:
    """K+V bytes alone."""
    return 2 * sum(int(x) for x in context_lens) * num_kv_heads * head_dim * elem_bytes


def workspace_bytes_moved(context_lens: Iterable[int], num_q_heads: int, head_dim: int,
                          partition_size: int) -> int:
    """Split-K partial traffic: each used partition writes and the merge reads
    (m, l, o[head_dim]) in fp32; the merge also writes out (counted above)."""
    if partition_size <= 0:
        return 0
    n = sum(-(-int(L) // partition_size) for L in context_lens if int(L) > partition_size)
    return 2 * n * num_q_heads * (head_dim + 2) * 4


def decode_step_kv_bytes(num_layers: int, num_kv_heads: int, head_dim: int, context_len: int,
                         elem_bytes: int = 2) -> int:
    """Whole-model KV bytes read by one decode step of one sequence."""
    return 2 * num_layers * num_kv_heads * head_dim * context_len * elem_bytes


def m_block(bytes_per_param: int, head_dim: int, block_tokens: int) -> int:
    """Bytes of one (block, head) tile: b * d_h * T_block."""
    return bytes_per_param * head_dim * block_tokens


def m_total(m_block_bytes: int, n_thread: int, num_heads: int, batch: int) -> int:
    """Bytes touched by one iteration of every warp over the batch."""
    return m_block_bytes * (n_thread // 32) * num_heads * batch


def l2_resident_batches(l2_bytes: int, m_block_bytes: int, n_thread: int, num_heads: int) -> int:
    """Largest batch whose per-iteration tiles fit in ``l2_bytes``."""
    return l2_bytes // m_total(m_block_bytes, n_thread, num_heads, 1)
