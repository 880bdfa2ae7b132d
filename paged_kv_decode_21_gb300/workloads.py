"""Seeded synthetic inputs for paged single-query decode attention.

This module only *draws* inputs: context lengths, a paged block table over a
physical block pool, and fp16 query / K / V values.  It contains none of the
attention arithmetic, so both the CUDA path and the CPU oracle may use it.

Layouts (shared by every consumer):

* ``q``            fp16  [num_seqs][num_q_heads][head_dim]
* ``k_cache``      fp16  [num_blocks][num_kv_heads][block_size][head_dim]
* ``v_cache``      fp16  same layout as ``k_cache``
* ``block_tables`` int32 [num_seqs][max_blocks_per_seq]; entry ``i`` of row
  ``b`` is the physical block holding logical tokens ``[i*bs, (i+1)*bs)`` of
  sequence ``b``; entries past ``ceil(L_b / bs)`` are ``-1`` (unused).
* ``context_lens`` int32 [num_seqs]

The paged layout follows the page-table description of the CSDN answer
"如何优化LLM推理引擎的内存访问延迟？" (section 2, the paged KV cache with a
logical-to-physical page table) and the block-table lookup ``bt[block_idx]`` of
Algorithm 1 in the review "Accelerating LLM Inference Throughput via
Asynchronous KV Cache Prefetching" (section 3.4).  One (block, kv-head) tile is
``block_size x head_dim`` contiguous fp16 values, the 4 KiB ``M_block`` of that
review's section 4.2 at head_dim=128, block_size=16.

Recipe (every config): lengths and the block permutation come from a CPU
``torch.Generator`` seeded with ``seed``; q/k/v are ``randn`` (fp32, then
rounded to fp16) from a generator seeded with ``seed + 1`` on the device that
will hold them.  The pool holds ``ceil(1.1 * needed)`` blocks unless a config
fixes it, and ``randperm(pool)[:needed]`` is dealt out to sequences in
(sequence, logical block) order.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import torch


@dataclasses.dataclass(frozen=True)
class DecodeConfig:
    """One decode-attention workload shape."""

    name: str
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    # either fixed per-sequence lengths, or a uniform [lo, hi] range
    context_lens: Optional[Sequence[int]] = None
    len_range: Optional[tuple] = None
    num_blocks: Optional[int] = None      # physical pool size; None -> ceil(1.1*needed)
    partition_size: int = 0               # split-K partition (tokens); 0 = unsplit
    seed: int = 0

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def max_context_len(self) -> int:
        if self.context_lens is not None:
            return int(max(self.context_lens))
        return int(self.len_range[1])

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)


# The five workloads of this library's test and benchmark suite.  The four
# model shapes are the attention layers of the models listed in section 5.1
# of the review (Llama2-7B 32:32, Llama3-8B 32:8, Qwen2.5-7B 28:4,
# Qwen2.5-14B 40:8), with head_dim=128 and block_size=16 as in section 4.2.
CONFIGS = {
    "tiny": DecodeConfig("tiny", 2, 4, 4, 64, 16, context_lens=(37, 100),
                         num_blocks=16, seed=0),
    "llama2_7b_mha": DecodeConfig("llama2_7b_mha", 64, 32, 32, 128, 16,
                                  context_lens=(2048,) * 64, seed=1),
    "llama3_8b_gqa4": DecodeConfig("llama3_8b_gqa4", 128, 32, 8, 128, 16,
                                   len_range=(512, 4096), seed=2),
    "qwen25_7b_gqa7": DecodeConfig("qwen25_7b_gqa7", 256, 28, 4, 128, 16,
                                   context_lens=(8192,) * 256, seed=3),
    "qwen25_14b_gqa5_splitk": DecodeConfig("qwen25_14b_gqa5_splitk", 32, 40, 8, 128, 16,
                                           len_range=(16384, 32768),
                                           partition_size=512, seed=4),
}
CONFIG_ORDER = ["tiny", "llama2_7b_mha", "llama3_8b_gqa4", "qwen25_7b_gqa7",
                "qwen25_14b_gqa5_splitk"]


@dataclasses.dataclass
class DecodeInputs:
    """Tensors of one workload (all on one device)."""

    q: torch.Tensor
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    block_tables: torch.Tensor
    context_lens: torch.Tensor
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    max_blocks_per_seq: int
    max_context_len: int
    scale: float

    def to(self, device) -> "DecodeInputs":
        kw = dataclasses.asdict(self)
        for k in ("q", "k_cache", "v_cache", "block_tables", "context_lens"):
            kw[k] = getattr(self, k).to(device)
        return DecodeInputs(**kw)


def draw_context_lens(cfg: DecodeConfig) -> torch.Tensor:
    """Per-sequence context lengths (int32, CPU)."""
    if cfg.context_lens is not None:
        assert len(cfg.context_lens) == cfg.num_seqs
        return torch.tensor(list(cfg.context_lens), dtype=torch.int32)
    g = torch.Generator().manual_seed(cfg.seed)
    lo, hi = cfg.len_range
    return torch.randint(lo, hi + 1, (cfg.num_seqs,), generator=g, dtype=torch.int64).to(torch.int32)


def draw_block_tables(context_lens: torch.Tensor, block_size: int, max_blocks_per_seq: int,
                      num_blocks: Optional[int], seed: int):
    """Deal a seeded permutation of the physical pool out to the sequences.

    Returns (block_tables int32 [B][max_blocks_per_seq], num_blocks).
    """
    lens = [int(x) for x in context_lens.tolist()]
    per_seq = [(n + block_size - 1) // block_size for n in lens]
    needed = sum(per_seq)
    if num_blocks is None:
        num_blocks = max(1, math.ceil(1.1 * needed))
    if num_blocks < needed:
        raise ValueError(f"pool of {num_blocks} blocks cannot hold {needed}")
    g = torch.Generator().manual_seed(seed + 7919)
    perm = torch.randperm(num_blocks, generator=g)[:needed].to(torch.int32)
    bt = torch.full((len(lens), max(1, max_blocks_per_seq)), -1, dtype=torch.int32)
    pos = 0
    for b, nb in enumerate(per_seq):
        if nb > max_blocks_per_seq:
            raise ValueError("context longer than the block table row")
        bt[b, :nb] = perm[pos:pos + nb]
        pos += nb
    return bt, num_blocks


def randn_f16(shape, generator: torch.Generator, device) -> torch.Tensor:
    """~N(0,1) fp32 draws rounded to fp16, generated in slices to bound memory."""
    out = torch.empty(shape, dtype=torch.float16, device=device)
    flat = out.view(-1)
    step = 1 << 26
    for s in range(0, flat.numel(), step):
        e = min(flat.numel(), s + step)
        flat[s:e] = torch.randn(e - s, generator=generator, device=device,
                                dtype=torch.float32).to(torch.float16)
    return out


# Per-cache scales (k_scale, v_scale) that go with each code set of rand_e4m3:
# they keep the scores of N(0,1) queries at a few units and |V| at most 1.75
# (448 / 256), so an fp16 output stays well inside the parity tolerance's
# range.  For the code sets, 448 = 0x7e and the subnormals are m * 2^-9.
E4M3_SCALES = {
    "full": (1.0 / 64, 1.0 / 256),
    "narrow": (0.05, 0.11),
    "max": (1.0 / 448, 1.0 / 256),
    "subnormal": (64.0, 64.0),
}


def rand_e4m3(shape, generator: torch.Generator, device, codes: str = "full") -> torch.Tensor:
    """Random E4M3 bit patterns (uint8), never a NaN code (0x7f, 0xff).  A
    bit-pattern generator: no rounding or scaling.

    codes:
      "full"       uniform over the 254 finite codes: +-0, the subnormals
                   (exponent field 0), every normal exponent 1..15, and the
                   largest magnitude 448 (0x7e, 0xfe)
      "narrow"     random sign and mantissa, biased exponent uniform in
                   [4, 10] (magnitudes 2^-3 .. 2^4)
      "max"        only +-448
      "subnormal"  only the exponent field 0: +-0 and the seven subnormal
                   magnitudes m * 2^-9
    """
    n = 1
    for x in shape:
        n *= int(x)
    bits = torch.randint(0, 1 << 16, (n,), generator=generator, device=device, dtype=torch.int32)
    sign = (bits & 1) << 7
    if codes == "full":
        r = (bits >> 1) % 254                  # 0..253 -> codes 0x00..0x7e, 0x80..0xfe
        code = torch.where(r < 127, r, r + 1)
    elif codes == "narrow":
        mant = (bits >> 1) & 7
        expo = 4 + ((bits >> 4) % 7)
        code = sign | (expo << 3) | mant
    elif codes == "max":
        code = sign | 0x7E
    elif codes == "subnormal":
        code = sign | ((bits >> 1) & 7)
    else:
        raise ValueError(f"unknown E4M3 code set {codes!r}")
    return code.to(torch.uint8).view(*shape)


def make_inputs(cfg: DecodeConfig, device="cpu", context_lens: Optional[torch.Tensor] = None,
                max_blocks_per_seq: Optional[int] = None) -> DecodeInputs:
    """Draw every tensor of ``cfg`` with its seed; q/k/v are drawn on ``device``."""
    device = torch.device(device)
    lens = draw_context_lens(cfg) if context_lens is None else context_lens.to(torch.int32).cpu()
    max_len = int(lens.max().item()) if lens.numel() else 0
    if max_blocks_per_seq is None:
        # size the table row for the longest length the config can draw
        row_len = max(max_len, cfg.max_context_len) if context_lens is None else max_len
        max_blocks_per_seq = max(1, (row_len + cfg.block_size - 1) // cfg.block_size)
    bt, nb = draw_block_tables(lens, cfg.block_size, max_blocks_per_seq, cfg.num_blocks, cfg.seed)
    g = torch.Generator(device=device).manual_seed(cfg.seed + 1)
    q = randn_f16((cfg.num_seqs, cfg.num_q_heads, cfg.head_dim), g, device)
    kshape = (nb, cfg.num_kv_heads, cfg.block_size, cfg.head_dim)
    k = randn_f16(kshape, g, device)
    v = randn_f16(kshape, g, device)
    return DecodeInputs(q=q, k_cache=k, v_cache=v, block_tables=bt.to(device),
                        context_lens=lens.to(device), num_seqs=cfg.num_seqs,
                        num_q_heads=cfg.num_q_heads, num_kv_heads=cfg.num_kv_heads,
                        head_dim=cfg.head_dim, block_size=cfg.block_size, num_blocks=nb,
                        max_blocks_per_seq=max_blocks_per_seq, max_context_len=max_len,
                        scale=cfg.scale)


def make_custom(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, context_lens,
                seed=0, num_blocks=None, device="cpu", max_blocks_per_seq=None,
                partition_size=0) -> DecodeInputs:
    """Inputs for an ad-hoc shape (tests): explicit lengths, same recipe."""
    cfg = DecodeConfig("custom", num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                       context_lens=tuple(int(x) for x in context_lens),
                       num_blocks=num_blocks, partition_size=partition_size, seed=seed)
    lens = torch.tensor([int(x) for x in context_lens], dtype=torch.int32)
    return make_inputs(cfg, device=device, context_lens=lens, max_blocks_per_seq=max_blocks_per_seq)
