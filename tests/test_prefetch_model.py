"""The rule that sizes the default L2 prefetch distance, pinned on the CPU.

pkd_l2_prefetch_model restates the L2 capacity model of the review
"Accelerating LLM Inference Throughput via Asynchronous KV Cache
Prefetching", section 4.2 (M_block = b * d_h * T_block, M_total = M_block *
(N_thread / 32) * H * B must fit in L2), and adds a Little's-law lower bound
(bytes in flight per SM against bandwidth x latency).  Pinned here by the
review's worked example (a 60 MB L2 holds the blocks of at most 120 batches),
by the closed forms of the footprint and the need, by monotonicity, and by
the choices it makes for the GB300 workloads of this library: distance 1 for
the CUDA-core L2-prefetch path, none for the staged and tensor-core paths
whose rings of copies already keep enough bytes in flight.
"""
import json
import os

import pytest

from paged_kv_decode_21_gb300 import build as pkd_build
from paged_kv_decode_21_gb300 import traffic, workloads

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_numbers.json")))
# a GB300 described by its numbers: 152 SMs, the L2 size the device reports,
# nominal HBM3e bandwidth 2 x 3996 MHz x 8192 bits
GB300 = dict(sm_count=152, l2_bytes=136314880, hbm_bytes_per_s=2 * 3996e6 * 8192 / 8)
LATENCY, FRACTION, MAX_D = 1.5e-6, 0.125, 8


@pytest.fixture(scope="module")
def ops():
    pkd_build.build()
    from paged_kv_decode_21_gb300 import ops as o
    o.lib()
    return o


def test_worked_example_of_the_capacity_model(ops):
    # the review's numbers: M_block from b=2, d_h=128, T_block=16; N_thread=128 (4 warps),
    # H=32 heads, a 60 MB L2; one tile per warp per iteration, every CTA resident.  No bytes
    # in flight without prefetching, so the need asks for a distance of at least 1, which
    # fits while the batch stays within the 120 the review prints, and not past it.
    g = GOLD["l2_resident_batches"]
    mb = traffic.m_block(2, 128, 16)
    assert mb == GOLD["m_block"]["value"]
    warps, H, B = g["n_thread"] // 32, g["num_heads"], g["value"]

    def model(batch):
        return ops.pkd_l2_prefetch_model(H * batch, 132, warps, mb, 1, 0, g["l2_bytes"], 1.0, 4e12, LATENCY, MAX_D)

    d, footprint, _, _ = model(B)
    assert d == 1 and footprint == traffic.m_total(mb, g["n_thread"], H, B) == g["l2_bytes"]
    assert model(B + 1)[0] == 0
    assert traffic.l2_resident_batches(g["l2_bytes"], mb, g["n_thread"], H) == B


def test_closed_forms(ops):
    # resident 600 CTAs on 152 SMs, 4 streams, 4 KiB tiles, K and V per step, 16 KiB ahead per CTA
    d, fp, inflight, need = ops.pkd_l2_prefetch_model(600, 152, 4, 4096, 2, 16384, 1 << 30, 1.0, 8e12, 2e-6, 8)
    assert need == int(8e12 / 152 * 2e-6)
    step = 4 * 2 * 4096
    # the smallest d whose bytes in flight per SM reach the need
    per_sm = 600 / 152
    assert per_sm * (16384 + d * step) >= need > per_sm * (16384 + (d - 1) * step)
    assert fp == 600 * d * step and inflight == int(per_sm * (16384 + d * step))
    # bytes already in flight that cover the need: no prefetch
    assert ops.pkd_l2_prefetch_model(600, 152, 4, 4096, 2, 10 ** 6, 1 << 30, 1.0, 8e12, 2e-6, 8)[0] == 0
    # a 10 us latency asks for 5 (600/152 CTAs x 5 x 32 KiB per SM >= 8e12 / 152 x 1e-5);
    # the capacity cap lowers d until the footprint fits (here: to 2, then 1)
    assert ops.pkd_l2_prefetch_model(600, 152, 4, 4096, 2, 0, 1 << 30, 1.0, 8e12, 1e-5, 8)[0] == 5
    cap = 600 * 2 * step
    assert ops.pkd_l2_prefetch_model(600, 152, 4, 4096, 2, 0, cap, 1.0, 8e12, 1e-5, 8)[0] == 2
    assert ops.pkd_l2_prefetch_model(600, 152, 4, 4096, 2, 0, cap - 1, 1.0, 8e12, 1e-5, 8)[0] == 1
    assert ops.pkd_l2_prefetch_model(600, 152, 4, 4096, 2, 0, cap, 0.5, 8e12, 1e-5, 8)[0] == 1
    # fewer CTAs than SMs: each SM has one CTA and must cover a larger share of the bandwidth
    d1 = ops.pkd_l2_prefetch_model(76, 152, 4, 4096, 2, 16384, 1 << 30, 1.0, 8e12, 2e-6, 8)
    assert d1[3] == int(8e12 / 76 * 2e-6)
    # invalid descriptions
    with pytest.raises(ops.PagedDecodeError):
        ops.pkd_l2_prefetch_model(10, 0, 4, 4096, 2, 0, 1 << 20, 1.0, 8e12, 1e-6, 8)
    with pytest.raises(ops.PagedDecodeError):
        ops.pkd_l2_prefetch_model(10, 152, 4, 4096, 2, 0, 1 << 20, -0.5, 8e12, 1e-6, 8)


def test_distance_never_grows_with_more_ctas(ops):
    last = None
    for resident in [1, 8, 40, 152, 304, 456, 1000, 5000]:
        d = ops.pkd_l2_prefetch_model(resident, 152, 4, 4096, 2, 32768, 136314880, FRACTION, 8.18e12, LATENCY,
                                      MAX_D)[0]
        assert last is None or d <= last
        last = d


@pytest.mark.parametrize("name", ["llama2_7b_mha", "llama3_8b_gqa4", "qwen25_7b_gqa7", "qwen25_14b_gqa5_splitk"])
def test_gb300_choices_on_the_large_workloads(ops, name):
    c = workloads.CONFIGS[name]
    P = c.partition_size or -1
    expect = {"l2_prefetch": 1, "tma_staged": 0, "tma_mma": 0, "no_prefetch": 0, "tcgen05": 0}
    for variant, want in expect.items():
        d, fp, inflight, need = ops.paged_decode_prefetch_model(
            c.num_seqs, 1, c.num_q_heads, c.num_kv_heads, c.head_dim, c.block_size, c.max_context_len,
            partition_size=P, variant=variant, **GB300)
        assert d == want, (variant, d, inflight, need)
        assert fp <= FRACTION * GB300["l2_bytes"]
    # the CUDA-core path: 2 CTAs x 4 warps x one 16-row group of K and V (8 KiB) per SM is
    # short of bandwidth x latency; distance 1 adds one block of K and V per warp
    d, fp, inflight, need = ops.paged_decode_prefetch_model(
        c.num_seqs, 1, c.num_q_heads, c.num_kv_heads, 128, 16, c.max_context_len, partition_size=P,
        variant="l2_prefetch", **GB300)
    assert need == int(GB300["hbm_bytes_per_s"] / 152 * LATENCY)
    assert inflight == 2 * 4 * (8192 + 8192) and fp == 2 * 152 * 4 * 8192


def test_small_grids_prefetch_further(ops):
    # 8 sequences x 4 kv heads of 8192 tokens: 32 CTAs, one per SM; each must keep its SM's
    # larger share of the bandwidth in flight, so the CUDA-core path prefetches further ahead,
    # up to the largest distance (32 KiB per unit cannot reach 8.18e12 / 32 x 1.5 us)
    d, fp, inflight, need = ops.paged_decode_prefetch_model(8, 1, 32, 4, 128, 16, 8192, partition_size=-1,
                                                            variant="l2_prefetch", **GB300)
    assert d == MAX_D and inflight == 32768 * (1 + MAX_D) < need and fp <= FRACTION * GB300["l2_bytes"]
    # 64 sequences x 8 kv heads: 512 CTAs, two resident per SM, reach it at distance 1
    d, _, inflight, need = ops.paged_decode_prefetch_model(64, 1, 32, 8, 128, 16, 8192, partition_size=-1,
                                                           variant="l2_prefetch", **GB300)
    assert d == 1 and inflight >= need
    # a warp's share of a short partition bounds it: 64 tokens = 4 blocks over 4 warps
    d, _, _, _ = ops.paged_decode_prefetch_model(8, 1, 32, 4, 128, 16, 8192, partition_size=64,
                                                 variant="l2_prefetch", **GB300)
    assert d == 0
