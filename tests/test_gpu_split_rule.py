"""GPU parity at the partitions the small-grid split picks.

A call whose (sequence, kv head) units cover less than one resident wave takes the
shortest power-of-two partition whose grid still fits that wave: down to 128 tokens on
the mma.sync path, up to 4096 and more on the tcgen05 path.  Each case checks the plan
picks that partition, runs the automatic call, and compares every output row with the
fp64 oracle (E4M3 also against the element bound of the tensor-core arithmetic).
"""
import pytest
import torch

import oracle
from helpers import assert_close, assert_close_weighted, e4m3_magnitudes, oracle_out
from paged_kv_decode_21_gb300 import ops, workloads

pytestmark = pytest.mark.gpu

KS, VS = workloads.E4M3_SCALES["full"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_decode_21_gb300 import build
    build.build()
    ops.lib()


def slots(path_ctas_per_sm):
    return torch.cuda.get_device_properties(0).multi_processor_count * path_ctas_per_sm


@pytest.mark.parametrize("fp8", [False, True])
@pytest.mark.parametrize("B,Hq,Hkv,L", [(1, 32, 8, 2048), (1, 28, 4, 8192), (4, 32, 32, 2048), (3, 32, 8, 3000)])
def test_single_query_small_grid(B, Hq, Hkv, L, fp8):
    lens = [L] + [max(1, L - 997 * i) for i in range(1, B)]  # the longest first, the rest shorter
    inp = workloads.make_custom(B, Hq, Hkv, 128, 16, lens, seed=B + Hkv, device="cuda")
    n, P, _, var, grid, _ = ops.paged_decode_call_plan(B, 1, Hq, Hkv, 128, 16, L, kv_fp8=fp8)
    assert var == "tma_mma" and 128 <= P <= 2048 and grid <= slots(3)
    assert P == 128 or B * Hkv * -(-L // (P // 2)) > slots(3)
    ew = torch.zeros(1, dtype=torch.int32, device="cuda")
    if fp8:
        g = torch.Generator(device="cuda").manual_seed(11)
        k8 = workloads.rand_e4m3(inp.k_cache.shape, g, "cuda")
        v8 = workloads.rand_e4m3(inp.v_cache.shape, g, "cuda")
        out = ops.paged_decode_attention_fp8(inp.q, k8, v8, inp.block_tables, inp.context_lens, inp.scale, KS, VS,
                                             max_context_len=L, error_word=ew)
        host = (inp.block_tables.cpu(), inp.context_lens.cpu())
        ref = oracle.attention_fp8(inp.q.cpu(), k8.cpu(), v8.cpu(), *host, inp.scale, KS, VS)
        absref = oracle.attention_fp8(inp.q.cpu(), k8.cpu(), e4m3_magnitudes(v8).cpu(), *host, inp.scale, KS, VS)
        assert_close_weighted(out, ref, absref, 448.0 * VS, L, f"E4M3 P={P}")
    else:
        out = ops.paged_decode_attention_ex(inp.q, inp.k_cache, inp.v_cache, inp.block_tables, inp.context_lens,
                                            inp.scale, max_context_len=L, error_word=ew)
        assert_close(out, oracle_out(inp), f"fp16 P={P}")
    assert ops.pkd_read_device_error(ew) == 0


@pytest.mark.parametrize("fp8", [False, True])
@pytest.mark.parametrize("B,Hq,Hkv,L", [(16, 32, 8, 8192), (1, 28, 4, 2048), (3, 28, 4, 5000)])
def test_multi_token_small_grid_on_tcgen05(B, Hq, Hkv, L, fp8):
    q_len = 8
    lens = [L] + [max(q_len, L - 1999 * i) for i in range(1, B)]
    inp = workloads.make_custom(B, Hq, Hkv, 128, 16, lens, seed=B + 3, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(13)
    q = workloads.randn_f16((B, q_len, Hq, 128), g, "cuda")
    n, P, _, var, grid, _ = ops.paged_decode_call_plan(B, q_len, Hq, Hkv, 128, 16, L, kv_fp8=fp8)
    assert var.startswith("tcgen05") and 256 <= P <= 8192 and grid <= slots(2)
    assert P == 256 or B * Hkv * -(-L // (P // 2)) > slots(2)
    ew = torch.zeros(1, dtype=torch.int32, device="cuda")
    host = (inp.block_tables.cpu(), inp.context_lens.cpu())
    if fp8:
        k8 = workloads.rand_e4m3(inp.k_cache.shape, g, "cuda")
        v8 = workloads.rand_e4m3(inp.v_cache.shape, g, "cuda")
        out = ops.paged_decode_attention_fp8(q, k8, v8, inp.block_tables, inp.context_lens, inp.scale, KS, VS,
                                             max_context_len=L, error_word=ew)
        ref = oracle.attention_fp8(q.cpu(), k8.cpu(), v8.cpu(), *host, inp.scale, KS, VS)
        absref = oracle.attention_fp8(q.cpu(), k8.cpu(), e4m3_magnitudes(v8).cpu(), *host, inp.scale, KS, VS)
        assert_close_weighted(out, ref, absref, 448.0 * VS, L, f"E4M3 q_len=8 P={P}")
    else:
        out = ops.paged_decode_attention_multi(q, inp.k_cache, inp.v_cache, inp.block_tables, inp.context_lens,
                                               inp.scale, max_context_len=L, error_word=ew)
        ref = oracle.attention_multi(q.cpu(), inp.k_cache.cpu(), inp.v_cache.cpu(), *host, inp.scale)
        assert_close(out, ref, f"fp16 q_len=8 P={P}")
    assert ops.pkd_read_device_error(ew) == 0


@pytest.mark.parametrize("B,Hq,q_len,P,fp8", [(16, 40, 8, 512, False), (16, 40, 8, 512, True),
                                              (16, 40, 4, 256, False), (16, 40, 8, 256, True),
                                              (64, 28, 8, 1024, False), (32, 40, 4, 1024, True)])
def test_tcgen05_partition_runs(B, Hq, q_len, P, fp8):
    # Many units at a short explicit partition: the tcgen05 plan gives each CTA a run of
    # consecutive partitions (fewer CTAs than partitions), each partial written on its own.
    # Ragged lengths put runs across the end of a sequence, a last run shorter than the others,
    # and sequences shorter than a partition or than the query tokens.
    Hkv = 8 if Hq == 40 else 4
    rng = torch.Generator().manual_seed(31 + P + q_len)
    lens = torch.randint(1, 16385, (B,), generator=rng).tolist()
    lens[:6] = [16384, 0, 5, P - 1, 3 * P + 1, 16384 - P]
    L = max(lens)
    inp = workloads.make_custom(B, Hq, Hkv, 128, 16, lens, seed=33, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(34)
    q = workloads.randn_f16((B, q_len, Hq, 128), g, "cuda")
    n, part, _, var, grid, _ = ops.paged_decode_call_plan(B, q_len, Hq, Hkv, 128, 16, L, kv_fp8=fp8, partition_size=P)
    units, npart = B * Hkv, -(-L // P)
    assert var == "tcgen05" and part == P and grid < units * npart  # runs of partitions
    ew = torch.zeros(1, dtype=torch.int32, device="cuda")
    host = (inp.block_tables.cpu(), inp.context_lens.cpu())
    if fp8:
        k8 = workloads.rand_e4m3(inp.k_cache.shape, g, "cuda")
        v8 = workloads.rand_e4m3(inp.v_cache.shape, g, "cuda")
        out = ops.paged_decode_attention_fp8(q, k8, v8, inp.block_tables, inp.context_lens, inp.scale, KS, VS,
                                             max_context_len=L, partition_size=P, error_word=ew)
        ref = oracle.attention_fp8(q.cpu(), k8.cpu(), v8.cpu(), *host, inp.scale, KS, VS)
        absref = oracle.attention_fp8(q.cpu(), k8.cpu(), e4m3_magnitudes(v8).cpu(), *host, inp.scale, KS, VS)
        assert_close_weighted(out, ref, absref, 448.0 * VS, L, "E4M3 runs")
    else:
        out = ops.paged_decode_attention_multi(q, inp.k_cache, inp.v_cache, inp.block_tables, inp.context_lens,
                                               inp.scale, max_context_len=L, partition_size=P, error_word=ew)
        ref = oracle.attention_multi(q.cpu(), inp.k_cache.cpu(), inp.v_cache.cpu(), *host, inp.scale)
        assert_close(out, ref, "fp16 runs")
    assert ops.pkd_read_device_error(ew) == 0


def tail_seqs(B, Hkv, q_chunks=1):
    # sequences the longest-first order of a tcgen05 grid splits in two: the last round of
    # resident CTAs (two per SM) at most half full
    slots = slots_of(2)
    units = B * Hkv * q_chunks
    last = units - (units - 1) // slots * slots
    return -(-last // (Hkv * q_chunks)) if units > slots and 2 * last <= slots else 0


def slots_of(per_sm):
    return torch.cuda.get_device_properties(0).multi_processor_count * per_sm


@pytest.mark.parametrize("fp8", [False, True])
@pytest.mark.parametrize("kind", ["uniform", "ragged", "tiny", "mostly_empty", "gqa4", "q_len4"])
def test_tcgen05_tail_split(kind, fp8):
    # An unsplit tcgen05 grid walked longest first whose last round is short: of the K shortest
    # sequences the order kernel splits those at least half as long as the longest in two
    # halves, each CTA of a half writes a partial, and the merge combines those sequences only.
    # Ragged lengths put shorter sequences among the K (they stay whole); "tiny" contexts (the
    # longest 130 tokens) split sequences of 65-130 tokens, whose second half can be one token,
    # next to whole ones of 1-64 tokens, shorter than the query; a mostly empty batch has fewer
    # sequences with tokens than K (the order pads with empty slots).
    Hq, Hkv, q_len = (32, 8, 8) if kind == "gqa4" else (28, 4, 4 if kind == "q_len4" else 8)
    B = -(-(slots_of(2) * 2 + 32) // Hkv)  # two full rounds and a short third one
    L = 2048
    if kind == "ragged":
        rng = torch.Generator().manual_seed(41)
        lens = torch.randint(1024, L + 1, (B,), generator=rng).tolist()
        lens[:10] = [L, 0, 1, 5, 64, 65, 100, 129, 700, 0]
    elif kind == "tiny":
        rng = torch.Generator().manual_seed(42)
        lens = torch.randint(65, 131, (B,), generator=rng).tolist()
        lens[:10] = [130, 0, 1, 5, 64, 65, 66, 100, 127, 129]
    elif kind == "mostly_empty":
        lens = [0] * B
        lens[3], lens[7], lens[20] = L, 1500, 90
    else:
        lens = [L] * B
    K = tail_seqs(B, Hkv)
    assert K > 0
    n, part, ordered, var, grid, _ = ops.paged_decode_call_plan(B, q_len, Hq, Hkv, 128, 16, L, kv_fp8=fp8)
    assert var.startswith("tcgen05") and part == -1 and ordered and grid == (B + K) * Hkv and n == 3
    # table rows of L tokens: the call passes max_context_len = L whatever the lengths
    inp = workloads.make_custom(B, Hq, Hkv, 128, 16, lens, seed=43, device="cuda", max_blocks_per_seq=L // 16)
    g = torch.Generator(device="cuda").manual_seed(44)
    q = workloads.randn_f16((B, q_len, Hq, 128), g, "cuda")
    ew = torch.zeros(1, dtype=torch.int32, device="cuda")
    host = (inp.block_tables.cpu(), inp.context_lens.cpu())
    if fp8:
        k8 = workloads.rand_e4m3(inp.k_cache.shape, g, "cuda")
        v8 = workloads.rand_e4m3(inp.v_cache.shape, g, "cuda")
        out = ops.paged_decode_attention_fp8(q, k8, v8, inp.block_tables, inp.context_lens, inp.scale, KS, VS,
                                             max_context_len=L, error_word=ew)
        ref = oracle.attention_fp8(q.cpu(), k8.cpu(), v8.cpu(), *host, inp.scale, KS, VS)
        absref = oracle.attention_fp8(q.cpu(), k8.cpu(), e4m3_magnitudes(v8).cpu(), *host, inp.scale, KS, VS)
        assert_close_weighted(out, ref, absref, 448.0 * VS, L, f"E4M3 tail split {kind}")
    else:
        out = ops.paged_decode_attention_multi(q, inp.k_cache, inp.v_cache, inp.block_tables, inp.context_lens,
                                               inp.scale, max_context_len=L, error_word=ew)
        ref = oracle.attention_multi(q.cpu(), inp.k_cache.cpu(), inp.v_cache.cpu(), *host, inp.scale)
        assert_close(out, ref, f"fp16 tail split {kind}")
    assert ops.pkd_read_device_error(ew) == 0
    # the same call with a workspace too small for the tail split runs it unsplit, to the same result
    if not fp8:
        small = ops.alloc_workspace(ops.paged_decode_workspace_size(B, Hq, Hkv, 128, 16, L, -1, "tcgen05+longest_first"),
                                    "cuda")
        out2 = ops.paged_decode_attention_multi(q, inp.k_cache, inp.v_cache, inp.block_tables, inp.context_lens,
                                                inp.scale, max_context_len=L, workspace=small, error_word=ew)
        assert_close(out2, ref, f"fp16 tail split {kind}, small workspace")
        assert ops.pkd_read_device_error(ew) == 0
