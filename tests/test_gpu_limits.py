"""GPU parity at the sizes where the library's limits sit.

* One sequence of 131,072 tokens (and one with a ragged tail): unsplit, at the
  automatic split, and split into 32-token partitions, so the split-K merge
  combines 4097 partitions; on every data path, over E4M3 caches and as a
  multi-token query on the tcgen05 path.
* Batches of 4096 sequences (the most the longest-first order kernel holds) and
  4097 (one past it: the order is skipped and the plain grid order runs), with
  the order requested: the results are bitwise those of the plain order.
* The largest group size (8) at head_dim 64 and block size 32.

Every output row is compared with the fp64 oracle.
"""
import pytest
import torch

import oracle
from helpers import assert_close, assert_close_weighted, e4m3_magnitudes, oracle_out
from paged_kv_decode_21_gb300 import ops, workloads

pytestmark = pytest.mark.gpu

VARIANTS = ["no_prefetch", "l2_prefetch", "tma_staged", "tma_mma"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_decode_21_gb300 import build
    build.build()
    ops.lib()


def run(inp, variant, partition, **kw):
    return ops.paged_decode_attention_ex(inp.q, inp.k_cache, inp.v_cache, inp.block_tables, inp.context_lens,
                                         inp.scale, max_context_len=inp.max_context_len, partition_size=partition,
                                         variant=variant, **kw)


@pytest.mark.parametrize("length", [131072, 131072 + 5])
def test_longest_context_every_path_and_split(length):
    # G = 8: one kv head serves 8 query heads; 32-token partitions make 4097 partials to merge
    inp = workloads.make_custom(1, 8, 1, 128, 16, [length], seed=5, device="cuda")
    ref = oracle_out(inp)
    for variant in VARIANTS:
        for partition in (-1, 0, 32):
            ew = torch.zeros(1, dtype=torch.int32, device="cuda")
            out = run(inp, variant, partition, error_word=ew)
            assert ops.pkd_read_device_error(ew) == 0
            assert_close(out, ref, f"L={length} {variant} P={partition}")


def test_longest_context_e4m3_and_tcgen05():
    length = 131072 + 5
    inp = workloads.make_custom(1, 8, 1, 128, 16, [length], seed=6, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(7)
    ks, vs = workloads.E4M3_SCALES["full"]
    k8 = workloads.rand_e4m3(inp.k_cache.shape, g, "cuda")
    v8 = workloads.rand_e4m3(inp.v_cache.shape, g, "cuda")
    q8 = workloads.randn_f16((1, 8, 8, 128), g, "cuda")  # 8 query tokens x 8 heads: 64 query rows
    host = (inp.block_tables.cpu(), inp.context_lens.cpu())
    ref8 = oracle.attention_fp8(inp.q.cpu(), k8.cpu(), v8.cpu(), *host, inp.scale, ks, vs)
    abs8 = oracle.attention_fp8(inp.q.cpu(), k8.cpu(), e4m3_magnitudes(v8).cpu(), *host, inp.scale, ks, vs)
    refm = oracle.attention_multi(q8.cpu(), inp.k_cache.cpu(), inp.v_cache.cpu(), *host, inp.scale)
    for partition in (-1, 0, 512):
        for variant in ("tma_mma", "tcgen05"):
            out = ops.paged_decode_attention_fp8(inp.q, k8, v8, inp.block_tables, inp.context_lens, inp.scale,
                                                 ks, vs, max_context_len=inp.max_context_len,
                                                 partition_size=partition, variant=variant)
            assert_close_weighted(out, ref8, abs8, 448.0 * vs, length, f"E4M3 {variant} P={partition}")
        outm = ops.paged_decode_attention_multi(q8, inp.k_cache, inp.v_cache, inp.block_tables, inp.context_lens,
                                                inp.scale, max_context_len=inp.max_context_len,
                                                partition_size=partition, variant="tcgen05")
        assert_close(outm, refm, f"tcgen05 q_len=8 P={partition}")


@pytest.mark.parametrize("num_seqs", [4096, 4097])
def test_order_at_and_past_its_capacity(num_seqs):
    lens = torch.randint(1, 400, (num_seqs,), generator=torch.Generator().manual_seed(num_seqs)).tolist()
    inp = workloads.make_custom(num_seqs, 2, 1, 64, 16, lens, seed=num_seqs, device="cuda")
    need = ops.paged_decode_workspace_size(num_seqs, 2, 1, 64, 16, inp.max_context_len, -1,
                                           "tma_mma+longest_first")
    ws = ops.alloc_workspace(need, "cuda")
    plain = run(inp, "tma_mma", -1)
    ordered = run(inp, "tma_mma+longest_first", -1, workspace=ws)
    assert torch.equal(plain, ordered)
    assert_close(ordered, oracle_out(inp), f"{num_seqs} sequences")


def test_largest_group_head_dim_64_block_32():
    lens = [1, 31, 32, 33, 5000, 16384]
    inp = workloads.make_custom(len(lens), 16, 2, 64, 32, lens, seed=9, device="cuda")
    ref = oracle_out(inp)
    for variant in VARIANTS:
        for partition in (-1, 0, 64):
            assert_close(run(inp, variant, partition), ref, f"G=8 D=64 BS=32 {variant} P={partition}")
