"""GPU parity of multi-token queries (q_len > 1, causal among the new tokens).

paged_decode_attention_multi is called through the C ABI and compared
element by element with ``oracle.attention_multi`` (max |err| <= 4e-3, mean
<= 5e-4).  The shapes cover every group size's query chunking (one chunk of
16 / G query tokens per CTA, and a ragged second chunk), sequences shorter
than q_len (queries that see no token give zeros), split and unsplit
contexts, and a full-size GQA workload on sampled rows.
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import assert_close, sample_rows
from paged_kv_decode_21_gb300 import ops, workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_decode_21_gb300 import build
    build.build()
    ops.lib()


def make(lens, q_len, Hq, Hkv, D, BS, seed):
    inp = workloads.make_custom(len(lens), Hq, Hkv, D, BS, lens, seed=seed, device="cuda",
                                max_blocks_per_seq=-(-max(max(lens), 1) // BS) + 1)
    g = torch.Generator(device="cuda").manual_seed(seed + 5)
    q = workloads.randn_f16((len(lens), q_len, Hq, D), g, "cuda")
    return inp, q


def oracle_multi(inp, q, rows=None):
    return oracle.attention_multi(q.cpu(), inp.k_cache.cpu(), inp.v_cache.cpu(), inp.block_tables.cpu(),
                                  inp.context_lens.cpu(), inp.scale, rows=rows)


def run_multi(inp, q, partition, **kw):
    return ops.paged_decode_attention_multi(q, inp.k_cache, inp.v_cache, inp.block_tables,
                                            inp.context_lens, inp.scale,
                                            max_context_len=inp.max_context_len,
                                            partition_size=partition, **kw)


SHAPES = [
    # (D, BS, Hq, Hkv, lens, q_len)
    (128, 16, 4, 4, [20, 100, 3], 2),          # G=1: one chunk of 16
    (128, 16, 4, 4, [50, 17], 16),
    (128, 16, 4, 4, [40, 300], 17),            # G=1: a second chunk of one token
    (128, 16, 32, 8, [64, 129, 513], 4),       # G=4: one chunk of 4
    (128, 16, 32, 8, [300, 33], 5),            # G=4: chunks of 4 + 1
    (128, 16, 28, 4, [0, 5, 257, 700], 2),     # G=7: one chunk of 2
    (128, 16, 28, 4, [90, 31], 3),             # G=7: chunks of 2 + 1
    (128, 16, 40, 8, [200, 64], 3),            # G=5: one chunk of 3
    (128, 32, 16, 2, [2, 100], 4),             # G=8: chunks of 2 + 2; L < q_len
    (128, 16, 12, 2, [77, 1], 2),              # G=6
    (128, 16, 6, 2, [150, 16], 6),             # G=3: chunks of 5 + 1
    (128, 16, 4, 2, [45, 99], 9),              # G=2: chunks of 8 + 1
    (64, 32, 14, 2, [1, 63, 64, 65, 190], 3),  # D=64, BS=32, G=7
    (64, 16, 4, 4, [37, 100], 5),              # D=64, G=1
]


@pytest.mark.parametrize("shape", SHAPES,
                         ids=lambda s: f"D{s[0]}BS{s[1]}G{s[2] // s[3]}Q{s[5]}")
@pytest.mark.parametrize("partition", [-1, 64, 0])
def test_multi_query_matches_oracle(shape, partition):
    D, BS, Hq, Hkv, lens, q_len = shape
    inp, q = make(lens, q_len, Hq, Hkv, D, BS, seed=D + BS + Hq + q_len)
    ew = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = run_multi(inp, q, partition, error_word=ew)
    assert ops.pkd_read_device_error(ew) == 0
    assert_close(out, oracle_multi(inp, q), f"{shape} P={partition}")


def test_short_sequences_give_zeros_for_blind_queries():
    # L = 2 with q_len = 4: queries 0 and 1 sit before the sequence start
    inp, q = make([2, 3], 4, 8, 2, 128, 16, seed=3)
    out = run_multi(inp, q, -1, out=torch.full_like(q, float("nan"))).cpu()
    assert torch.all(out[0, :2] == 0) and torch.all(out[1, :1] == 0)
    assert torch.isfinite(out).all()
    assert_close(out, oracle_multi(inp, q.cpu()), "short sequences")


def test_q_len_one_is_single_query_decode():
    inp, q = make([300, 17, 129], 1, 28, 4, 128, 16, seed=7)
    for partition in (-1, 64):
        a = run_multi(inp, q, partition)
        b = ops.paged_decode_attention_ex(q.view(3, 28, 128), inp.k_cache, inp.v_cache, inp.block_tables,
                                          inp.context_lens, inp.scale, max_context_len=inp.max_context_len,
                                          partition_size=partition, variant="tma_mma")
        assert torch.equal(a.view(3, 28, 128), b)


def test_last_query_matches_single_query_decode():
    # the last new token sees the whole context, like a plain decode step
    inp, q = make([129, 64, 511], 4, 32, 8, 128, 16, seed=9)
    multi = run_multi(inp, q, 0)
    single = ops.paged_decode_attention_ex(q[:, -1].contiguous(), inp.k_cache, inp.v_cache,
                                           inp.block_tables, inp.context_lens, inp.scale,
                                           max_context_len=inp.max_context_len)
    ref = oracle.attention(q[:, -1].cpu(), inp.k_cache.cpu(), inp.v_cache.cpu(), inp.block_tables.cpu(),
                           inp.context_lens.cpu(), inp.scale)
    assert_close(multi[:, -1], ref, "last query")
    assert_close(single, ref, "single query")


def test_multi_query_nan_poison_in_unused_slots():
    lens = [21, 9, 70]
    inp, q = make(lens, 3, 8, 2, 128, 16, seed=13)
    used = torch.zeros(inp.num_blocks, 16, dtype=torch.bool)
    for b, L in enumerate(lens):
        for t in range(L):
            used[int(inp.block_tables[b, t // 16]), t % 16] = True
    a = run_multi(inp, q, -1)
    mask = (~used).cuda()
    inp.k_cache.permute(0, 2, 1, 3)[mask] = float("nan")
    inp.v_cache.permute(0, 2, 1, 3)[mask] = float("nan")
    b = run_multi(inp, q, -1)
    assert torch.isfinite(b).all()
    assert torch.equal(a, b)


def test_multi_query_full_size_gqa_all_rows():
    # Llama3-8B shape (128 sequences, 32 q / 8 kv heads, contexts U[512, 4096])
    # verifying 4 draft tokens per sequence, at the automatic split
    cfg = workloads.CONFIGS["llama3_8b_gqa4"]
    inp = workloads.make_inputs(cfg, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(77)
    q = workloads.randn_f16((cfg.num_seqs, 4, cfg.num_q_heads, cfg.head_dim), g, "cuda")
    ew = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = run_multi(inp, q, 0, error_word=ew)
    assert ops.pkd_read_device_error(ew) == 0
    assert_close(out, oracle_multi(inp, q), "llama3_8b_gqa4 q_len=4")


def test_multi_query_automatic_order_is_bitwise_neutral():
    # ragged batch whose unsplit grid the automatic split walks longest first
    B, Hq, Hkv, q_len = 128, 32, 8, 2
    lens = torch.randint(1024, 4097, (B,), generator=torch.Generator().manual_seed(23)).tolist()
    inp, q = make(lens, q_len, Hq, Hkv, 128, 16, seed=23)
    n, part, ordered = ops.paged_decode_auto_plan(B, q_len, Hq, Hkv, 128, 16, inp.max_context_len)
    assert ordered and part == -1
    a = run_multi(inp, q, 0)
    b = run_multi(inp, q, -1)
    assert torch.equal(a, b)
    rows = sample_rows(B * q_len, Hq, 96, seed=23)
    got = a.view(-1, 128)[torch.from_numpy(rows).long().cuda()]
    assert_close(got, oracle_multi(inp, q, rows=rows), "multi longest first")
