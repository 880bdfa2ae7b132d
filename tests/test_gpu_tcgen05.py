"""GPU parity of the tcgen05 data path (PKD_VARIANT_TCGEN05).

The kernel keeps S = Q K^T and O in tensor memory and serves up to 64 query
rows (query tokens x group heads) per CTA.  It is called through the C ABI
and compared element by element with the fp64 oracle (max |err| <= 4e-3,
mean <= 5e-4), or checked for exact properties: a single token returns its
V row, a key spike selects its V row, the physical block placement, NaN in
unused cache slots, the L2 hints and the longest-first order change no bit.
Shapes cover every group size, both block sizes, partitions that split a
64-token tile and ones that do not, ragged last tiles, query chunks that fill
the 64 rows exactly and ones that spill one token into a second chunk.
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import assert_close, assert_close_weighted, e4m3_magnitudes, oracle_out, sample_rows
from paged_kv_decode_21_gb300 import ops, workloads

pytestmark = pytest.mark.gpu

TC = "tcgen05"


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_decode_21_gb300 import build
    build.build()
    ops.lib()


def errword():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


def run_ex(inp, variant=TC, partition_size=0, **kw):
    return ops.paged_decode_attention_ex(inp.q, inp.k_cache, inp.v_cache, inp.block_tables,
                                         inp.context_lens, inp.scale, max_context_len=inp.max_context_len,
                                         partition_size=partition_size, variant=variant, **kw)


def make_multi(lens, q_len, Hq, Hkv, BS, seed, D=128):
    inp = workloads.make_custom(len(lens), Hq, Hkv, D, BS, lens, seed=seed, device="cuda",
                                max_blocks_per_seq=-(-max(max(lens), 1) // BS) + 1)
    g = torch.Generator(device="cuda").manual_seed(seed + 5)
    q = workloads.randn_f16((len(lens), q_len, Hq, D), g, "cuda")
    return inp, q


def run_multi(inp, q, partition, variant=TC, **kw):
    return ops.paged_decode_attention_multi(q, inp.k_cache, inp.v_cache, inp.block_tables, inp.context_lens,
                                            inp.scale, max_context_len=inp.max_context_len,
                                            partition_size=partition, variant=variant, **kw)


def oracle_multi(inp, q, rows=None):
    return oracle.attention_multi(q.cpu(), inp.k_cache.cpu(), inp.v_cache.cpu(), inp.block_tables.cpu(),
                                  inp.context_lens.cpu(), inp.scale, rows=rows)


# --------------------------------------------------------------------------- single-query decode
SHAPES = [
    # (BS, Hq, Hkv, lens)
    (16, 4, 4, [1, 15, 16, 17, 63, 64, 65, 100, 333]),   # G=1
    (16, 28, 4, [0, 5, 31, 32, 33, 127, 128, 129, 700]),  # G=7
    (16, 32, 8, [64, 1, 129, 513]),                       # G=4
    (16, 40, 8, [300, 47]),                               # G=5
    (32, 16, 2, [1, 31, 32, 33, 250]),                    # G=8, BS=32
    (16, 6, 2, [90, 3]),                                  # G=3
    (16, 12, 2, [150]),                                   # G=6
    (32, 4, 2, [45, 99, 64]),                             # G=2, BS=32
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"BS{s[0]}G{s[1] // s[2]}")
@pytest.mark.parametrize("partition", [-1, 32, 64, 0])
def test_single_query_matches_oracle(shape, partition):
    BS, Hq, Hkv, lens = shape
    if partition == 32 and BS == 32:
        partition = 96  # a partition that splits a 64-token tile at block size 32
    inp = workloads.make_custom(len(lens), Hq, Hkv, 128, BS, lens, seed=BS + Hq, device="cuda",
                                max_blocks_per_seq=-(-max(lens) // BS) + 2)
    ew = errword()
    out = run_ex(inp, TC, partition, error_word=ew)
    assert ops.pkd_read_device_error(ew) == 0
    assert_close(out, oracle_out(inp), f"{shape} P={partition}")


HD64 = [
    # (BS, Hq, Hkv, lens): head_dim 64 (one 64-dim half per row)
    (16, 4, 4, [1, 37, 64, 65, 100]),
    (32, 14, 2, [1, 63, 64, 65, 190]),
    (16, 5, 1, [40, 128, 0]),
]


@pytest.mark.parametrize("shape", HD64, ids=lambda s: f"D64BS{s[0]}G{s[1] // s[2]}")
@pytest.mark.parametrize("partition", [-1, 64])
def test_head_dim_64_single_query_matches_oracle(shape, partition):
    BS, Hq, Hkv, lens = shape
    inp = workloads.make_custom(len(lens), Hq, Hkv, 64, BS, lens, seed=BS + Hq + 64, device="cuda",
                                max_blocks_per_seq=-(-max(lens) // BS) + 2)
    ew = errword()
    out = run_ex(inp, TC, partition, error_word=ew)
    assert ops.pkd_read_device_error(ew) == 0
    assert_close(out, oracle_out(inp), f"D64 {shape} P={partition}")


@pytest.mark.parametrize("shape", [(32, 14, 2, [1, 63, 64, 65, 190], 3), (16, 4, 4, [37, 100], 17),
                                   (16, 28, 4, [130, 5], 8)],
                         ids=lambda s: f"D64BS{s[0]}G{s[1] // s[2]}Q{s[4]}")
@pytest.mark.parametrize("partition", [-1, 64, 0])
def test_head_dim_64_multi_query_matches_oracle(shape, partition):
    BS, Hq, Hkv, lens, q_len = shape
    inp, q = make_multi(lens, q_len, Hq, Hkv, BS, seed=BS + Hq + q_len + 64, D=64)
    ew = errword()
    out = run_multi(inp, q, partition, error_word=ew)
    assert ops.pkd_read_device_error(ew) == 0
    assert_close(out, oracle_multi(inp, q), f"D64 {shape} P={partition}")


def test_single_token_is_exactly_v0():
    inp = workloads.make_custom(6, 14, 2, 128, 16, [1] * 6, seed=3, device="cuda")
    out = run_ex(inp, TC, -1).cpu()
    for b in range(6):
        p = int(inp.block_tables[b, 0])
        for h in range(14):
            assert torch.equal(out[b, h], inp.v_cache[p, h // 7, 0].cpu())


def test_spike_selects_each_position():
    L, BS = 37, 16
    inp = workloads.make_custom(L, 2, 1, 128, BS, [L] * L, seed=5, device="cuda")
    inp.q.fill_(1.0)
    for b in range(L):
        inp.k_cache[int(inp.block_tables[b, b // BS]), 0, b % BS, :] = 1000.0
    out = run_ex(inp, TC, -1).cpu()
    for b in range(L):
        vb = inp.v_cache[int(inp.block_tables[b, b // BS]), 0, b % BS].cpu()
        assert torch.equal(out[b, 0], vb) and torch.equal(out[b, 1], vb), b


@pytest.mark.parametrize("partition", [-1, 64])
def test_block_permutation_bitwise(partition):
    lens = [200, 77, 129]
    a = workloads.make_custom(3, 8, 2, 128, 16, lens, seed=11, device="cuda")
    nb = a.num_blocks
    perm = torch.randperm(nb, generator=torch.Generator().manual_seed(99)).to(torch.int32)
    b_k = torch.empty_like(a.k_cache)
    b_v = torch.empty_like(a.v_cache)
    b_k[perm.long().cuda()] = a.k_cache
    b_v[perm.long().cuda()] = a.v_cache
    bt = a.block_tables.clone()
    used = bt >= 0
    bt[used] = perm.cuda()[bt[used].long()]
    b = workloads.DecodeInputs(**{**a.__dict__, "k_cache": b_k, "v_cache": b_v, "block_tables": bt})
    assert torch.equal(run_ex(a, TC, partition), run_ex(b, TC, partition))


def test_nan_poison_in_unused_slots():
    lens = [21, 9, 70, 130]
    clean = workloads.make_custom(4, 8, 2, 128, 16, lens, seed=13, device="cuda")
    pois = workloads.DecodeInputs(**{**clean.__dict__, "k_cache": clean.k_cache.clone(),
                                     "v_cache": clean.v_cache.clone()})
    used = torch.zeros(clean.num_blocks, 16, dtype=torch.bool)
    for b, L in enumerate(lens):
        for t in range(L):
            used[int(clean.block_tables[b, t // 16]), t % 16] = True
    mask = (~used).cuda()
    pois.k_cache.permute(0, 2, 1, 3)[mask] = float("nan")
    pois.v_cache.permute(0, 2, 1, 3)[mask] = float("nan")
    for partition in (-1, 96):
        a = run_ex(clean, TC, partition)
        b = run_ex(pois, TC, partition)
        assert torch.isfinite(b).all()
        assert torch.equal(a, b)


def test_context_zero_gives_zeros():
    inp = workloads.make_custom(3, 8, 2, 128, 16, [0, 20, 0], seed=17, device="cuda", max_blocks_per_seq=2)
    out = torch.full_like(inp.q, float("nan"))
    run_ex(inp, TC, -1, out=out)
    assert torch.all(out[0] == 0) and torch.all(out[2] == 0)
    assert_close(out, oracle_out(inp))


@pytest.mark.parametrize("partition", [-1, 64])
def test_l2_eviction_hints_change_nothing(partition):
    inp = workloads.make_custom(4, 28, 4, 128, 16, [300, 17, 129, 64], seed=37, device="cuda")
    a = run_ex(inp, TC, partition)
    b = run_ex(inp, TC + "+l2_hints", partition)
    assert torch.equal(a, b)
    assert_close(b, oracle_out(inp), "with L2 hints")


# --------------------------------------------------------------------------- split-K partials
def test_partition_token_counts_exact_at_scale_zero():
    lens = [100, 32, 1, 64, 0, 257]
    P = 32
    inp = workloads.make_custom(len(lens), 10, 2, 128, 16, lens, seed=19, device="cuda")
    NP = -(-max(lens) // P)
    tmp = torch.zeros(len(lens), 10, NP, 128, dtype=torch.float32, device="cuda")
    ml = torch.full((len(lens), 10, NP), 123.0, dtype=torch.float32, device="cuda")
    es = torch.full((len(lens), 10, NP), -1.0, dtype=torch.float32, device="cuda")
    ops.paged_decode_partitions(inp.q, inp.k_cache, inp.v_cache, inp.block_tables, inp.context_lens,
                                0.0, P, tmp, ml, es, max_context_len=max(lens), variant=TC)
    es, ml = es.cpu(), ml.cpu()
    for b, L in enumerate(lens):
        for j in range(NP):
            n = min(P, L - j * P)
            if n > 0:
                assert torch.all(es[b, :, j] == float(n)), (b, j, es[b, :, j])
                assert torch.all(ml[b, :, j] == 0.0)
            else:
                assert torch.all(es[b, :, j] == -1.0) and torch.all(ml[b, :, j] == 123.0)


def test_partitions_match_oracle():
    lens = [300, 64, 129]
    P = 64
    inp = workloads.make_custom(3, 14, 2, 128, 16, lens, seed=23, device="cuda")
    NP = -(-max(lens) // P)
    tmp = torch.zeros(3, 14, NP, 128, dtype=torch.float32, device="cuda")
    ml = torch.zeros(3, 14, NP, dtype=torch.float32, device="cuda")
    es = torch.zeros(3, 14, NP, dtype=torch.float32, device="cuda")
    ops.paged_decode_partitions(inp.q, inp.k_cache, inp.v_cache, inp.block_tables, inp.context_lens,
                                inp.scale, P, tmp, ml, es, max_context_len=max(lens), variant=TC)
    m, l, o = oracle.partitions(inp.q.cpu(), inp.k_cache.cpu(), inp.v_cache.cpu(), inp.block_tables.cpu(),
                                inp.context_lens.cpu(), inp.scale, P, max_partitions=NP)
    for b, L in enumerate(lens):
        npb = -(-L // P)
        g_m = ml.cpu().double().numpy()[b, :, :npb]
        g_l = es.cpu().double().numpy()[b, :, :npb]
        g_o = tmp.cpu().double().numpy()[b, :, :npb]
        # the maximum is exact (the lazy shift is folded out of the partial)
        assert np.max(np.abs(g_m - m[b, :, :npb])) <= 1e-4
        assert np.max(np.abs(g_l - l[b, :, :npb]) / l[b, :, :npb]) <= 1e-4
        assert np.max(np.abs(g_o - o[b, :, :npb])) <= 1e-3 * np.max(l[b, :, :npb])


# --------------------------------------------------------------------------- device errors
@pytest.mark.parametrize("partition", [-1, 64])
def test_bad_block_id_sets_error_word_and_is_skipped(partition):
    lens = [140, 20, 70]
    inp = workloads.make_custom(3, 8, 2, 128, 16, lens, seed=29, device="cuda")
    ref = oracle_out(inp)
    inp.block_tables[0, 1] = inp.num_blocks + 1000  # outside the pool: checked, never dereferenced
    ew = errword()
    out = run_ex(inp, TC, partition, error_word=ew)
    assert ops.pkd_read_device_error(ew) & ops.DEVERR_BAD_BLOCK
    assert torch.isfinite(out).all()
    assert_close(out[1:], ref[1:], "other sequences")


@pytest.mark.parametrize("partition", [-1, 64])
def test_length_past_the_table_row_is_reported_and_contained(partition):
    lens = [100, 60, 37]
    inp = workloads.make_custom(len(lens), 8, 2, 128, 16, lens, seed=41, device="cuda", max_blocks_per_seq=7)
    ref = oracle_out(inp)
    bad = inp.context_lens.clone()
    bad[1] = 10_000
    ew = errword()
    out = ops.paged_decode_attention_ex(inp.q, inp.k_cache, inp.v_cache, inp.block_tables, bad, inp.scale,
                                        max_context_len=112, partition_size=partition, variant=TC,
                                        error_word=ew)
    assert ops.pkd_read_device_error(ew) & ops.DEVERR_BAD_BLOCK
    assert_close(out[[0, 2]], ref[[0, 2]], "sequences with valid lengths")


# --------------------------------------------------------------------------- multi-token queries
MULTI = [
    # (BS, Hq, Hkv, lens, q_len)
    (16, 28, 4, [0, 5, 257, 700], 8),      # G=7: 56 rows, one chunk
    (16, 28, 4, [90, 31, 200], 9),         # G=7: 63 rows
    (16, 28, 4, [130, 64], 10),            # G=7: chunks of 9 + 1
    (32, 16, 2, [2, 100, 65], 8),          # G=8: exactly 64 rows; L < q_len
    (32, 16, 2, [300, 9], 9),              # G=8: chunks of 8 + 1
    (16, 32, 8, [64, 129, 513], 16),       # G=4: 64 rows
    (16, 32, 8, [300, 33], 17),            # G=4: chunks of 16 + 1
    (16, 40, 8, [200, 64, 1], 12),         # G=5: 60 rows
    (16, 4, 4, [50, 17, 200], 64),         # G=1: 64 query tokens
    (16, 4, 4, [40, 300], 65),             # G=1: chunks of 64 + 1
    (16, 6, 2, [150, 16], 22),             # G=3: chunks of 21 + 1
    (32, 12, 2, [77, 1, 129], 11),         # G=6: chunks of 10 + 1
    (16, 28, 4, [300, 3], 2),              # G=7: 14 rows (also the mma.sync path's size)
]


@pytest.mark.parametrize("shape", MULTI, ids=lambda s: f"BS{s[0]}G{s[1] // s[2]}Q{s[4]}")
@pytest.mark.parametrize("partition", [-1, 64, 0])
def test_multi_query_matches_oracle(shape, partition):
    BS, Hq, Hkv, lens, q_len = shape
    inp, q = make_multi(lens, q_len, Hq, Hkv, BS, seed=BS + Hq + q_len)
    ew = errword()
    out = run_multi(inp, q, partition, error_word=ew)
    assert ops.pkd_read_device_error(ew) == 0
    assert_close(out, oracle_multi(inp, q), f"{shape} P={partition}")


def test_multi_query_both_tensor_core_paths_agree():
    inp, q = make_multi([700, 129, 33, 1000], 8, 28, 4, 16, seed=61)
    a = run_multi(inp, q, 0, variant=TC)
    b = run_multi(inp, q, 0, variant="tma_mma")
    ref = oracle_multi(inp, q)
    assert_close(a, ref, "tcgen05")
    assert_close(b, ref, "tma_mma")
    assert float((a.float() - b.float()).abs().max()) <= 4e-3


def test_multi_query_nan_poison_in_unused_slots():
    lens = [21, 9, 70]
    inp, q = make_multi(lens, 8, 28, 4, 16, seed=13)
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


def test_multi_query_longest_first_is_bitwise_neutral():
    B, Hq, Hkv, q_len = 96, 28, 4, 8
    lens = torch.randint(1024, 4097, (B,), generator=torch.Generator().manual_seed(29)).tolist()
    inp, q = make_multi(lens, q_len, Hq, Hkv, 16, seed=29)
    a = run_multi(inp, q, -1, variant=TC)
    b = run_multi(inp, q, -1, variant=TC + "+longest_first")
    assert torch.equal(a, b)
    rows = sample_rows(B * q_len, Hq, 96, seed=29)
    got = b.view(-1, 128)[torch.from_numpy(rows).long().cuda()]
    assert_close(got, oracle_multi(inp, q, rows=rows), "tcgen05 longest first")


@pytest.mark.parametrize("name,q_len,min_partition", [("qwen25_7b_gqa7", 8, None), ("llama3_8b_gqa4", 8, None),
                                                     ("qwen25_14b_gqa5_splitk", 8, 2049)])
def test_multi_query_full_size_all_rows(name, q_len, min_partition):
    # the full workloads verifying q_len draft tokens per sequence, at the automatic split; the
    # GQA 5:1 long-context batch has too few (sequence, kv head) units for two waves, so the
    # tcgen05 plan splits it into partitions longer than the mma.sync path's 2048 tokens
    cfg = workloads.CONFIGS[name]
    inp = workloads.make_inputs(cfg, device="cuda")
    # the host bound of the context lengths sizes the split: the configured one (32768 tokens
    # for the GQA 5:1 batch, whose longest drawn context is a little shorter)
    inp.max_context_len = cfg.max_context_len
    _, part, _, path, _, _ = ops.paged_decode_call_plan(cfg.num_seqs, q_len, cfg.num_q_heads, cfg.num_kv_heads,
                                                    cfg.head_dim, cfg.block_size, inp.max_context_len)
    assert path.split("+")[0] == TC
    if min_partition is not None:
        assert part >= min_partition, part
    g = torch.Generator(device="cuda").manual_seed(78)
    q = workloads.randn_f16((cfg.num_seqs, q_len, cfg.num_q_heads, cfg.head_dim), g, "cuda")
    ew = errword()
    out = run_multi(inp, q, 0, variant="auto", error_word=ew)
    assert ops.pkd_read_device_error(ew) == 0
    assert_close(out, oracle_multi(inp, q), f"{name} q_len={q_len}")


@pytest.mark.parametrize("q_len", [1, 8])
def test_long_partitions_on_tcgen05(q_len):
    # partitions of 4096 tokens, as the automatic tcgen05 split picks for long contexts:
    # lengths just under, at and past one and two partitions, and a ragged last tile
    lens = [4095, 4096, 4097, 8192 + 33, 9000, 70]
    inp, q = make_multi(lens, q_len, 28, 4, 16, seed=97)
    ew = errword()
    out = run_multi(inp, q, 4096, variant=TC, error_word=ew)
    assert ops.pkd_read_device_error(ew) == 0
    assert_close(out, oracle_multi(inp, q), f"tcgen05 P=4096 q_len={q_len}")


# --------------------------------------------------------------------------- E4M3 caches
# caches drawn over every finite E4M3 code, with the scales that go with that draw
K_SCALE, V_SCALE = workloads.E4M3_SCALES["full"]


def make_fp8(lens, q_len, Hq, Hkv, BS, seed):
    inp, q = make_multi(lens, q_len, Hq, Hkv, BS, seed)
    g = torch.Generator(device="cuda").manual_seed(seed + 3)
    k8 = workloads.rand_e4m3(inp.k_cache.shape, g, "cuda")
    v8 = workloads.rand_e4m3(inp.v_cache.shape, g, "cuda")
    return inp, q, k8, v8


def run_fp8(inp, q, k8, v8, partition, **kw):
    return ops.paged_decode_attention_fp8(q, k8, v8, inp.block_tables, inp.context_lens, inp.scale, K_SCALE,
                                          V_SCALE, max_context_len=inp.max_context_len, partition_size=partition,
                                          **kw)


def oracle_fp8(inp, q, k8, v8, rows=None):
    return oracle.attention_fp8(q.cpu(), k8.cpu(), v8.cpu(), inp.block_tables.cpu(), inp.context_lens.cpu(),
                                inp.scale, K_SCALE, V_SCALE, rows=rows)


def check_fp8(got, inp, q, k8, v8, what, rows=None):
    """The absolute tolerance and the element bound of the tensor-core arithmetic."""
    absref = oracle_fp8(inp, q, k8, e4m3_magnitudes(v8), rows=rows)
    return assert_close_weighted(got, oracle_fp8(inp, q, k8, v8, rows=rows), absref, 448.0 * V_SCALE,
                                 int(inp.max_context_len), what)


FP8_MULTI = [
    # (BS, Hq, Hkv, lens, q_len): three or more 16-row tiles, so the automatic path is tcgen05
    (16, 28, 4, [0, 5, 257, 700], 8),      # G=7: 56 rows
    (16, 28, 4, [130, 64], 10),            # G=7: chunks of 9 + 1
    (32, 16, 2, [2, 100, 65], 8),          # G=8: 64 rows, L < q_len, BS=32
    (16, 32, 8, [300, 33], 17),            # G=4: chunks of 16 + 1
    (16, 4, 4, [40, 300], 65),             # G=1: chunks of 64 + 1
    (16, 40, 8, [200, 64, 1], 9),          # G=5: 45 rows (three mma.sync tiles)
]


@pytest.mark.parametrize("shape", FP8_MULTI, ids=lambda s: f"BS{s[0]}G{s[1] // s[2]}Q{s[4]}")
@pytest.mark.parametrize("partition", [-1, 64, 0])
def test_fp8_multi_query_on_tcgen05_matches_oracle(shape, partition):
    BS, Hq, Hkv, lens, q_len = shape
    assert ops.paged_decode_call_plan(len(lens), q_len, Hq, Hkv, 128, BS, max(lens), kv_fp8=True)[3] == TC
    inp, q, k8, v8 = make_fp8(lens, q_len, Hq, Hkv, BS, seed=BS + Hq + q_len + 1)
    ew = errword()
    out = run_fp8(inp, q, k8, v8, partition, error_word=ew)
    assert ops.pkd_read_device_error(ew) == 0
    check_fp8(out, inp, q, k8, v8, f"E4M3 {shape} P={partition}")


def test_fp8_multi_query_nan_codes_in_unused_slots():
    lens = [21, 9, 70]
    inp, q, k8, v8 = make_fp8(lens, 8, 28, 4, 16, seed=17)
    used = torch.zeros(inp.num_blocks, 16, dtype=torch.bool)
    for b, L in enumerate(lens):
        for t in range(L):
            used[int(inp.block_tables[b, t // 16]), t % 16] = True
    a = run_fp8(inp, q, k8, v8, -1)
    mask = (~used).cuda()
    k8.permute(0, 2, 1, 3)[mask] = 0x7F  # the NaN code
    v8.permute(0, 2, 1, 3)[mask] = 0xFF
    b = run_fp8(inp, q, k8, v8, -1)
    assert torch.isfinite(b).all()
    assert torch.equal(a, b)


def test_fp8_multi_query_full_size_all_rows():
    # Qwen2.5-7B shape over E4M3 caches verifying 8 draft tokens, at the automatic split
    cfg = workloads.CONFIGS["qwen25_7b_gqa7"]
    inp = workloads.make_inputs(cfg, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(81)
    k8 = workloads.rand_e4m3(inp.k_cache.shape, g, "cuda")
    v8 = workloads.rand_e4m3(inp.v_cache.shape, g, "cuda")
    del inp.k_cache, inp.v_cache
    q = workloads.randn_f16((cfg.num_seqs, 8, cfg.num_q_heads, cfg.head_dim), g, "cuda")
    ew = errword()
    out = ops.paged_decode_attention_fp8(q, k8, v8, inp.block_tables, inp.context_lens, inp.scale, K_SCALE, V_SCALE,
                                         max_context_len=inp.max_context_len, error_word=ew)
    assert ops.pkd_read_device_error(ew) == 0
    check_fp8(out, inp, q, k8, v8, "qwen25_7b_gqa7 E4M3 q_len=8")


@pytest.mark.parametrize("q_len", [4, 8])
@pytest.mark.parametrize("variant", ["tma_mma", "tcgen05"])
def test_fp8_ex_runs_the_requested_path(q_len, variant):
    # paged_decode_attention_fp8_ex: either tensor-core path on request, whichever the
    # automatic choice would take (GQA 7:1: q_len 4 is two 16-row mma.sync tiles, q_len 8
    # four; both run tcgen05 by default)
    lens = [300, 33, 130, 1]
    inp, q, k8, v8 = make_fp8(lens, q_len, 28, 4, 16, seed=101 + q_len)
    plan = ops.paged_decode_call_plan(len(lens), q_len, 28, 4, 128, 16, max(lens), kv_fp8=True, variant=variant)
    assert plan[3].split("+")[0] == variant
    ew = errword()
    out = ops.paged_decode_attention_fp8(q, k8, v8, inp.block_tables, inp.context_lens, inp.scale, K_SCALE, V_SCALE,
                                         max_context_len=inp.max_context_len, variant=variant, error_word=ew)
    assert ops.pkd_read_device_error(ew) == 0
    check_fp8(out, inp, q, k8, v8, f"E4M3 {variant} q_len={q_len}")


def test_fp8_ex_refuses_cuda_core_paths():
    inp, q, k8, v8 = make_fp8([64, 20], 4, 28, 4, 16, seed=7)
    with pytest.raises(ops.PagedDecodeError) as e:
        ops.paged_decode_attention_fp8(q, k8, v8, inp.block_tables, inp.context_lens, inp.scale, K_SCALE, V_SCALE,
                                       max_context_len=inp.max_context_len, variant="tma_staged")
    assert e.value.status == 3  # PKD_ERR_UNSUPPORTED
