"""GPU parity: the CUDA path through the C ABI against the fp64 CPU oracle.

Every test here runs the library's kernels on cuda:0 on seeded inputs and
compares element by element with ``oracle`` (max |err| <= 4e-3 and mean
|err| <= 5e-4 on the fp16 output), or checks exact properties (block
permutation, single token, one-token spike, partition token counts).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from helpers import MAX_ABS_TOL, assert_close, oracle_out
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


def run_ex(inp, variant="auto", partition_size=0, **kw):
    return ops.paged_decode_attention_ex(inp.q, inp.k_cache, inp.v_cache, inp.block_tables,
                                         inp.context_lens, inp.scale,
                                         max_context_len=inp.max_context_len,
                                         partition_size=partition_size, variant=variant, **kw)


def errword(device="cuda"):
    return torch.zeros(1, dtype=torch.int32, device=device)


# --------------------------------------------------------------------------- tiny config
@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("partition", [-1, 32, 64])
def test_tiny_config(variant, partition):
    inp = workloads.make_inputs(workloads.CONFIGS["tiny"], device="cuda")
    ref = oracle_out(inp)
    ew = errword()
    out = run_ex(inp, variant, partition, error_word=ew)
    assert ops.pkd_read_device_error(ew) == 0
    assert_close(out, ref, f"tiny {variant} P={partition}")


def test_basic_entry_point_tiny():
    inp = workloads.make_inputs(workloads.CONFIGS["tiny"], device="cuda")
    out = ops.paged_decode_attention(inp.q, inp.k_cache, inp.v_cache, inp.block_tables,
                                     inp.context_lens, inp.scale, max_context_len=inp.max_context_len)
    assert_close(out, oracle_out(inp), "basic")


# --------------------------------------------------------------------------- shape matrix
SHAPES = [
    # (D, BS, Hq, Hkv, lens)
    (128, 16, 4, 4, [1, 15, 16, 17, 100, 333]),
    (128, 16, 28, 4, [0, 5, 31, 32, 33, 257, 700]),
    (128, 16, 32, 8, [64, 1, 129, 513]),
    (128, 16, 40, 8, [300, 47]),
    (128, 32, 16, 2, [1, 31, 32, 33, 250]),
    (128, 16, 16, 2, [77, 200]),   # G=8
    (128, 16, 6, 2, [90, 3]),      # G=3
    (128, 16, 12, 2, [150]),       # G=6
    (128, 16, 4, 2, [45, 99]),     # G=2
    (64, 16, 4, 4, [37, 100]),
    (64, 32, 14, 2, [1, 63, 64, 65, 190]),
    (64, 16, 5, 1, [40, 128]),
]


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"D{s[0]}BS{s[1]}G{s[2]//s[3]}")
@pytest.mark.parametrize("partition", [-1, 64])
def test_shape_matrix(variant, shape, partition):
    D, BS, Hq, Hkv, lens = shape
    inp = workloads.make_custom(len(lens), Hq, Hkv, D, BS, lens, seed=D + BS + Hq,
                                device="cuda", max_blocks_per_seq=-(-max(lens) // BS) + 2)
    ref = oracle_out(inp)
    ew = errword()
    out = run_ex(inp, variant, partition, error_word=ew)
    assert ops.pkd_read_device_error(ew) == 0
    assert_close(out, ref, f"{shape} {variant} P={partition}")


# --------------------------------------------------------------------------- exact properties
@pytest.mark.parametrize("variant", VARIANTS)
def test_single_token_is_exactly_v0(variant):
    lens = [1] * 6
    inp = workloads.make_custom(6, 14, 2, 128, 16, lens, seed=3, device="cuda")
    out = run_ex(inp, variant, -1).cpu()
    G = 7
    for b in range(6):
        p = int(inp.block_tables[b, 0])
        for h in range(14):
            v0 = inp.v_cache[p, h // G, 0].cpu()
            assert torch.equal(out[b, h], v0)


@pytest.mark.parametrize("variant", VARIANTS)
def test_spike_selects_each_position(variant):
    # sequence b has a key spike at logical position b: out must be exactly v_b
    L, BS, D = 37, 16, 128
    inp = workloads.make_custom(L, 2, 1, D, BS, [L] * L, seed=5, device="cuda")
    inp.q.fill_(1.0)
    for b in range(L):
        p = int(inp.block_tables[b, b // BS])
        inp.k_cache[p, 0, b % BS, :] = 1000.0
    out = run_ex(inp, variant, -1).cpu()
    for b in range(L):
        p = int(inp.block_tables[b, b // BS])
        vb = inp.v_cache[p, 0, b % BS].cpu()
        assert torch.equal(out[b, 0], vb), b
        assert torch.equal(out[b, 1], vb), b


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("partition", [-1, 64])
def test_block_permutation_bitwise(variant, partition):
    lens = [200, 77, 129]
    a = workloads.make_custom(3, 8, 2, 128, 16, lens, seed=11, device="cuda")
    # same logical K/V placed in a different set of physical blocks
    nb = a.num_blocks
    perm = torch.randperm(nb, generator=torch.Generator().manual_seed(99)).to(torch.int32)
    inv = torch.empty_like(perm)
    inv[perm.long()] = torch.arange(nb, dtype=torch.int32)
    b_k = torch.empty_like(a.k_cache)
    b_v = torch.empty_like(a.v_cache)
    b_k[perm.long().cuda()] = a.k_cache
    b_v[perm.long().cuda()] = a.v_cache
    bt = a.block_tables.clone()
    used = bt >= 0
    bt[used] = perm.cuda()[bt[used].long()]
    b = workloads.DecodeInputs(**{**a.__dict__, "k_cache": b_k, "v_cache": b_v, "block_tables": bt})
    oa = run_ex(a, variant, partition)
    ob = run_ex(b, variant, partition)
    assert torch.equal(oa, ob)


@pytest.mark.parametrize("variant", VARIANTS)
def test_nan_poison_in_unused_slots(variant):
    lens = [21, 9, 70]
    clean = workloads.make_custom(3, 8, 2, 128, 16, lens, seed=13, device="cuda")
    pois = workloads.DecodeInputs(**{**clean.__dict__, "k_cache": clean.k_cache.clone(),
                                     "v_cache": clean.v_cache.clone()})
    used = torch.zeros(clean.num_blocks, 16, dtype=torch.bool)
    for b, L in enumerate(lens):
        for t in range(L):
            used[int(clean.block_tables[b, t // 16]), t % 16] = True
    mask = (~used).cuda()
    pois.k_cache.permute(0, 2, 1, 3)[mask] = float("nan")
    pois.v_cache.permute(0, 2, 1, 3)[mask] = float("nan")
    a = run_ex(clean, variant, -1)
    b = run_ex(pois, variant, -1)
    assert torch.isfinite(b).all()
    assert torch.equal(a, b)


@pytest.mark.parametrize("variant", VARIANTS)
def test_context_zero_and_empty_batch(variant):
    inp = workloads.make_custom(3, 4, 4, 64, 16, [0, 20, 0], seed=17, device="cuda",
                                max_blocks_per_seq=2)
    out = torch.full_like(inp.q, float("nan"))
    run_ex(inp, variant, -1, out=out)
    assert torch.all(out[0] == 0) and torch.all(out[2] == 0)
    assert_close(out, oracle_out(inp))
    empty = torch.empty(0, 4, 64, dtype=torch.float16, device="cuda")
    ops.paged_decode_attention_ex(empty, inp.k_cache, inp.v_cache, inp.block_tables[:0],
                                  inp.context_lens[:0], inp.scale, max_context_len=0, variant=variant)


# --------------------------------------------------------------------------- split-K pieces
@pytest.mark.parametrize("variant", VARIANTS)
def test_partition_token_counts_exact_at_scale_zero(variant):
    lens = [100, 32, 1, 64, 0, 257]
    P = 32
    inp = workloads.make_custom(len(lens), 10, 2, 128, 16, lens, seed=19, device="cuda")
    NP = -(-max(lens) // P)
    tmp = torch.zeros(len(lens), 10, NP, 128, dtype=torch.float32, device="cuda")
    ml = torch.full((len(lens), 10, NP), 123.0, dtype=torch.float32, device="cuda")
    es = torch.full((len(lens), 10, NP), -1.0, dtype=torch.float32, device="cuda")
    ops.paged_decode_partitions(inp.q, inp.k_cache, inp.v_cache, inp.block_tables, inp.context_lens,
                                0.0, P, tmp, ml, es, max_context_len=max(lens), variant=variant)
    es = es.cpu()
    ml = ml.cpu()
    for b, L in enumerate(lens):
        for j in range(NP):
            n = min(P, L - j * P)
            if n > 0:
                assert torch.all(es[b, :, j] == float(n)), (b, j, es[b, :, j])
                assert torch.all(ml[b, :, j] == 0.0)
            else:  # partitions past the context are not written
                assert torch.all(es[b, :, j] == -1.0) and torch.all(ml[b, :, j] == 123.0)


@pytest.mark.parametrize("variant", VARIANTS)
def test_partitions_match_oracle(variant):
    lens = [300, 64, 129]
    P = 64
    inp = workloads.make_custom(3, 14, 2, 128, 16, lens, seed=23, device="cuda")
    NP = -(-max(lens) // P)
    tmp = torch.zeros(3, 14, NP, 128, dtype=torch.float32, device="cuda")
    ml = torch.zeros(3, 14, NP, dtype=torch.float32, device="cuda")
    es = torch.zeros(3, 14, NP, dtype=torch.float32, device="cuda")
    ops.paged_decode_partitions(inp.q, inp.k_cache, inp.v_cache, inp.block_tables, inp.context_lens,
                                inp.scale, P, tmp, ml, es, max_context_len=max(lens), variant=variant)
    m, l, o = oracle.partitions(inp.q.cpu(), inp.k_cache.cpu(), inp.v_cache.cpu(),
                                inp.block_tables.cpu(), inp.context_lens.cpu(), inp.scale, P,
                                max_partitions=NP)
    for b, L in enumerate(lens):
        npb = -(-L // P)
        g_m = ml.cpu().double().numpy()[b, :, :npb]
        g_l = es.cpu().double().numpy()[b, :, :npb]
        g_o = tmp.cpu().double().numpy()[b, :, :npb]
        assert np.max(np.abs(g_m - m[b, :, :npb])) <= 1e-4
        assert np.max(np.abs(g_l - l[b, :, :npb]) / l[b, :, :npb]) <= 1e-4
        assert np.max(np.abs(g_o - o[b, :, :npb])) <= 1e-3 * np.max(l[b, :, :npb])
    # the merge kernel on the oracle's own partials equals the unsplit oracle
    out = torch.empty(3, 14, 128, dtype=torch.float16, device="cuda")
    ops.paged_decode_reduce(torch.from_numpy(o).float().cuda(), torch.from_numpy(m).float().cuda(),
                            torch.from_numpy(l).float().cuda(), inp.context_lens, out, P)
    assert_close(out, oracle_out(inp), "reduce of oracle partials")


def test_reduce_merges_every_sequence_when_min_is_zero():
    # empty and single-partition sequences included: merged from partials alone
    lens = [0, 40, 300, 0, 1]
    P = 64
    inp = workloads.make_custom(len(lens), 8, 2, 128, 16, lens, seed=31, device="cuda")
    NP = -(-max(lens) // P)
    tmp = torch.zeros(len(lens), 8, NP, 128, dtype=torch.float32, device="cuda")
    ml = torch.zeros(len(lens), 8, NP, dtype=torch.float32, device="cuda")
    es = torch.zeros(len(lens), 8, NP, dtype=torch.float32, device="cuda")
    ops.paged_decode_partitions(inp.q, inp.k_cache, inp.v_cache, inp.block_tables, inp.context_lens,
                                inp.scale, P, tmp, ml, es, max_context_len=max(lens))
    out = torch.full_like(inp.q, float("nan"))
    ops.paged_decode_reduce(tmp, ml, es, inp.context_lens, out, P, min_partitions_to_merge=0)
    assert torch.all(out[0] == 0) and torch.all(out[3] == 0)
    assert_close(out, oracle_out(inp), "partitions + reduce(min=0)")
    # min = 1 leaves sequences with at most one partition untouched
    out1 = torch.full_like(inp.q, 7.0)
    ops.paged_decode_reduce(tmp, ml, es, inp.context_lens, out1, P, min_partitions_to_merge=1)
    for b in (0, 1, 3, 4):
        assert torch.all(out1[b] == 7.0)
    assert torch.equal(out1[2], out[2])


# --------------------------------------------------------------------------- device errors
@pytest.mark.parametrize("variant", VARIANTS)
def test_bad_block_id_sets_error_word(variant):
    inp = workloads.make_custom(2, 4, 4, 128, 16, [40, 20], seed=29, device="cuda")
    inp.block_tables[0, 1] = inp.num_blocks + 1000   # outside the pool: checked, never dereferenced
    ew = errword()
    run_ex(inp, variant, -1, error_word=ew)
    assert ops.pkd_read_device_error(ew) & ops.DEVERR_BAD_BLOCK
    ew2 = errword()
    ops.paged_decode_validate_tables(inp.block_tables, inp.context_lens, 16, inp.num_blocks, ew2)
    assert ops.pkd_read_device_error(ew2) & ops.DEVERR_BAD_BLOCK
    inp.block_tables[0, 1] = 0
    ew3 = errword()
    ops.paged_decode_validate_tables(inp.block_tables, inp.context_lens, 16, inp.num_blocks, ew3)
    assert ops.pkd_read_device_error(ew3) == 0


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("partition", [-1, 64])
def test_l2_eviction_hints_change_nothing(variant, partition):
    # the hints only set L2 eviction priorities: outputs are bitwise equal
    inp = workloads.make_custom(4, 28, 4, 128, 16, [300, 17, 129, 64], seed=37, device="cuda")
    a = run_ex(inp, variant, partition)
    b = run_ex(inp, variant + "+l2_hints", partition)
    assert torch.equal(a, b)
    assert_close(b, oracle_out(inp), "with L2 hints")


def test_bounded_wait_times_out_and_reports():
    # a barrier nothing completes: the wait must give up and set the timeout bit
    ew = errword()
    ops.pkd_selftest_bounded_wait(ew, budget_ns=2_000_000)
    assert ops.pkd_read_device_error(ew) == ops.DEVERR_TIMEOUT
    # the context is still usable afterwards
    inp = workloads.make_inputs(workloads.CONFIGS["tiny"], device="cuda")
    assert_close(run_ex(inp, "tma_staged", -1), oracle_out(inp), "after self-test")


# --------------------------------------------------------------------------- full-size configs
FULL = ["llama2_7b_mha", "llama3_8b_gqa4", "qwen25_7b_gqa7", "qwen25_14b_gqa5_splitk"]


@pytest.mark.parametrize("name", FULL)
def test_full_config_all_rows(name):
    # every output row of the full workload, on every data path, against the oracle
    cfg = workloads.CONFIGS[name]
    inp = workloads.make_inputs(cfg, device="cuda")
    ref = oracle_out(inp)
    for variant in VARIANTS:
        ew = errword()
        out = run_ex(inp, variant, cfg.partition_size or 0, error_word=ew)
        assert ops.pkd_read_device_error(ew) == 0
        assert_close(out, ref, f"{name} {variant}")


# --------------------------------------------------------------------------- longest-first order
@pytest.mark.parametrize("partition", [-1, 64, 0])
@pytest.mark.parametrize("lens,Hq,Hkv", [([300, 17, 5000, 0, 129, 64, 2048, 1], 32, 8),
                                         ([700, 31, 2, 900, 90], 28, 4),
                                         ([1000] * 5 + [3], 8, 8)])
def test_longest_first_order_is_bitwise_neutral(lens, Hq, Hkv, partition):
    # the order only changes which CTA starts when: every CTA computes the same
    inp = workloads.make_custom(len(lens), Hq, Hkv, 128, 16, lens, seed=len(lens) + Hq, device="cuda")
    ew = errword()
    a = run_ex(inp, "tma_mma", partition)
    b = run_ex(inp, "tma_mma+longest_first", partition, error_word=ew)
    assert ops.pkd_read_device_error(ew) == 0
    assert torch.equal(a, b)
    assert_close(b, oracle_out(inp), f"longest first P={partition}")


def test_longest_first_full_size_ragged_all_rows():
    cfg = workloads.CONFIGS["llama3_8b_gqa4"]
    inp = workloads.make_inputs(cfg, device="cuda")
    a = run_ex(inp, "tma_mma", -1)
    b = run_ex(inp, "tma_mma+longest_first", -1)
    assert torch.equal(a, b)
    assert_close(b, oracle_out(inp), "llama3_8b_gqa4 longest first")


def test_longest_first_order_kernel_ranks_by_length():
    # the order the grid walks: decreasing length, ties by index
    lens = [5, 9, 9, 0, 12, 5, 1]
    inp = workloads.make_custom(len(lens), 4, 4, 64, 16, lens, seed=3, device="cuda")
    need = ops.paged_decode_workspace_size(len(lens), 4, 4, 64, 16, max(lens), -1, "tma_mma+longest_first")
    ws = ops.alloc_workspace(need, "cuda")
    ws.fill_(0xFF)
    run_ex(inp, "tma_mma+longest_first", -1, workspace=ws)
    torch.cuda.synchronize()
    order = ws[:4 * len(lens)].view(torch.int32).cpu().tolist()
    assert order == sorted(range(len(lens)), key=lambda b: (-lens[b], b))


def test_longest_first_piece_order_of_a_split_grid():
    # partition 64: full pieces by sequence, then last pieces by decreasing length, then empties
    lens = [130, 0, 64, 200, 7, 129]
    P, NP = 64, 4
    inp = workloads.make_custom(len(lens), 4, 4, 64, 16, lens, seed=5, device="cuda")
    need = ops.paged_decode_workspace_size(len(lens), 4, 4, 64, 16, max(lens), P, "tma_mma+longest_first")
    ws = ops.alloc_workspace(need, "cuda")
    ws.fill_(0xFF)
    out = run_ex(inp, "tma_mma+longest_first", P, workspace=ws)
    assert_close(out, oracle_out(inp), "piece order")
    torch.cuda.synchronize()
    # the order follows the split partials in the workspace
    rows = len(lens) * 4 * NP
    off = -(-rows * 64 * 4 // 256) * 256 + 2 * (-(-rows * 4 // 256) * 256)
    got = ws[off:off + 4 * len(lens) * NP].view(torch.int32).cpu().tolist()
    n = [min(-(-L // P), NP) for L in lens]
    last = [L - (k - 1) * P if k else 0 for L, k in zip(lens, n)]
    full = [b * NP + j for b in range(len(lens)) for j in range(n[b] - 1)]
    lasts = [b * NP + n[b] - 1 for b in sorted((b for b in range(len(lens)) if n[b]), key=lambda b: (-last[b], b))]
    empties = [b * NP + j for b in range(len(lens)) for j in range(n[b], NP)]
    assert got == full + lasts + empties


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("partition", [-1, 64])
def test_length_past_the_table_row_is_reported_and_contained(variant, partition):
    # sequence 1 claims more tokens than its block-table row holds: the kernels read only the
    # row, report PKD_DEVERR_BAD_BLOCK, and the other sequences are unaffected
    lens = [100, 60, 37]
    inp = workloads.make_custom(len(lens), 8, 2, 128, 16, lens, seed=41, device="cuda", max_blocks_per_seq=7)
    ref = oracle_out(inp)
    bad = inp.context_lens.clone()
    bad[1] = 10_000
    ew = errword()
    out = ops.paged_decode_attention_ex(inp.q, inp.k_cache, inp.v_cache, inp.block_tables, bad, inp.scale,
                                        max_context_len=112, partition_size=partition, variant=variant,
                                        error_word=ew)
    assert ops.pkd_read_device_error(ew) & ops.DEVERR_BAD_BLOCK
    assert_close(out[[0, 2]], ref[[0, 2]], "sequences with valid lengths")


# --------------------------------------------------------------------------- prefetch distance
def test_call_plan_reports_the_model_distance_for_this_device():
    # the plan's default distance is the capacity model on this GPU's own numbers
    props = torch.cuda.get_device_properties(0)
    for name in FULL:
        cfg = workloads.CONFIGS[name]
        for variant in ("l2_prefetch", "tma_staged", "tma_mma"):
            plan = ops.paged_decode_call_plan(cfg.num_seqs, 1, cfg.num_q_heads, cfg.num_kv_heads, cfg.head_dim,
                                              cfg.block_size, cfg.max_context_len,
                                              partition_size=cfg.partition_size or 0, variant=variant)
            # the device's nominal bandwidth is not exposed to Python: a distance that the model gives
            # for a range of bandwidths around GB300's must contain the one the library picked
            ds = {ops.paged_decode_prefetch_model(cfg.num_seqs, 1, cfg.num_q_heads, cfg.num_kv_heads, cfg.head_dim,
                                                  cfg.block_size, cfg.max_context_len, props.multi_processor_count,
                                                  props.L2_cache_size, bw, partition_size=cfg.partition_size or 0,
                                                  variant=variant)[0]
                  for bw in (7.0e12, 8.18e12, 9.0e12)}
            assert plan[5] in ds, (name, variant, plan, ds)


@pytest.mark.parametrize("variant", ["l2_prefetch", "tma_staged", "tma_mma"])
def test_prefetch_distances_change_no_bit(variant):
    # none (-1), the model's default (0) and explicit distances give the same result bitwise
    lens = [700, 33, 1500, 0, 129]
    inp = workloads.make_custom(len(lens), 28, 4, 128, 16, lens, seed=61, device="cuda")
    ref = run_ex(inp, variant, -1, prefetch_distance=-1)
    for pd in (0, 1, 3):
        assert torch.equal(run_ex(inp, variant, -1, prefetch_distance=pd), ref), pd
    assert_close(ref, oracle_out(inp), f"{variant} without L2 prefetch")
