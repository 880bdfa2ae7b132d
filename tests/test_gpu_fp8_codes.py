"""GPU parity of decode over E4M3 caches made of extreme codes only.

The E4M3 reading of the CSDN answer "如何优化LLM推理引擎的内存访问延迟？"
(section 4, FP8 precision for the KV footprint) is OCP E4M3: +-0, subnormals
m * 2^-9, normal exponents 1..15, largest magnitude 448, no infinities.
Every data path that reads E4M3 caches (the mma.sync kernel at three and at
four CTAs per SM, single-query and multi-token, and the tcgen05 kernel that
widens tiles in shared memory) is run here on caches whose K and V codes
are all of one kind -- every finite code, only +-448, only +-0 and the
subnormals, and the two mixes of those -- plus keys so large that the
softmax is one-hot, and compared with ``oracle.attention_fp8`` under the
absolute tolerance and the element bound of helpers.assert_close_weighted.
"""
import pytest
import torch

import oracle
from helpers import assert_close_weighted, e4m3_magnitudes, sample_rows
from paged_kv_decode_21_gb300 import ops, workloads

pytestmark = pytest.mark.gpu

# largest |value| of each code set, before the scale
CODE_MAX = {"full": 448.0, "max": 448.0, "subnormal": 7 * 2.0 ** -9}

# (K codes, V codes, k_scale, v_scale); the scales are the ones that go with
# each code set, except the last case, whose unit K scale puts the scores of
# +-448 keys tens to hundreds apart (a nearly one-hot softmax)
CODE_CASES = [
    ("full", "full", *workloads.E4M3_SCALES["full"]),
    ("max", "max", *workloads.E4M3_SCALES["max"]),
    ("subnormal", "subnormal", *workloads.E4M3_SCALES["subnormal"]),
    ("max", "subnormal", workloads.E4M3_SCALES["max"][0], workloads.E4M3_SCALES["subnormal"][1]),
    ("subnormal", "max", workloads.E4M3_SCALES["subnormal"][0], workloads.E4M3_SCALES["max"][1]),
    ("max", "full", 1.0, workloads.E4M3_SCALES["full"][1]),
]
CODE_IDS = ["full", "max", "subnormal", "Kmax-Vsub", "Ksub-Vmax", "Kmax-unit-scale"]

# (D, BS, Hq, Hkv, lens, q_len, data path the automatic choice runs)
PATHS = [
    (128, 16, 28, 4, [1, 17, 700, 33], 1, "tma_mma"),
    (64, 32, 8, 8, [5, 100, 64], 1, "tma_mma"),
    (128, 16, 32, 8, [300, 33, 2], 2, "tma_mma"),
    (128, 16, 28, 4, [0, 5, 257, 700], 8, "tcgen05"),
    (128, 32, 8, 8, [100, 300], 40, "tcgen05"),
]
PATH_IDS = ["mma-G7", "mma-D64", "mma-q2", "tc-G7q8", "tc-G1q40"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_decode_21_gb300 import build
    build.build()
    ops.lib()


def make(lens, q_len, Hq, Hkv, D, BS, kcodes, vcodes, seed):
    inp = workloads.make_custom(len(lens), Hq, Hkv, D, BS, lens, seed=seed, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(seed + 5)
    k8 = workloads.rand_e4m3(inp.k_cache.shape, g, "cuda", codes=kcodes)
    v8 = workloads.rand_e4m3(inp.v_cache.shape, g, "cuda", codes=vcodes)
    q = inp.q if q_len == 1 else workloads.randn_f16((len(lens), q_len, Hq, D), g, "cuda")
    return inp, q, k8, v8


def check(got, inp, q, k8, v8, ks, vs, vcodes, what, rows=None):
    args = (q.cpu(), k8.cpu())
    tail = (inp.block_tables.cpu(), inp.context_lens.cpu(), inp.scale, ks, vs)
    expect = oracle.attention_fp8(*args, v8.cpu(), *tail, rows=rows)
    absref = oracle.attention_fp8(*args, e4m3_magnitudes(v8).cpu(), *tail, rows=rows)
    return assert_close_weighted(got, expect, absref, CODE_MAX[vcodes] * vs, int(inp.max_context_len), what)


@pytest.mark.parametrize("path", PATHS, ids=PATH_IDS)
@pytest.mark.parametrize("codes", CODE_CASES, ids=CODE_IDS)
@pytest.mark.parametrize("partition", [-1, 64])
def test_extreme_codes_match_oracle(path, codes, partition):
    D, BS, Hq, Hkv, lens, q_len, expect_path = path
    kcodes, vcodes, ks, vs = codes
    assert ops.paged_decode_call_plan(len(lens), q_len, Hq, Hkv, D, BS, max(lens), kv_fp8=True)[3] == expect_path
    inp, q, k8, v8 = make(lens, q_len, Hq, Hkv, D, BS, kcodes, vcodes, seed=D + Hq + q_len + BS)
    ew = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = ops.paged_decode_attention_fp8(q, k8, v8, inp.block_tables, inp.context_lens, inp.scale, ks, vs,
                                         max_context_len=inp.max_context_len, partition_size=partition,
                                         error_word=ew)
    assert ops.pkd_read_device_error(ew) == 0
    check(out, inp, q, k8, v8, ks, vs, vcodes, f"{path[:6]} K={kcodes} V={vcodes} P={partition}")


@pytest.mark.parametrize("codes", CODE_CASES[:3], ids=CODE_IDS[:3])
def test_extreme_codes_four_per_sm_build(codes):
    # 64 x 32 single-query units of ~256 tokens: three waves of four CTAs per SM on 152 SMs,
    # so the automatic choice runs the four-per-SM build with its single QK chain
    kcodes, vcodes, ks, vs = codes
    B, Hq, Hkv, D, BS = 64, 32, 32, 128, 16
    lens = torch.randint(200, 301, (B,), generator=torch.Generator().manual_seed(7)).tolist()
    inp, q, k8, v8 = make(lens, 1, Hq, Hkv, D, BS, kcodes, vcodes, seed=71)
    ew = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = ops.paged_decode_attention_fp8(q, k8, v8, inp.block_tables, inp.context_lens, inp.scale, ks, vs,
                                         max_context_len=inp.max_context_len, error_word=ew)
    assert ops.pkd_read_device_error(ew) == 0
    rows = sample_rows(B, Hq, 256, seed=71)
    got = out.view(-1, D)[torch.from_numpy(rows).long().cuda()]
    check(got, inp, q, k8, v8, ks, vs, vcodes, f"wide K={kcodes} V={vcodes}", rows=rows)


def test_one_hot_softmax_returns_the_winning_row():
    # +-448 keys at k_scale 4 put most rows' scores hundreds apart: every weight
    # but the winner's underflows to 0 in the fp32 kernel, so the output row is
    # that token's V row times v_scale (a power of two keeps it exact), rounded
    # once.  The oracle's fp64 weights (over K widened to fp16, exact for every
    # E4M3 value times 4) pick the rows where the runner-up's weight is below
    # 2^-40; every row also meets the element bound.
    ks, vs = 4.0, 0.125
    inp, q, k8, v8 = make([300, 45, 1], 1, 8, 2, 128, 16, "max", "full", seed=88)
    out = ops.paged_decode_attention_fp8(q, k8, v8, inp.block_tables, inp.context_lens, inp.scale, ks, vs,
                                         max_context_len=inp.max_context_len, partition_size=64)
    got = out.cpu().double()
    check(out, inp, q, k8, v8, ks, vs, "full", "one-hot")
    k16 = torch.from_numpy(oracle.e4m3_to_double(k8.cpu().numpy()).reshape(k8.shape) * ks).half()
    qc, bt, cl = q.cpu(), inp.block_tables.cpu(), inp.context_lens.cpu()
    ref = torch.from_numpy(oracle.attention_fp8(qc, k8.cpu(), v8.cpu(), bt, cl, inp.scale, ks, vs))
    one_hot = 0
    for b in range(3):
        for h in range(8):
            w = sorted(oracle.weights(qc, k16, k16, bt, cl, inp.scale, b, h))
            if len(w) == 1 or w[-2] < 2.0 ** -40:
                one_hot += 1
                assert torch.equal(got[b, h], ref[b, h].half().double()), (b, h)
    assert one_hot >= 12, one_hot
