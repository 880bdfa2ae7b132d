"""GPU parity of decode over FP8 (E4M3) KV caches and of the FP8 cache write.

paged_decode_attention_fp8 reads one byte per K/V element (value = code *
per-cache scale) and is compared with ``oracle.attention_fp8`` element by
element (max |err| <= 4e-3, mean <= 5e-4, and the per-element bound of
helpers.assert_close_weighted), single-query and multi-token;
paged_kv_append_fp8 is compared with ``oracle.append_fp8`` bit for bit.  The
caches are drawn over every finite E4M3 code (+-0, subnormals, exponents
1..15, +-448); test_gpu_fp8_codes.py adds caches of only extreme codes.
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import assert_close_weighted, e4m3_magnitudes, sample_rows
from paged_kv_decode_21_gb300 import ops, workloads

pytestmark = pytest.mark.gpu

K_SCALE, V_SCALE = workloads.E4M3_SCALES["full"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_decode_21_gb300 import build
    build.build()
    ops.lib()


def make(lens, Hq, Hkv, D, BS, seed, q_len=1, extra_blocks=1):
    inp = workloads.make_custom(len(lens), Hq, Hkv, D, BS, lens, seed=seed, device="cuda",
                                max_blocks_per_seq=-(-max(max(lens), 1) // BS) + extra_blocks)
    g = torch.Generator(device="cuda").manual_seed(seed + 3)
    k8 = workloads.rand_e4m3(inp.k_cache.shape, g, "cuda")
    v8 = workloads.rand_e4m3(inp.v_cache.shape, g, "cuda")
    q = inp.q if q_len == 1 else workloads.randn_f16((len(lens), q_len, Hq, D), g, "cuda")
    return inp, q, k8, v8


def run(inp, q, k8, v8, partition, ks=K_SCALE, vs=V_SCALE, **kw):
    return ops.paged_decode_attention_fp8(q, k8, v8, inp.block_tables, inp.context_lens, inp.scale,
                                          ks, vs, max_context_len=inp.max_context_len,
                                          partition_size=partition, **kw)


def check(got, inp, q, k8, v8, what, rows=None, context_lens=None):
    """got against the oracle: the absolute tolerance and the element bound."""
    cl = (inp.context_lens if context_lens is None else context_lens).cpu()
    args = (q.cpu(), k8.cpu())
    expect = oracle.attention_fp8(*args, v8.cpu(), inp.block_tables.cpu(), cl, inp.scale, K_SCALE, V_SCALE,
                                  rows=rows)
    absref = oracle.attention_fp8(*args, e4m3_magnitudes(v8).cpu(), inp.block_tables.cpu(), cl, inp.scale,
                                  K_SCALE, V_SCALE, rows=rows)
    vmax = 448.0 * V_SCALE
    return assert_close_weighted(got, expect, absref, vmax, int(cl.max()) if cl.numel() else 0, what)


SHAPES = [
    # (D, BS, Hq, Hkv, lens, q_len)
    (128, 16, 4, 4, [1, 15, 16, 17, 100, 333], 1),
    (128, 16, 28, 4, [0, 5, 31, 32, 33, 257, 700], 1),
    (128, 16, 32, 8, [64, 1, 129, 513], 1),
    (128, 32, 16, 2, [1, 31, 32, 33, 250], 1),
    (128, 16, 40, 8, [300, 47], 1),
    (64, 16, 4, 4, [37, 100], 1),
    (64, 32, 14, 2, [1, 63, 64, 65, 190], 1),
    (128, 16, 32, 8, [300, 33], 5),
    (128, 16, 28, 4, [90, 31, 2], 3),
    (64, 16, 4, 4, [40, 17], 17),
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"D{s[0]}BS{s[1]}G{s[2] // s[3]}Q{s[5]}")
@pytest.mark.parametrize("partition", [-1, 64, 0])
def test_fp8_matches_oracle(shape, partition):
    D, BS, Hq, Hkv, lens, q_len = shape
    inp, q, k8, v8 = make(lens, Hq, Hkv, D, BS, seed=D + BS + Hq + q_len, q_len=q_len)
    ew = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = run(inp, q, k8, v8, partition, error_word=ew)
    assert ops.pkd_read_device_error(ew) == 0
    check(out, inp, q, k8, v8, f"{shape} P={partition}")


def test_fp8_single_token_is_scaled_v0():
    # one token: out = v_0 * v_scale exactly (a power-of-two scale keeps the
    # product exact), then rounded once to fp16
    inp, q, k8, v8 = make([1] * 4, 14, 2, 128, 16, seed=3)
    out = run(inp, q, k8, v8, -1, ks=0.0625, vs=0.125).cpu().double()
    vals = torch.from_numpy(oracle.e4m3_to_double(np.arange(256, dtype=np.uint8)))
    for b in range(4):
        p = int(inp.block_tables[b, 0])
        for h in range(14):
            v0 = vals[v8[p, h // 7, 0].cpu().long()] * 0.125
            assert torch.equal(out[b, h], v0.to(torch.float16).double())


def test_fp8_nan_codes_in_unused_slots():
    lens = [21, 9, 70]
    inp, q, k8, v8 = make(lens, 8, 2, 128, 16, seed=13)
    used = torch.zeros(inp.num_blocks, 16, dtype=torch.bool)
    for b, L in enumerate(lens):
        for t in range(L):
            used[int(inp.block_tables[b, t // 16]), t % 16] = True
    a = run(inp, q, k8, v8, -1)
    mask = (~used).cuda()
    k8.permute(0, 2, 1, 3)[mask] = 0x7F  # the NaN code
    v8.permute(0, 2, 1, 3)[mask] = 0xFF
    b_ = run(inp, q, k8, v8, -1)
    assert torch.isfinite(b_).all()
    assert torch.equal(a, b_)


@pytest.mark.parametrize("D,BS,Hkv", [(128, 16, 4), (64, 32, 8), (16, 16, 3)])
def test_fp8_append_is_bit_exact(D, BS, Hkv):
    lens = [0, 1, BS - 1, BS, BS + 1, 2 * BS, 37, 700]
    inp, _, k8, v8 = make([L + 1 for L in lens], Hkv, Hkv, D, BS, seed=D + BS)
    cl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(11)
    # a wide range of values, with some beyond the saturation point after scaling
    k_new = (workloads.randn_f16((len(lens), Hkv, D), g, "cuda").float() * 8).half()
    v_new = (workloads.randn_f16((len(lens), Hkv, D), g, "cuda").float() * 8).half()
    ks, vs = 0.03, 0.125
    ref_k, ref_v = oracle.append_fp8(k_new.cpu(), v_new.cpu(), inp.block_tables.cpu(), cl.cpu(), k8.cpu(),
                                     v8.cpu(), ks, vs)
    ew = torch.zeros(1, dtype=torch.int32, device="cuda")
    ops.paged_kv_append_fp8(k_new, v_new, inp.block_tables, cl, k8, v8, ks, vs, error_word=ew)
    assert ops.pkd_read_device_error(ew) == 0
    assert np.array_equal(k8.cpu().numpy(), ref_k)
    assert np.array_equal(v8.cpu().numpy(), ref_v)


def test_fp8_append_then_decode():
    lens = [15, 16, 100, 511]
    inp, q, k8, v8 = make([L + 1 for L in lens], 28, 4, 128, 16, seed=21)
    cl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(22)
    k_new = workloads.randn_f16((4, 4, 128), g, "cuda")
    v_new = workloads.randn_f16((4, 4, 128), g, "cuda")
    ops.paged_kv_append_fp8(k_new, v_new, inp.block_tables, cl, k8, v8, K_SCALE, V_SCALE)
    grown = cl + 1
    out = ops.paged_decode_attention_fp8(q, k8, v8, inp.block_tables, grown, inp.scale, K_SCALE, V_SCALE,
                                         max_context_len=max(lens) + 1)
    check(out, inp, q, k8, v8, "fp8 append + decode", context_lens=grown)


def test_fp8_full_size_gqa_all_rows():
    # Qwen2.5-7B attention shape (256 sequences x 8192 tokens, 28 q / 4 kv heads) in E4M3
    cfg = workloads.CONFIGS["qwen25_7b_gqa7"]
    inp = workloads.make_inputs(cfg, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(31)
    k8 = workloads.rand_e4m3(inp.k_cache.shape, g, "cuda")
    v8 = workloads.rand_e4m3(inp.v_cache.shape, g, "cuda")
    del inp.k_cache, inp.v_cache
    torch.cuda.empty_cache()
    ew = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = run(inp, inp.q, k8, v8, 0, error_word=ew)
    assert ops.pkd_read_device_error(ew) == 0
    check(out, inp, inp.q, k8, v8, "qwen25_7b_gqa7 fp8")


@pytest.mark.parametrize("shape", [
    # (D, BS, Hq, Hkv, B, length range): single-query grids of >= 3 waves of four CTAs per
    # SM (>= 1824 CTAs on 152 SMs), which run the four-per-SM build
    (128, 16, 32, 32, 64, (200, 300)),
    (128, 16, 32, 8, 256, (100, 500)),
    (128, 16, 28, 4, 512, (1, 480)),
    (64, 32, 16, 16, 128, (150, 220)),
])
def test_fp8_wide_grid_four_per_sm_build(shape):
    D, BS, Hq, Hkv, B, (lo, hi) = shape
    lens = torch.randint(lo, hi + 1, (B,), generator=torch.Generator().manual_seed(B + Hq)).tolist()
    inp, q, k8, v8 = make(lens, Hq, Hkv, D, BS, seed=B + D)
    ew = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = run(inp, q, k8, v8, 0, error_word=ew)
    assert ops.pkd_read_device_error(ew) == 0
    rows = sample_rows(B, Hq, 256, seed=B)
    got = out.view(-1, D)[torch.from_numpy(rows).long().cuda()]
    check(got, inp, q, k8, v8, f"wide fp8 {shape}", rows=rows)


def test_fp8_automatic_order_is_bitwise_neutral():
    # 1024 (sequence, kv head) units of ragged length: the automatic split keeps the grid
    # unsplit and walks it longest first; the order only reschedules CTAs
    B, Hq, Hkv = 128, 32, 8
    lens = torch.randint(512, 4097, (B,), generator=torch.Generator().manual_seed(21)).tolist()
    inp, q, k8, v8 = make(lens, Hq, Hkv, 128, 16, seed=21)
    n, part, ordered = ops.paged_decode_auto_plan(B, 1, Hq, Hkv, 128, 16, inp.max_context_len, kv_fp8=True)
    assert ordered and part == -1 and n == 2
    a = run(inp, q, k8, v8, 0)
    b = run(inp, q, k8, v8, -1)
    assert torch.equal(a, b)
    rows = sample_rows(B, Hq, 128, seed=21)
    got = a.view(-1, 128)[torch.from_numpy(rows).long().cuda()]
    check(got, inp, q, k8, v8, "fp8 longest first", rows=rows)
