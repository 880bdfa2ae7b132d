"""GPU parity over seeded random shapes: every data path, split and flag the ABI accepts.

Each case draws a shape (kv heads, group size, head_dim, block size, batch, lengths including
0 and 1, query tokens), a cache type (fp16, or E4M3 at head_dim 128), a data path the ABI
accepts for it, and a partition (automatic, unsplit, or an explicit multiple of 32 and of the
block size), runs the call through the C ABI and compares every output row with the fp64
oracle: within 4e-3 / 5e-4 (max / mean absolute error), and for E4M3 also within the element
bound of the tensor-core arithmetic.  The device error word must stay clear.
"""
import random

import pytest
import torch

import oracle
from helpers import assert_close, assert_close_weighted, e4m3_magnitudes
from paged_kv_decode_21_gb300 import ops, workloads

pytestmark = pytest.mark.gpu

KS, VS = workloads.E4M3_SCALES["full"]
N_CASES = 200


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_decode_21_gb300 import build
    build.build()
    ops.lib()


def draw(i):
    rng = random.Random(1000 + i)
    Hkv = rng.choice([1, 2, 4, 8])
    G = rng.randint(1, 8)
    fp8 = rng.random() < 0.3
    D = 128 if fp8 else rng.choice([64, 128])
    BS = rng.choice([16, 32])
    B = rng.randint(1, 12)
    lens = [rng.choice([0, 1, rng.randint(2, 64), rng.randint(65, 3000)]) for _ in range(B)]
    lens[rng.randrange(B)] = max(max(lens), 1)
    q_len = rng.choice([1, 1, 1, 1, 2, 4, 8, 17])
    if q_len == 1 and not fp8:
        variant = rng.choice(["auto", "no_prefetch", "l2_prefetch", "tma_staged", "tma_mma", "tcgen05",
                              "tma_mma+longest_first", "tcgen05+longest_first"])
    else:
        variant = rng.choice(["auto", "tma_mma", "tcgen05"])
        if fp8 and variant == "tcgen05" and D != 128:
            variant = "auto"
    step = max(32, BS)
    partition = rng.choice([0, 0, -1, step * rng.randint(1, 16)])
    return dict(Hkv=Hkv, G=G, D=D, BS=BS, lens=lens, q_len=q_len, fp8=fp8, variant=variant,
                partition=partition, seed=2000 + i)


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_shape_matches_oracle(i):
    c = draw(i)
    Hq = c["Hkv"] * c["G"]
    B, D, q_len = len(c["lens"]), c["D"], c["q_len"]
    inp = workloads.make_custom(B, Hq, c["Hkv"], D, c["BS"], c["lens"], seed=c["seed"], device="cuda")
    g = torch.Generator(device="cuda").manual_seed(c["seed"] + 1)
    q = inp.q if q_len == 1 else workloads.randn_f16((B, q_len, Hq, D), g, "cuda")
    ew = torch.zeros(1, dtype=torch.int32, device="cuda")
    host = (inp.block_tables.cpu(), inp.context_lens.cpu())
    what = str(c)
    if c["fp8"]:
        k8 = workloads.rand_e4m3(inp.k_cache.shape, g, "cuda")
        v8 = workloads.rand_e4m3(inp.v_cache.shape, g, "cuda")
        out = ops.paged_decode_attention_fp8(q, k8, v8, inp.block_tables, inp.context_lens, inp.scale, KS, VS,
                                             max_context_len=inp.max_context_len, partition_size=c["partition"],
                                             error_word=ew,
                                             variant=None if c["variant"] == "auto" else c["variant"])
        ref = oracle.attention_fp8(q.cpu(), k8.cpu(), v8.cpu(), *host, inp.scale, KS, VS)
        absref = oracle.attention_fp8(q.cpu(), k8.cpu(), e4m3_magnitudes(v8).cpu(), *host, inp.scale, KS, VS)
        assert_close_weighted(out, ref, absref, 448.0 * VS, max(c["lens"]), what)
    elif q_len > 1:
        out = ops.paged_decode_attention_multi(q, inp.k_cache, inp.v_cache, inp.block_tables, inp.context_lens,
                                               inp.scale, max_context_len=inp.max_context_len,
                                               partition_size=c["partition"], error_word=ew,
                                               variant=c["variant"])
        ref = oracle.attention_multi(q.cpu(), inp.k_cache.cpu(), inp.v_cache.cpu(), *host, inp.scale)
        assert_close(out, ref, what)
    else:
        out = ops.paged_decode_attention_ex(inp.q, inp.k_cache, inp.v_cache, inp.block_tables, inp.context_lens,
                                            inp.scale, max_context_len=inp.max_context_len,
                                            partition_size=c["partition"], variant=c["variant"], error_word=ew)
        ref = oracle.attention(inp.q.cpu(), inp.k_cache.cpu(), inp.v_cache.cpu(), *host, inp.scale)
        assert_close(out, ref, what)
    assert ops.pkd_read_device_error(ew) == 0, what
