"""GPU parity over seeded random shapes sized for the tcgen05 path's scheduling: the split of
a short last round (an unsplit grid walked longest first) and runs of short partitions per CTA.

Each case draws a group size, kv heads, query tokens, cache type and a length mix (uniform,
ragged, with empty and tiny sequences), and a batch just past a whole number of rounds of
resident CTAs (two per SM) or an explicit partition of 256-1024 tokens with enough units for
runs.  The plan must take the scheduling the case is for; every output row is compared with
the fp64 oracle (E4M3 also against the element bound of the tensor-core arithmetic), and the
device error word must stay clear.
"""
import random

import pytest
import torch

import oracle
from helpers import assert_close, assert_close_weighted, e4m3_magnitudes
from paged_kv_decode_21_gb300 import ops, workloads

pytestmark = pytest.mark.gpu

KS, VS = workloads.E4M3_SCALES["full"]
N_CASES = 48


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_decode_21_gb300 import build
    build.build()
    ops.lib()


def slots():
    return torch.cuda.get_device_properties(0).multi_processor_count * 2


def draw(i):
    rng = random.Random(5000 + i)
    G = rng.choice([4, 5, 7])
    Hkv = rng.choice([4, 8])
    q_len = rng.choice([4, 8]) if G > 4 else 8  # two 16-row tiles or more: the tcgen05 path
    fp8 = rng.random() < 0.4
    L = rng.choice([1024, 1536, 2048, 3000])
    mix = rng.choice(["uniform", "ragged", "zeros", "tiny_tail"])
    if i % 2 == 0:  # a short last round: rounds + a few sequences' worth of CTAs
        kind = "tail"
        rounds = rng.choice([2, 3])
        B = (rounds * slots()) // Hkv + rng.randint(1, max(1, slots() // (4 * Hkv)))
        P = 0
    else:  # runs of short partitions: enough units that runs of two keep four waves of CTAs
        kind = "runs"
        P = rng.choice([256, 512, 1024])
        L = max(L, 2048)
        pairs = -(-(-(-L // P)) // 2)
        B = -(-4 * slots() // (Hkv * pairs)) + rng.randint(0, 8)
    lens = [L] * B
    if mix == "ragged":
        lens = [rng.randint(L // 2, L) for _ in range(B)]
    elif mix == "zeros":
        lens = [rng.choice([0, rng.randint(1, L)]) for _ in range(B)]
    elif mix == "tiny_tail":
        lens = [rng.randint(L // 2, L) for _ in range(B)]
        for k in rng.sample(range(B), 6):
            lens[k] = rng.choice([0, 1, q_len - 1, 63, 64, 65, 200])
    lens[rng.randrange(B)] = L
    return dict(kind=kind, G=G, Hkv=Hkv, q_len=q_len, fp8=fp8, L=L, B=B, P=P, lens=lens, mix=mix, seed=6000 + i)


@pytest.mark.parametrize("i", range(N_CASES))
def test_scheduling_matches_oracle(i):
    c = draw(i)
    B, Hkv, G, q_len, L, P = c["B"], c["Hkv"], c["G"], c["q_len"], c["L"], c["P"]
    Hq = Hkv * G
    what = {k: v for k, v in c.items() if k != "lens"}
    n, part, ordered, var, grid, _ = ops.paged_decode_call_plan(B, q_len, Hq, Hkv, 128, 16, L, kv_fp8=c["fp8"],
                                                                partition_size=P)
    assert var.startswith("tcgen05"), what
    units = B * Hkv
    if c["kind"] == "tail":
        last = units - (units - 1) // slots() * slots()
        assert part == -1 and ordered and 2 * last <= slots() and grid == (B + -(-last // Hkv)) * Hkv, what
    else:
        assert part == P and grid < units * -(-L // P), what
    inp = workloads.make_custom(B, Hq, Hkv, 128, 16, c["lens"], seed=c["seed"], device="cuda",
                                max_blocks_per_seq=-(-L // 16))
    g = torch.Generator(device="cuda").manual_seed(c["seed"] + 1)
    q = workloads.randn_f16((B, q_len, Hq, 128), g, "cuda")
    ew = torch.zeros(1, dtype=torch.int32, device="cuda")
    host = (inp.block_tables.cpu(), inp.context_lens.cpu())
    if c["fp8"]:
        k8 = workloads.rand_e4m3(inp.k_cache.shape, g, "cuda")
        v8 = workloads.rand_e4m3(inp.v_cache.shape, g, "cuda")
        out = ops.paged_decode_attention_fp8(q, k8, v8, inp.block_tables, inp.context_lens, inp.scale, KS, VS,
                                             max_context_len=L, partition_size=P, error_word=ew)
        ref = oracle.attention_fp8(q.cpu(), k8.cpu(), v8.cpu(), *host, inp.scale, KS, VS)
        absref = oracle.attention_fp8(q.cpu(), k8.cpu(), e4m3_magnitudes(v8).cpu(), *host, inp.scale, KS, VS)
        assert_close_weighted(out, ref, absref, 448.0 * VS, L, str(what))
    else:
        out = ops.paged_decode_attention_multi(q, inp.k_cache, inp.v_cache, inp.block_tables, inp.context_lens,
                                               inp.scale, max_context_len=L, partition_size=P, error_word=ew)
        ref = oracle.attention_multi(q.cpu(), inp.k_cache.cpu(), inp.v_cache.cpu(), *host, inp.scale)
        assert_close(out, ref, str(what))
    assert ops.pkd_read_device_error(ew) == 0, what
