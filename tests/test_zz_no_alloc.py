"""The split-K entry point for callers that cannot allocate device memory.

paged_decode_attention_static_scratch keeps its partials in a fixed device
array owned by the library (for callers such as plugins or code under a
foreign allocator that may not call cudaMalloc nor pass a workspace).  Here it
is called through the C ABI twice in a row, on two different shapes, and each
result is checked against the fp64 CPU oracle and against the ordinary entry
point, paged_decode_attention_ex with a caller workspace, within the parity
tolerance of the GPU suite.  A shape whose partials would not fit in the array
is refused before launch.

This file is collected last on purpose; it also passes alone in a fresh
process.
"""
import numpy as np
import pytest
import torch

from helpers import MAX_ABS_TOL, MEAN_ABS_TOL, assert_close, oracle_out
from paged_kv_decode_21_gb300 import ops, workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_decode_21_gb300 import build
    build.build()
    ops.lib()


def _close(a: torch.Tensor, b: torch.Tensor, what: str):
    d = (a.double() - b.double()).abs().cpu().numpy()
    assert np.all(np.isfinite(a.cpu().double().numpy())), what
    assert d.max(initial=0.0) <= MAX_ABS_TOL and d.mean() <= MEAN_ABS_TOL, (what, d.max(), d.mean())


def _both(inp, partition_size, variant):
    ew = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = ops.paged_decode_attention_static_scratch(
        inp.q, inp.k_cache, inp.v_cache, inp.block_tables, inp.context_lens, inp.scale,
        max_context_len=inp.max_context_len, partition_size=partition_size, variant=variant,
        error_word=ew)
    ref = ops.paged_decode_attention_ex(
        inp.q, inp.k_cache, inp.v_cache, inp.block_tables, inp.context_lens, inp.scale,
        max_context_len=inp.max_context_len, partition_size=partition_size, variant=variant)
    torch.cuda.synchronize()
    assert ops.pkd_read_device_error(ew) == 0
    return got, ref


@pytest.mark.parametrize("variant", ["tma_staged", "l2_prefetch"])
def test_static_scratch_matches_workspace_path_twice(variant):
    # first call: GQA 7:1 with long, ragged and empty sequences, split at 256
    a = workloads.make_custom(4, 28, 4, 128, 16, [700, 33, 0, 1500], seed=41, device="cuda")
    got_a, ref_a = _both(a, 256, variant)
    assert_close(got_a, oracle_out(a), "first call against the oracle")
    _close(got_a, ref_a, "first call")
    # second call in a row: a smaller, different shape reusing the same array
    b = workloads.make_custom(3, 8, 8, 64, 32, [100, 37, 300], seed=43, device="cuda")
    got_b, ref_b = _both(b, 64, variant)
    assert_close(got_b, oracle_out(b), "second call against the oracle")
    _close(got_b, ref_b, "second call")
    # and the first shape again, after the array holds the second call's partials
    got_a2, _ = _both(a, 256, variant)
    assert torch.equal(got_a2, got_a)


def test_static_scratch_automatic_partition():
    c = workloads.make_custom(2, 40, 8, 128, 16, [5000, 9000], seed=47, device="cuda")
    got, ref = _both(c, 0, "auto")
    assert_close(got, oracle_out(c), "automatic partition against the oracle")
    _close(got, ref, "automatic partition")


def test_static_scratch_rejects_oversized_shapes():
    # 64 x 40 heads x 64 partitions x 130 floats > the array: refused on the host
    big = workloads.make_custom(1, 40, 8, 128, 16, [64], seed=53, device="cuda")
    q = torch.zeros(64, 40, 128, dtype=torch.float16, device="cuda")
    bt = torch.zeros(64, 128, dtype=torch.int32, device="cuda")
    cl = torch.full((64,), 64, dtype=torch.int32, device="cuda")
    with pytest.raises(ops.PagedDecodeError) as e:
        ops.paged_decode_attention_static_scratch(q, big.k_cache, big.v_cache, bt, cl, big.scale,
                                                  max_context_len=64 * 32, partition_size=32)
    assert e.value.status == 5  # PKD_ERR_WORKSPACE
