"""The whole operation from host buffers (paged_decode_attention_host).

Inputs live in page-locked host memory; the library copies them to the
caller's device buffers (the cache pools either whole or only the blocks the
tables reference, read in place over the host link), decodes, and copies the
output back.  The result must equal the device-resident call bit for bit (the
same kernels on the same used bytes) and match the fp64 oracle.
"""
import pytest
import torch

from helpers import assert_close, oracle_out
from paged_kv_decode_21_gb300 import ops, workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_decode_21_gb300 import build
    build.build()
    ops.lib()


class Dev:
    """Device buffers the host call copies into (the pools start as NaN)."""

    def __init__(self, inp):
        self.q = torch.empty_like(inp.q, device="cuda")
        self.k_cache = torch.full(inp.k_cache.shape, float("nan"), dtype=inp.k_cache.dtype, device="cuda")
        self.v_cache = torch.full(inp.v_cache.shape, float("nan"), dtype=inp.v_cache.dtype, device="cuda")
        self.block_tables = torch.empty_like(inp.block_tables, device="cuda")
        self.context_lens = torch.empty_like(inp.context_lens, device="cuda")
        self.out = torch.empty_like(inp.q, device="cuda")


def host_inputs(lens, Hq, Hkv, D, BS, seed, share=False):
    inp = workloads.make_custom(len(lens), Hq, Hkv, D, BS, lens, seed=seed, device="cpu")
    if share and len(lens) >= 2:
        # sequence 1 reuses sequence 0's first block (a shared prefix)
        inp.block_tables[1, 0] = inp.block_tables[0, 0]
    for n in ("q", "k_cache", "v_cache", "block_tables", "context_lens"):
        setattr(inp, n, getattr(inp, n).pin_memory())
    return inp


def device_reference(inp):
    d = inp.to("cuda")
    return ops.paged_decode_attention_ex(d.q, d.k_cache, d.v_cache, d.block_tables, d.context_lens, d.scale,
                                         max_context_len=d.max_context_len, partition_size=0)


@pytest.mark.parametrize("used_only", [True, False])
@pytest.mark.parametrize("shape", [
    ([37, 100], 4, 4, 64, 16, False),
    ([300, 17, 2048, 0, 129], 32, 8, 128, 16, True),
    ([1, 31, 32, 33, 700], 16, 2, 128, 32, True),
])
def test_host_call_matches_device_call(shape, used_only):
    lens, Hq, Hkv, D, BS, share = shape
    inp = host_inputs(lens, Hq, Hkv, D, BS, seed=len(lens) + D, share=share)
    dev = Dev(inp)
    out = torch.empty(inp.q.shape, dtype=inp.q.dtype).pin_memory()
    ew = torch.zeros(1, dtype=torch.int32, device="cuda")
    ops.paged_decode_attention_host(inp.q, inp.k_cache, inp.v_cache, inp.block_tables, inp.context_lens, out, dev,
                                    inp.scale, max_context_len=inp.max_context_len, used_blocks_only=used_only,
                                    error_word=ew)
    torch.cuda.synchronize()
    assert ops.pkd_read_device_error(ew) == 0
    assert torch.equal(out, device_reference(inp).cpu())
    assert_close(out, oracle_out(inp), f"host call {lens[:3]}")


def test_host_call_full_size():
    cfg = workloads.CONFIGS["llama3_8b_gqa4"]
    inp = workloads.make_inputs(cfg, device="cpu")
    for n in ("q", "k_cache", "v_cache", "block_tables", "context_lens"):
        setattr(inp, n, getattr(inp, n).pin_memory())
    dev = Dev(inp)
    out = torch.empty(inp.q.shape, dtype=inp.q.dtype).pin_memory()
    ops.paged_decode_attention_host(inp.q, inp.k_cache, inp.v_cache, inp.block_tables, inp.context_lens, out, dev,
                                    inp.scale, max_context_len=inp.max_context_len)
    torch.cuda.synchronize()
    assert torch.equal(out, device_reference(inp).cpu())


def test_host_call_bad_block_is_reported():
    inp = host_inputs([40, 20], 4, 4, 128, 16, seed=29)
    inp.block_tables[0, 1] = inp.num_blocks + 1000   # outside the pool: checked, never dereferenced
    dev = Dev(inp)
    out = torch.empty(inp.q.shape, dtype=inp.q.dtype).pin_memory()
    ew = torch.zeros(1, dtype=torch.int32, device="cuda")
    ops.paged_decode_attention_host(inp.q, inp.k_cache, inp.v_cache, inp.block_tables, inp.context_lens, out, dev,
                                    inp.scale, max_context_len=inp.max_context_len, error_word=ew)
    torch.cuda.synchronize()
    assert ops.pkd_read_device_error(ew) & ops.DEVERR_BAD_BLOCK
