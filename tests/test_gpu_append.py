"""GPU parity of the paged KV append (the cache write before each decode step).

paged_kv_append is called through the C ABI and its caches are compared with
``oracle.append`` bit for bit (it is pure data movement: every element must
match exactly, and every row it does not target must be left untouched).
Then the decode kernels read the grown sequences back and are compared with
the oracle's attention over the oracle-appended caches.
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


def new_rows(num_seqs, num_kv_heads, head_dim, seed, device="cuda"):
    g = torch.Generator(device=device).manual_seed(seed)
    k = workloads.randn_f16((num_seqs, num_kv_heads, head_dim), g, device)
    v = workloads.randn_f16((num_seqs, num_kv_heads, head_dim), g, device)
    return k, v


def grown_problem(lens, Hq, Hkv, D, BS, seed, **kw):
    """Inputs whose tables already hold the block of position lens[b]."""
    inp = workloads.make_custom(len(lens), Hq, Hkv, D, BS, [L + 1 for L in lens], seed=seed,
                                device="cuda", **kw)
    cl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    return inp, cl


@pytest.mark.parametrize("D,BS,Hkv", [(128, 16, 4), (64, 32, 8), (8, 16, 3), (72, 1, 2)])
def test_append_is_bit_exact(D, BS, Hkv):
    # ragged lengths: empty, block boundaries on both sides, one long sequence
    lens = [0, 1, BS - 1, BS, BS + 1, 2 * BS, 37, 700]
    inp, cl = grown_problem(lens, Hkv, Hkv, D, BS, seed=D + BS)
    k_new, v_new = new_rows(len(lens), Hkv, D, seed=11)
    ref_k, ref_v = oracle.append(k_new.cpu(), v_new.cpu(), inp.block_tables.cpu(), cl.cpu(),
                                 inp.k_cache.cpu(), inp.v_cache.cpu())
    ew = torch.zeros(1, dtype=torch.int32, device="cuda")
    ops.paged_kv_append(k_new, v_new, inp.block_tables, cl, inp.k_cache, inp.v_cache, error_word=ew)
    assert ops.pkd_read_device_error(ew) == 0
    assert np.array_equal(inp.k_cache.cpu().numpy().view(np.uint16), ref_k.view(np.uint16))
    assert np.array_equal(inp.v_cache.cpu().numpy().view(np.uint16), ref_v.view(np.uint16))


def test_append_then_decode_matches_oracle():
    lens = [0, 15, 16, 31, 100, 511, 1023]
    Hq, Hkv, D, BS = 28, 4, 128, 16
    inp, cl = grown_problem(lens, Hq, Hkv, D, BS, seed=5)
    k_new, v_new = new_rows(len(lens), Hkv, D, seed=6)
    ref_k, ref_v = oracle.append(k_new.cpu(), v_new.cpu(), inp.block_tables.cpu(), cl.cpu(),
                                 inp.k_cache.cpu(), inp.v_cache.cpu())
    ops.paged_kv_append(k_new, v_new, inp.block_tables, cl, inp.k_cache, inp.v_cache)
    grown = cl + 1
    ref = oracle.attention(inp.q.cpu(), ref_k, ref_v, inp.block_tables.cpu(), grown.cpu(), inp.scale)
    for variant, P in [("auto", 0), ("tma_staged", 256), ("l2_prefetch", -1), ("no_prefetch", 64)]:
        out = ops.paged_decode_attention_ex(inp.q, inp.k_cache, inp.v_cache, inp.block_tables, grown,
                                            inp.scale, max_context_len=max(lens) + 1,
                                            partition_size=P, variant=variant)
        assert_close(out, ref, f"append+decode {variant} P={P}")


def test_append_skips_and_reports_bad_rows():
    lens = [5, 32, 9, 20]
    Hkv, D, BS = 2, 64, 16
    inp, cl = grown_problem(lens, Hkv, Hkv, D, BS, seed=9, max_blocks_per_seq=3)
    bt = inp.block_tables.clone()
    cl[1] = 48                   # 48 / 16 = 3 >= max_blocks_per_seq: no room
    bt[2, 0] = inp.num_blocks    # entry outside the pool
    bt[3, 1] = -1                # unallocated entry
    k_new, v_new = new_rows(len(lens), Hkv, D, seed=10)
    k0, v0 = inp.k_cache.clone(), inp.v_cache.clone()
    ew = torch.zeros(1, dtype=torch.int32, device="cuda")
    ops.paged_kv_append(k_new, v_new, bt, cl, inp.k_cache, inp.v_cache, error_word=ew)
    assert ops.pkd_read_device_error(ew) == ops.DEVERR_BAD_BLOCK
    # only sequence 0 was written, exactly where the oracle writes it
    one = torch.tensor([lens[0]], dtype=torch.int32)
    ref_k, ref_v = oracle.append(k_new[:1].cpu(), v_new[:1].cpu(), bt[:1].cpu(), one,
                                 k0.cpu(), v0.cpu())
    assert np.array_equal(inp.k_cache.cpu().numpy().view(np.uint16), ref_k.view(np.uint16))
    assert np.array_equal(inp.v_cache.cpu().numpy().view(np.uint16), ref_v.view(np.uint16))
    # and the oracle flags the same sequences
    with pytest.raises(oracle.OracleError):
        oracle.append(k_new.cpu(), v_new.cpu(), bt.cpu(), cl.cpu(), k0.cpu(), v0.cpu())


def test_append_full_size_mha():
    # Llama2-7B shape (64 sequences x 32 kv heads x 128) at 2048 tokens: the
    # append of token 2047 into the last slot of each sequence's last block.
    cfg = workloads.CONFIGS["llama2_7b_mha"]
    inp = workloads.make_inputs(cfg, device="cuda")
    cl = inp.context_lens - 1
    k_new, v_new = new_rows(cfg.num_seqs, cfg.num_kv_heads, cfg.head_dim, seed=21)
    k0, v0 = inp.k_cache.clone(), inp.v_cache.clone()
    ew = torch.zeros(1, dtype=torch.int32, device="cuda")
    ops.paged_kv_append(k_new, v_new, inp.block_tables, cl, inp.k_cache, inp.v_cache, error_word=ew)
    assert ops.pkd_read_device_error(ew) == 0
    # the targets hold the new rows ...
    b = torch.arange(cfg.num_seqs, device="cuda")
    phys = inp.block_tables[b, (cl // cfg.block_size).long()].long()
    slot = (cl % cfg.block_size).long()
    assert torch.equal(inp.k_cache[phys, :, slot, :], k_new)
    assert torch.equal(inp.v_cache[phys, :, slot, :], v_new)
    # ... and putting the old rows back restores the caches bit for bit
    inp.k_cache[phys, :, slot, :] = k0[phys, :, slot, :]
    inp.v_cache[phys, :, slot, :] = v0[phys, :, slot, :]
    assert torch.equal(inp.k_cache, k0) and torch.equal(inp.v_cache, v0)
    del k0, v0
    # decode over the appended caches, sampled rows against the oracle
    ops.paged_kv_append(k_new, v_new, inp.block_tables, cl, inp.k_cache, inp.v_cache)
    rows = sample_rows(cfg.num_seqs, cfg.num_q_heads, 48, seed=3)
    out = ops.paged_decode_attention_ex(inp.q, inp.k_cache, inp.v_cache, inp.block_tables,
                                        inp.context_lens, inp.scale,
                                        max_context_len=inp.max_context_len)
    ref = oracle.attention(inp.q.cpu(), inp.k_cache.cpu(), inp.v_cache.cpu(), inp.block_tables.cpu(),
                           inp.context_lens.cpu(), inp.scale, rows=rows)
    got = out.view(-1, cfg.head_dim)[torch.as_tensor(rows, device="cuda").long()]
    assert_close(got, ref.reshape(len(rows), cfg.head_dim), "full-size append+decode")
