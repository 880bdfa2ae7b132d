"""The library's calls inside CUDA graphs: a serving loop captures each step
(cache write + decode) once and replays it.  Every call here is captured on
torch's capture stream and the replay must equal the direct calls bit for
bit (same kernels, same inputs)."""
import numpy as np
import pytest
import torch

from paged_kv_decode_21_gb300 import ops, workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_decode_21_gb300 import build
    build.build()
    ops.lib()


def test_append_then_decode_step_replays_in_a_graph():
    lens = [100, 33, 700, 512]
    Hq, Hkv, D, BS = 32, 8, 128, 16
    inp = workloads.make_custom(len(lens), Hq, Hkv, D, BS, [L + 1 for L in lens], seed=5, device="cuda")
    cl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    grown = cl + 1
    g = torch.Generator(device="cuda").manual_seed(6)
    k_new = workloads.randn_f16((len(lens), Hkv, D), g, "cuda")
    v_new = workloads.randn_f16((len(lens), Hkv, D), g, "cuda")
    P = 256  # split, so the merge kernel is captured as well
    need = ops.paged_decode_workspace_size(len(lens), Hq, Hkv, D, BS, max(lens) + 1, P, 0)
    ws = ops.alloc_workspace(need, "cuda")
    out = torch.empty_like(inp.q)
    k0, v0 = inp.k_cache.clone(), inp.v_cache.clone()

    def step():
        ops.paged_kv_append(k_new, v_new, inp.block_tables, cl, inp.k_cache, inp.v_cache)
        ops.paged_decode_attention_ex(inp.q, inp.k_cache, inp.v_cache, inp.block_tables, grown, inp.scale,
                                      out=out, max_context_len=max(lens) + 1, partition_size=P, workspace=ws)

    step()  # direct (also loads every kernel before capture)
    torch.cuda.synchronize()
    direct = out.clone()
    k_direct = inp.k_cache.clone()
    # restore the caches, capture, replay
    inp.k_cache.copy_(k0)
    inp.v_cache.copy_(v0)
    out.zero_()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, direct)
    assert torch.equal(inp.k_cache, k_direct)
    # replay again with new queries: the graph reads the live buffers
    inp.q.mul_(-1)
    graph.replay()
    torch.cuda.synchronize()
    again = out.clone()
    ops.paged_decode_attention_ex(inp.q, inp.k_cache, inp.v_cache, inp.block_tables, grown, inp.scale,
                                  out=out, max_context_len=max(lens) + 1, partition_size=P, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(again, out)


def test_fp8_and_multi_token_calls_replay_in_a_graph():
    lens = [300, 64, 129]
    Hq, Hkv, D, BS = 28, 4, 128, 16
    inp = workloads.make_custom(len(lens), Hq, Hkv, D, BS, lens, seed=9, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(10)
    k8 = workloads.rand_e4m3(inp.k_cache.shape, g, "cuda")
    v8 = workloads.rand_e4m3(inp.v_cache.shape, g, "cuda")
    qm = workloads.randn_f16((len(lens), 3, Hq, D), g, "cuda")
    need8 = ops.paged_decode_multi_workspace_size(len(lens), 1, Hq, Hkv, D, BS, max(lens), 64)
    needm = ops.paged_decode_multi_workspace_size(len(lens), 3, Hq, Hkv, D, BS, max(lens), 64)
    ws8 = ops.alloc_workspace(need8, "cuda")
    wsm = ops.alloc_workspace(needm, "cuda")
    out8 = torch.empty_like(inp.q)
    outm = torch.empty_like(qm)

    def step():
        ops.paged_decode_attention_fp8(inp.q, k8, v8, inp.block_tables, inp.context_lens, inp.scale, 0.05, 0.11,
                                       out=out8, max_context_len=max(lens), partition_size=64, workspace=ws8)
        ops.paged_decode_attention_multi(qm, inp.k_cache, inp.v_cache, inp.block_tables, inp.context_lens,
                                         inp.scale, out=outm, max_context_len=max(lens), partition_size=64,
                                         workspace=wsm)

    step()
    torch.cuda.synchronize()
    d8, dm = out8.clone(), outm.clone()
    out8.zero_()
    outm.zero_()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(out8, d8)
    assert torch.equal(outm, dm)
