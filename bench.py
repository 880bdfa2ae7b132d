"""Benchmark: paged single-query decode attention on GB300.

One step = one call of paged_decode_attention_ex (every stage of the hot
path: block-table gather, Q.K^T, online softmax, P.V, and the split-K merge
when the shape splits) over one batch of synthetic inputs already resident
in HBM.  The default workload is the Llama2-7B-shaped MHA decode (batch 64,
32 q / 32 kv heads, head_dim 128, block_size 16, context 2048).

Prints ONE JSON line (rank 0).  ``--impl reference`` times the CPU oracle
instead.  ``--sweep`` prints one line per (workload, variant) to stdout.

Timing: W warm-up calls, then K timed calls, each bracketed by CUDA events
on the launching stream.  A workload whose algorithmic bytes exceed 4x the
L2 size runs its calls back to back: the inputs are larger than L2, and a
call's first reads are the blocks the previous call read first, long
evicted.  Smaller workloads get an L2 flush before every call: a read of a
buffer twice the L2 size, which leaves only clean lines behind.  (A write
flush would leave L2 full of dirty lines whose write-back lands inside the
next call: about 5% of the MHA call, more of a short one.)  value =
algorithmic bytes (K and V rows used, Q, out) per call / mean call time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time
import types

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from paged_kv_decode_21_gb300 import traffic, workloads  # noqa: E402

METRIC = "paged decode-attention achieved HBM GB/s (% of GB300 peak); μs per call"
DEFAULT_CONFIG = "llama2_7b_mha"
# the other large workloads the default run also times and checks, each as an extra key of the line
EXTRA_CONFIGS = ["llama3_8b_gqa4", "qwen25_7b_gqa7", "qwen25_14b_gqa5_splitk"]
FALLBACK_HBM_GBS = 6800.0
# GB300's nominal HBM3e bandwidth (datasheet figure), for a fraction of the nameplate peak
NOMINAL_HBM_GBS = 7900.0
# parity contract of the fp16 output against the fp64 oracle, over every output element
PARITY_MAX_ABS = 4e-3
PARITY_MEAN_ABS = 5e-4
KERNEL_SOURCES = ["paged_kv_decode_21_gb300/csrc/pkd_decode.cuh", "paged_kv_decode_21_gb300/csrc/pkd_decode_ws.cuh",
                  "paged_kv_decode_21_gb300/csrc/pkd_decode_mma.cuh", "paged_kv_decode_21_gb300/csrc/pkd_ptx.cuh",
                  "paged_kv_decode_21_gb300/csrc/pkd_launch.cuh", "paged_kv_decode_21_gb300/csrc/pkd_inst_tma_mma.cu"]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "ncu_traffic.json")


def describe(cfg: workloads.DecodeConfig) -> str:
    if cfg.context_lens is not None:
        lens = sorted(set(cfg.context_lens))
        ltxt = f"context_len={lens[0]}" if len(lens) == 1 else f"context_lens={lens}"
    else:
        ltxt = f"context_lens~U[{cfg.len_range[0]},{cfg.len_range[1]}]"
    ptxt = f", partition={cfg.partition_size}" if cfg.partition_size else ""
    return (f"{cfg.name}: batch={cfg.num_seqs}, {cfg.num_q_heads} q / {cfg.num_kv_heads} kv heads, "
            f"head_dim={cfg.head_dim}, block_size={cfg.block_size}, {ltxt}{ptxt}, fp16")


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_hash() -> str:
    h = hashlib.sha256()
    for p in KERNEL_SOURCES:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def kernel_name(cfg: workloads.DecodeConfig, variant: str, kv_fp8: bool = False, wide: bool = False,
                q_len: int = 1) -> str:
    """The decode kernel a resolved variant launches for a shape (template arguments: head
    dim, block size, group, query tokens per CTA, bytes per K/V element, CTAs per SM with 0
    for the default three; the tcgen05 kernel takes the block size only)."""
    path = variant.split("+")[0]
    shape = f"{cfg.head_dim},{cfg.block_size},{cfg.group}"
    if path == "tcgen05":
        return f"paged_decode_tc_kernel<{cfg.block_size},{1 if kv_fp8 else 2},{cfg.head_dim}>"
    if path == "tma_mma":
        # single-query E4M3 grids of 3+ waves of four CTAs per SM run the four-per-SM build
        qc = 1 if q_len <= 1 else 16 // cfg.group
        return f"paged_decode_mma_kernel<{shape},{qc},{1 if kv_fp8 else 2},{4 if (kv_fp8 and wide) else 0}>"
    if path == "tma_staged" and cfg.group >= 6:
        return f"paged_decode_ws_kernel<{shape}>"
    return f"paged_decode_kernel<{shape},{variant}>"


def dtype_label(resolved: str, kv_fp8: bool) -> str:
    """The arithmetic a resolved data path does: fp32 scores, softmax and
    accumulation; on the tensor-core paths the weights p are rounded to fp16
    before P.V (the normaliser sums the fp32 p)."""
    tc = resolved.split("+")[0] in ("tma_mma", "tcgen05")
    base = ("e4m3 K/V (widened exactly to f16), f16 q/out" if kv_fp8 else "f16 q/K/V/out") + ", f32 arithmetic"
    return base + ("; p rounded to f16 for P.V" if tc else "")


def parity(out: torch.Tensor, ref) -> dict:
    """Element-by-element comparison of a GPU output with the oracle's, over every row."""
    import numpy as np
    got = out.detach().cpu().to(torch.float64).numpy().reshape(ref.shape)
    err = np.abs(got - ref)
    finite = bool(np.isfinite(got).all())
    mx = float(err.max(initial=0.0)) if finite else float("inf")
    mean = float(err.mean()) if finite and err.size else 0.0
    return {"max_abs": mx, "mean_abs": mean, "max_abs_ref": float(np.abs(ref).max(initial=0.0)),
            "rows": "all", "n_rows": int(err.size // ref.shape[-1]),
            "tol": {"max_abs": PARITY_MAX_ABS, "mean_abs": PARITY_MEAN_ABS},
            "ok": bool(finite and mx <= PARITY_MAX_ABS and mean <= PARITY_MEAN_ABS)}


def ncu_traffic(workload: str, variant: str):
    """dram bytes per launch from the committed ncu capture, if it matches this kernel."""
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f)
    except Exception:
        return None
    ent = rec.get("entries", {}).get(f"{workload}/{variant}")
    if not ent or ent.get("kernel_hash") != kernel_hash():
        return None
    return ent.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the timed loop runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap,clocks.mem,temperature.memory")

    def __init__(self, device_index: int):
        self.samples = []
        self.proc = None
        self.idx = device_index

    def __enter__(self):
        try:
            bus = torch.cuda.get_device_properties(self.idx).pci_bus_id
        except Exception:
            bus = None
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100"]
        if bus:
            cmd += ["-i", str(bus)]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append([x.strip() for x in line.split(",")])

    def __exit__(self, *exc):
        if self.proc:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons, mem, mtemp = [], [], set(), [], []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for s in self.samples:
            try:
                sm.append(float(s[0]))
                mx.append(float(s[1]))
            except Exception:
                continue
            for n, v in zip(names, s[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
            for dst, v in ((mem, s[7:8]), (mtemp, s[8:9])):
                try:
                    dst.append(float(v[0]))
                except Exception:
                    pass
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        out = {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
               "samples": len(sm)}
        if mem:
            out["mem_mhz"] = statistics.median(mem)
        if mtemp:
            out["mem_temp_c_max"] = max(mtemp)
        return out


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def aggregate_over_ranks(mean_ms: float, algo_bytes: int, world_size: int, device=None):
    """Whole-job value of N replicas: each rank ran the same workload; the
    job's per-call time is the max over ranks, and the job moved N x the
    bytes.  Returns (max per-call ms, aggregate GB/s)."""
    if world_size > 1:
        t = torch.tensor([mean_ms], dtype=torch.float64, device=device)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        mean_ms = float(t.item())
    return mean_ms, world_size * algo_bytes / (mean_ms * 1e-3) / 1e9


class L2Flush:
    """Evicts L2 by reading a buffer of twice its size (clean lines only: no
    write-back of the flush can land inside the next timed call)."""

    def __init__(self, dev, l2):
        self.buf = torch.ones(max(2 * l2, 256 << 20) // 4, dtype=torch.int32, device=dev)
        self.sink = torch.empty((), dtype=torch.int64, device=dev)

    def __call__(self):
        torch.sum(self.buf, dim=0, dtype=torch.int64, out=self.sink)


def time_gpu(args, cfg, variant, dev, inp, steps, warmup, with_e2e=True, with_clocks=True):
    """Kernel-resident timing (+ optional end-to-end leg) of one workload and variant."""
    from paged_kv_decode_21_gb300 import ops
    stream = torch.cuda.current_stream(dev)
    lens = inp.context_lens.cpu().tolist()
    algo = traffic.algorithmic_bytes(lens, inp.num_q_heads, inp.num_kv_heads, inp.head_dim)
    P = args.partition_size if args.partition_size is not None else (cfg.partition_size or 0)
    var = ops._variant(variant)
    need = ops.paged_decode_workspace_size(inp.num_seqs, inp.num_q_heads, inp.num_kv_heads,
                                           inp.head_dim, inp.block_size, inp.max_context_len, P, var)
    ws = ops.alloc_workspace(need, dev)
    q_len = getattr(args, "q_len", 1)
    kv_fp8 = getattr(args, "kv_fp8", False)
    # the library's own plan: partition, order, data path, decode CTAs, launches
    launches, eff_P, ordered, resolved, grid, pdist = ops.paged_decode_call_plan(
        inp.num_seqs, q_len, inp.num_q_heads, inp.num_kv_heads, inp.head_dim, inp.block_size,
        inp.max_context_len, kv_fp8, P, variant)
    split = eff_P > 0
    out = torch.empty_like(inp.q)
    ew = torch.zeros(1, dtype=torch.int32, device=dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = L2Flush(dev, l2)

    def call():
        ops.paged_decode_attention_ex(inp.q, inp.k_cache, inp.v_cache, inp.block_tables,
                                      inp.context_lens, inp.scale, out=out,
                                      max_context_len=inp.max_context_len, partition_size=P,
                                      variant=variant, prefetch_distance=args.prefetch_distance,
                                      workspace=ws, error_word=ew, stream=stream)

    def oracle_ref(threads):
        import oracle
        return oracle.attention(inp.q.cpu(), inp.k_cache.cpu(), inp.v_cache.cpu(), inp.block_tables.cpu(),
                                inp.context_lens.cpu(), inp.scale, threads=threads)

    if kv_fp8:
        # E4M3 caches (one byte per element): the K/V stream halves
        g = torch.Generator(device=dev).manual_seed(cfg.seed + 9)
        codes = getattr(args, "e4m3_codes", "full")
        k8 = workloads.rand_e4m3(inp.k_cache.shape, g, dev, codes=codes)
        v8 = workloads.rand_e4m3(inp.v_cache.shape, g, dev, codes=codes)
        ks, vs = workloads.E4M3_SCALES[codes]
        kv16 = 2 * sum(lens) * inp.num_kv_heads * inp.head_dim * 2
        algo -= kv16 // 2
        qm = inp.q
        if q_len > 1:
            qm = workloads.randn_f16((inp.num_seqs, q_len, inp.num_q_heads, inp.head_dim), g, dev)
            algo += (q_len - 1) * 2 * inp.num_seqs * inp.num_q_heads * inp.head_dim * 2
        out = torch.empty_like(qm)
        need = ops.paged_decode_multi_workspace_size(inp.num_seqs, q_len, inp.num_q_heads, inp.num_kv_heads,
                                                     inp.head_dim, inp.block_size, inp.max_context_len, P)
        ws = ops.alloc_workspace(need, dev)

        def call():  # noqa: F811
            ops.paged_decode_attention_fp8(qm, k8, v8, inp.block_tables, inp.context_lens, inp.scale,
                                           ks, vs, out=out, max_context_len=inp.max_context_len,
                                           partition_size=P, workspace=ws, error_word=ew, stream=stream,
                                           variant=None if variant == "auto" else variant)

        def oracle_ref(threads):  # noqa: F811
            import oracle
            return oracle.attention_fp8(qm.cpu(), k8.cpu(), v8.cpu(), inp.block_tables.cpu(),
                                        inp.context_lens.cpu(), inp.scale, ks, vs, threads=threads)
    elif q_len > 1:
        # q_len new tokens per sequence (causal among them): the K/V stream is
        # the same, q and out grow by q_len
        g = torch.Generator(device=dev).manual_seed(cfg.seed + 5)
        qm = workloads.randn_f16((inp.num_seqs, q_len, inp.num_q_heads, inp.head_dim), g, dev)
        out = torch.empty_like(qm)
        algo += (q_len - 1) * 2 * inp.num_seqs * inp.num_q_heads * inp.head_dim * 2
        need = ops.paged_decode_multi_workspace_size(inp.num_seqs, q_len, inp.num_q_heads, inp.num_kv_heads,
                                                     inp.head_dim, inp.block_size, inp.max_context_len, P)
        ws = ops.alloc_workspace(need, dev)

        def call():  # noqa: F811
            ops.paged_decode_attention_multi(qm, inp.k_cache, inp.v_cache, inp.block_tables,
                                             inp.context_lens, inp.scale, out=out,
                                             max_context_len=inp.max_context_len, partition_size=P,
                                             workspace=ws, error_word=ew, stream=stream, variant=variant)

        def oracle_ref(threads):  # noqa: F811
            import oracle
            return oracle.attention_multi(qm.cpu(), inp.k_cache.cpu(), inp.v_cache.cpu(), inp.block_tables.cpu(),
                                          inp.context_lens.cpu(), inp.scale, threads=threads)

    use_flush = algo < 4 * l2

    def maybe_flush():
        if use_flush:
            flush()

    for _ in range(warmup):
        maybe_flush()
        call()
    torch.cuda.synchronize(dev)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    sampler = ClockSampler(dev.index or 0) if with_clocks else None
    if sampler:
        sampler.__enter__()
    if torch.distributed.is_initialized():
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    t_wall = time.perf_counter()
    torch.cuda.nvtx.range_push("timed")
    for i in range(steps):
        maybe_flush()
        starts[i].record(stream)
        call()
        ends[i].record(stream)
    torch.cuda.synchronize(dev)
    torch.cuda.nvtx.range_pop()
    t_wall = time.perf_counter() - t_wall
    if sampler:
        sampler.__exit__(None, None, None)
    times_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    errbits = ops.pkd_read_device_error(ew)
    res = {
        "algo_bytes": algo, "mean_ms": statistics.mean(times_ms), "median_ms": statistics.median(times_ms),
        "min_ms": min(times_ms), "wall_s": t_wall, "launches_per_call": launches, "grid": grid,
        "partition_size": eff_P if split else -1, "longest_first": ordered, "device_error": errbits,
        # the L2 prefetch distance the call ran: -1 asks for none, 0 for the model's default
        "prefetch_distance": 0 if args.prefetch_distance < 0 else (args.prefetch_distance or pdist),
        "variant": resolved, "out": out, "oracle_ref": oracle_ref,
        "clocks": sampler.summary() if sampler else None,
        "l2": (f"an L2 flush (2x L2 read) before every timed call; inputs {algo / 1e6:.0f} MB" if use_flush
               else f"inputs larger than L2 ({algo / 1e9:.2f} GB against {l2 / 1e6:.0f} MB): calls back to "
                    "back, no flush"),
    }
    if with_e2e:
        e2e_steps = max(10, min(20, steps // 10))
        if variant == "auto" and q_len == 1 and not kv_fp8 and P == 0:
            res["e2e"] = time_e2e_host_api(inp, stream, dev, algo, e2e_steps)
        else:
            res["e2e"] = time_e2e(call, inp, out, stream, dev, algo, e2e_steps)
    return res


def time_append(cfg, inp, dev, steps, warmup, peak):
    """The cache write before a decode step: paged_kv_append of token L-1 of
    every sequence (its slot exists), timed alone and followed by the decode
    call over the L tokens, each with an L2 flush before the timed region."""
    from paged_kv_decode_21_gb300 import ops
    stream = torch.cuda.current_stream(dev)
    B, Hkv, D = inp.num_seqs, inp.num_kv_heads, inp.head_dim
    g = torch.Generator(device=dev).manual_seed(cfg.seed + 99)
    k_new = workloads.randn_f16((B, Hkv, D), g, dev)
    v_new = workloads.randn_f16((B, Hkv, D), g, dev)
    pos = (inp.context_lens - 1).clamp(min=0)
    out = torch.empty_like(inp.q)
    ew = torch.zeros(1, dtype=torch.int32, device=dev)
    need = ops.paged_decode_workspace_size(B, inp.num_q_heads, Hkv, D, inp.block_size,
                                           inp.max_context_len, 0, 0)
    ws = ops.alloc_workspace(need, dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = L2Flush(dev, l2)

    def append():
        ops.paged_kv_append(k_new, v_new, inp.block_tables, pos, inp.k_cache, inp.v_cache,
                            error_word=ew, stream=stream)

    def decode():
        ops.paged_decode_attention_ex(inp.q, inp.k_cache, inp.v_cache, inp.block_tables,
                                      inp.context_lens, inp.scale, out=out,
                                      max_context_len=inp.max_context_len, workspace=ws,
                                      error_word=ew, stream=stream)

    def both():
        append()
        decode()

    def timed(fn):
        for _ in range(warmup):
            flush()
            fn()
        torch.cuda.synchronize(dev)
        st = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        en = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        for i in range(steps):
            flush()
            st[i].record(stream)
            fn()
            en[i].record(stream)
        torch.cuda.synchronize(dev)
        return statistics.mean(a.elapsed_time(b) for a, b in zip(st, en)) * 1e3

    n = min(steps, 500)
    steps = n
    t_app = timed(append)
    t_dec = timed(decode)
    t_both = timed(both)
    # algorithmic bytes of the append: new K and V rows read once, written once
    app_bytes = 2 * 2 * B * Hkv * D * 2
    return {"mode": "paged_kv_append", "workload": describe(cfg), "steps": n,
            "append_us": round(t_app, 3), "append_bytes": app_bytes,
            "append_GB_s": round(app_bytes / (t_app * 1e-6) / 1e9, 1),
            "append_frac_of_peak": round(app_bytes / (t_app * 1e-6) / 1e9 / peak, 4),
            "decode_us": round(t_dec, 2), "append_then_decode_us": round(t_both, 2),
            "device_error": ops.pkd_read_device_error(ew),
            "l2": "an L2 flush (2x L2 read) before every timed call"}


def time_e2e_host_api(inp, stream, dev, algo, steps):
    """The library's host-buffer call, paged_decode_attention_host: every step
    copies q, the tables and lengths to the device, reads the cache blocks the
    tables reference from pinned host memory (a gather over the host link),
    decodes, and copies the output back.  Events bracket the whole call."""
    from paged_kv_decode_21_gb300 import ops
    names = ["q", "k_cache", "v_cache", "block_tables", "context_lens"]
    host = {n: getattr(inp, n).cpu().pin_memory() for n in names}
    out_h = torch.empty(inp.q.shape, dtype=inp.q.dtype).pin_memory()
    need = ops.paged_decode_workspace_size(inp.num_seqs, inp.num_q_heads, inp.num_kv_heads, inp.head_dim,
                                           inp.block_size, inp.max_context_len, 0, "auto")
    ws = ops.alloc_workspace(need, dev)
    lens = host["context_lens"].tolist()
    used_blocks = sum(-(-max(L, 0) // inp.block_size) for L in lens)
    block_bytes = inp.num_kv_heads * inp.block_size * inp.head_dim * 2
    h2d = (host["q"].numel() * 2 + host["block_tables"].numel() * 4 + host["context_lens"].numel() * 4
           + 2 * used_blocks * block_bytes)
    d2h = out_h.numel() * out_h.element_size()
    devbuf = types.SimpleNamespace(q=inp.q, k_cache=inp.k_cache, v_cache=inp.v_cache, block_tables=inp.block_tables,
                                   context_lens=inp.context_lens, out=torch.empty_like(inp.q))

    def call():
        ops.paged_decode_attention_host(host["q"], host["k_cache"], host["v_cache"], host["block_tables"],
                                        host["context_lens"], out_h, devbuf, inp.scale,
                                        max_context_len=inp.max_context_len, used_blocks_only=True,
                                        workspace=ws, stream=stream)

    st = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    en = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    # the host link itself, right before the timed steps: a pinned 512 MiB copy to the device,
    # best of three (what any host-buffer call on this machine can reach)
    probe_h = torch.empty(512 << 20, dtype=torch.uint8).pin_memory()
    probe_d = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    link = []
    for _ in range(3):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        probe_d.copy_(probe_h, non_blocking=True)
        b.record(stream)
        torch.cuda.synchronize(dev)
        link.append(probe_h.numel() / (a.elapsed_time(b) * 1e-3) / 1e9)
    del probe_h, probe_d
    # warm-up calls (their times are recorded below); the timed steps follow them
    warm = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(3)]
    for a, b in warm:
        a.record(stream)
        call()
        b.record(stream)
    torch.cuda.synchronize(dev)
    for i in range(steps):
        st[i].record(stream)
        call()
        en[i].record(stream)
    torch.cuda.synchronize(dev)
    ms = statistics.mean(s.elapsed_time(e) for s, e in zip(st, en))
    return {"value": round(algo / (ms * 1e-3) / 1e9, 2), "unit": "GB/s", "ms_per_step": round(ms, 4),
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "warmup_ms": [round(a.elapsed_time(b), 3) for a, b in warm],
            "h2d_link_gbs": round(max(link), 1),
            "host_numa_node": host_numa_node(dev),
            "api": "paged_decode_attention_host (used blocks only)"}


def host_numa_node(dev):
    """The host NUMA node the driver reports closest to the GPU
    (cudaDevAttrHostNumaId), or None where it cannot be read."""
    try:
        import ctypes
        import glob
        libs = sorted(glob.glob("/usr/local/cuda/lib64/libcudart.so*"))
        if not libs:
            return None
        rt = ctypes.CDLL(libs[0])
        v = ctypes.c_int(-1)
        if rt.cudaDeviceGetAttribute(ctypes.byref(v), 134, int(dev.index or 0)) != 0:  # cudaDevAttrHostNumaId
            return None
        return v.value
    except Exception:
        return None


def time_e2e(call, inp, out, stream, dev, algo, steps):
    """Same call with the inputs copied from pinned host memory every step and
    the result copied back; events bracket copies + call."""
    names = ["q", "k_cache", "v_cache", "block_tables", "context_lens"]
    host = {n: getattr(inp, n).cpu().pin_memory() for n in names}
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = out.numel() * out.element_size()
    st = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    en = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for i in range(steps + 1):
        if i > 0:
            st[i - 1].record(stream)
        for n in names:
            getattr(inp, n).copy_(host[n], non_blocking=True)
        call()
        out_h.copy_(out, non_blocking=True)
        if i > 0:
            en[i - 1].record(stream)
    torch.cuda.synchronize(dev)
    ms = statistics.mean(s.elapsed_time(e) for s, e in zip(st, en))
    return {"value": round(algo / (ms * 1e-3) / 1e9, 2), "unit": "GB/s", "ms_per_step": round(ms, 4),
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps}


def cpu_oracle_rate(inp, target_s=10.0, max_passes=50):
    """The oracle, as it stands, on the host cores: passes over the whole
    workload until about target_s seconds; returns (GB/s, cores, sample)."""
    import oracle
    cores = os.cpu_count() or 1
    cpu = inp.to("cpu")
    lens = cpu.context_lens.tolist()
    algo = traffic.algorithmic_bytes(lens, cpu.num_q_heads, cpu.num_kv_heads, cpu.head_dim)
    passes, t, ref = 0, 0.0, None
    while passes < max_passes and (t < target_s or passes == 0):
        t0 = time.perf_counter()
        ref = oracle.attention(cpu.q, cpu.k_cache, cpu.v_cache, cpu.block_tables, cpu.context_lens, cpu.scale,
                               threads=cores)
        t += time.perf_counter() - t0
        passes += 1
    sample = f"{passes} full pass(es) over the workload ({algo / 1e9:.3f} GB each), {t:.1f} s"
    return algo * passes / t / 1e9, cores, sample, t / passes, ref


def cpu_oracle_rate_1thread(inp, nseq=4):
    """The oracle on one host thread, over all query rows of the first `nseq`
    sequences (a bounded sample of the same workload); returns (GB/s, sample)."""
    import oracle
    cpu = inp.to("cpu")
    nseq = max(1, min(nseq, cpu.num_seqs))
    lens = cpu.context_lens.tolist()[:nseq]
    algo = traffic.algorithmic_bytes(lens, cpu.num_q_heads, cpu.num_kv_heads, cpu.head_dim)
    rows = [b * cpu.num_q_heads + h for b in range(nseq) for h in range(cpu.num_q_heads)]
    t0 = time.perf_counter()
    oracle.attention(cpu.q, cpu.k_cache, cpu.v_cache, cpu.block_tables, cpu.context_lens, cpu.scale,
                     rows=rows, threads=1)
    t = time.perf_counter() - t0
    return algo / t / 1e9, f"all query rows of {nseq} sequences ({algo / 1e6:.1f} MB) on 1 thread, {t:.2f} s"


def make_workload(name, dev, batch=None):
    import dataclasses
    cfg = workloads.CONFIGS[name]
    if batch is not None and batch != cfg.num_seqs:
        lens = None if cfg.context_lens is None else tuple(cfg.context_lens[:1]) * batch
        cfg = dataclasses.replace(cfg, name=f"{cfg.name}_b{batch}", num_seqs=batch, context_lens=lens)
    return cfg, workloads.make_inputs(cfg, device=dev)


def time_extra_config(args, name, dev, peak):
    """One more large workload timed like the headline one (its configured
    partition, L2 rule and clock sampling; no e2e leg), with every output row
    compared with the oracle."""
    import copy
    cfg, inp = make_workload(name, dev)
    a = copy.copy(args)
    a.partition_size = None
    r = time_gpu(a, cfg, args.variant, dev, inp, min(args.steps, 200), args.warmup, with_e2e=False)
    gbs = r["algo_bytes"] / (r["mean_ms"] * 1e-3) / 1e9
    par = parity(r["out"], r["oracle_ref"](os.cpu_count() or 1))
    res = {"workload": describe(cfg), "variant": r["variant"], "partition_size": r["partition_size"],
           "longest_first": r["longest_first"],
           "us_per_call": round(r["mean_ms"] * 1e3, 2), "us_per_call_median": round(r["median_ms"] * 1e3, 2),
           "us_per_call_min": round(r["min_ms"] * 1e3, 2), "steps": min(args.steps, 200),
           "algorithmic_bytes_per_call": r["algo_bytes"], "GB_s": round(gbs, 1),
           "frac": round(gbs / peak, 4), "frac_of_nominal": round(gbs / NOMINAL_HBM_GBS, 4),
           "kernel": kernel_name(cfg, r["variant"], False, wide=False),
           "gpu_launches_per_call": r["launches_per_call"], "l2": r["l2"], "clocks": r["clocks"],
           "device_error_bits": r["device_error"], "parity": par}
    del inp, r
    torch.cuda.empty_cache()
    return res


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    cfg = workloads.CONFIGS[args.config]
    inp = workloads.make_inputs(cfg, device="cuda" if torch.cuda.is_available() else "cpu")
    import oracle
    cores = os.cpu_count() or 1
    cpu = inp.to("cpu")
    lens = cpu.context_lens.tolist()
    algo = traffic.algorithmic_bytes(lens, cpu.num_q_heads, cpu.num_kv_heads, cpu.head_dim)
    for _ in range(args.warmup):
        oracle.attention(cpu.q, cpu.k_cache, cpu.v_cache, cpu.block_tables, cpu.context_lens, cpu.scale,
                         threads=cores)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.attention(cpu.q, cpu.k_cache, cpu.v_cache, cpu.block_tables, cpu.context_lens, cpu.scale,
                         threads=cores)
        times.append(time.perf_counter() - t0)
    dt = statistics.mean(times)
    value = algo / dt / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "GB/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        # the same keys as the GPU arm's config: the same workload, run by the oracle
        "config": {"workload": describe(cfg), "variant": "oracle", "partition_size": -1,
                   "us_per_call": round(dt * 1e6, 2), "us_per_call_median": round(statistics.median(times) * 1e6, 2),
                   "us_per_call_min": round(min(times) * 1e6, 2), "algorithmic_bytes_per_call": algo,
                   "l2": "CPU fp64 oracle (plain C, pthreads): host memory, no GPU L2",
                   "parallelism": f"host threads x{cores} (no collective)"},
        "cpu_baseline": {"value": round(value, 3), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": f"each step is one full pass over the workload ({algo / 1e9:.3f} GB)"},
        "e2e": {"value": round(value, 3), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default=DEFAULT_CONFIG, choices=list(workloads.CONFIGS))
    ap.add_argument("--variant", default="auto",
                    help="auto|no_prefetch|l2_prefetch|tma_staged|tma_mma, optionally +l2_hints "
                         "(L2 eviction priorities)")
    ap.add_argument("--partition-size", type=int, default=None)
    ap.add_argument("--prefetch-distance", type=int, default=0,
                    help="L2 prefetch distance: -1 none, 0 the library's model (default), >= 1 that distance")
    ap.add_argument("--sweep", action="store_true", help="every workload x variant, one line each")
    ap.add_argument("--sweep-configs", default=",".join(workloads.CONFIG_ORDER[1:]))
    ap.add_argument("--sweep-variants", default="no_prefetch,l2_prefetch,tma_staged")
    ap.add_argument("--sweep-partitions", default="", help="comma list of partition sizes (default: the config's)")
    ap.add_argument("--sweep-pd", default="",
                    help="comma list of prefetch distances (-1 none, 0 the library's model; default: the model)")
    ap.add_argument("--fig4", action="store_true",
                    help="batch x context grid on the MHA shape: each data path's speed over NO_PREFETCH")
    ap.add_argument("--fig4-config", default=DEFAULT_CONFIG,
                    help="workload whose head shape the grid uses (batch and context are swept)")
    ap.add_argument("--fig4-variants", default="no_prefetch,l2_prefetch,tma_staged,tma_mma,auto")
    ap.add_argument("--fig4-batches", default="1,4,16,64,128,256")
    ap.add_argument("--fig4-contexts", default="512,1024,2048,4096,8192")
    ap.add_argument("--fig4-ragged", action="store_true",
                    help="per-sequence contexts drawn from U[context/8, context] (seeded) instead of all equal")
    ap.add_argument("--split-sweep", action="store_true",
                    help="small grids: the automatic split against every partition of --split-partitions, "
                         "over --split-batches x --split-contexts of --config's heads (--q-len, --kv-fp8, "
                         "--variant and --fig4-ragged apply); one line per batch x context")
    ap.add_argument("--split-batches", default="1,4,16")
    ap.add_argument("--split-contexts", default="2048,8192")
    ap.add_argument("--split-partitions", default="128,256,512,1024,2048,4096")
    ap.add_argument("--append", action="store_true",
                    help="time paged_kv_append alone and in front of the decode call, on --config")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-parity", action="store_true",
                    help="skip the all-row comparison of the timed call's output with the oracle")
    ap.add_argument("--no-extra-configs", action="store_true",
                    help="time only --config (the default run also times and checks the other large workloads)")
    ap.add_argument("--e4m3-codes", default="full", choices=sorted(workloads.E4M3_SCALES),
                    help="code set of the E4M3 caches of --kv-fp8 (and its per-cache scales)")
    ap.add_argument("--batch", type=int, default=None, help="override the workload's batch (profiling runs)")
    ap.add_argument("--kv-fp8", action="store_true",
                    help="E4M3 K/V caches (one byte per element, per-cache scales)")
    ap.add_argument("--q-len", type=int, default=1,
                    help="query tokens per sequence (> 1: multi-token queries, causal among them)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    if args.impl == "reference":
        return run_reference(args)

    ws, rank, local = dist_env()
    if ws > 1:
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    from paged_kv_decode_21_gb300 import build as pkd_build
    from paged_kv_decode_21_gb300 import ops
    if rank == 0 or ws == 1:
        pkd_build.build()
    if ws > 1:
        torch.distributed.barrier()
    ops.lib()
    peak, peak_kind = hbm_peak()

    if args.fig4:
        import dataclasses
        base = workloads.CONFIGS[args.fig4_config]
        for L in [int(x) for x in args.fig4_contexts.split(",")]:
            for B in [int(x) for x in args.fig4_batches.split(",")]:
                if args.fig4_ragged:
                    cfg = dataclasses.replace(base, name=f"{base.name}_b{B}_L{L}r", num_seqs=B,
                                              context_lens=None, len_range=(max(1, L // 8), L),
                                              num_blocks=None, partition_size=0)
                else:
                    cfg = dataclasses.replace(base, name=f"{base.name}_b{B}_L{L}", num_seqs=B,
                                              context_lens=(L,) * B, len_range=None, num_blocks=None,
                                              partition_size=0)
                inp = workloads.make_inputs(cfg, device=dev)
                res = {}
                for variant in ["no_prefetch"] + [v for v in args.fig4_variants.split(",")
                                                  if v and v != "no_prefetch"]:
                    args.partition_size = None
                    r = time_gpu(args, cfg, variant, dev, inp, min(args.steps, 50), args.warmup,
                                 with_e2e=False, with_clocks=False)
                    res[variant] = r
                base_us = res["no_prefetch"]["mean_ms"] * 1e3
                line = {"shape": f"{cfg.num_q_heads}q/{cfg.num_kv_heads}kv", "batch": B, "context": L,
                        "ragged": bool(args.fig4_ragged),
                        "algo_bytes": res["auto"]["algo_bytes"],
                        "partition_size": res["auto"]["partition_size"],
                        "longest_first": res["auto"]["longest_first"],
                        "auto_variant": ops.variant_name(ops.paged_decode_auto_variant(
                            B, cfg.num_q_heads, cfg.num_kv_heads, cfg.head_dim, cfg.block_size,
                            inp.max_context_len, cfg.partition_size or 0))}
                for variant, r in res.items():
                    us = r["mean_ms"] * 1e3
                    gbs = r["algo_bytes"] / (r["mean_ms"] * 1e-3) / 1e9
                    line[variant] = {"us": round(us, 2), "frac_of_peak": round(gbs / peak, 4),
                                     "speedup_vs_no_prefetch": round(base_us / us, 3)}
                print(json.dumps(line), flush=True)
                del inp
                torch.cuda.empty_cache()
        return 0

    if args.split_sweep:
        import dataclasses
        base = workloads.CONFIGS[args.config]
        parts = [int(x) for x in args.split_partitions.split(",") if x.strip()]
        for L in [int(x) for x in args.split_contexts.split(",")]:
            for B in [int(x) for x in args.split_batches.split(",")]:
                if args.fig4_ragged:
                    cfg = dataclasses.replace(base, name=f"{base.name}_b{B}_L{L}r", num_seqs=B, context_lens=None,
                                              len_range=(max(1, L // 8), L), num_blocks=None, partition_size=0)
                else:
                    cfg = dataclasses.replace(base, name=f"{base.name}_b{B}_L{L}", num_seqs=B,
                                              context_lens=(L,) * B, len_range=None, num_blocks=None,
                                              partition_size=0)
                inp = workloads.make_inputs(cfg, device=dev)
                res = {}
                # the automatic split last, so that it is not the first call timed on fresh inputs
                for P in [-1] + [p for p in parts if p < inp.max_context_len] + [0]:
                    args.partition_size = P
                    r = time_gpu(args, cfg, args.variant, dev, inp, min(args.steps, 50), args.warmup,
                                 with_e2e=False, with_clocks=False)
                    res[P] = r
                us = {str(P): round(r["median_ms"] * 1e3, 2) for P, r in res.items()}
                best = min(us, key=us.get)
                print(json.dumps({"shape": f"{cfg.num_q_heads}q/{cfg.num_kv_heads}kv", "batch": B, "context": L,
                                  "ragged": bool(args.fig4_ragged), "q_len": args.q_len, "kv_fp8": bool(args.kv_fp8),
                                  "automatic": {"partition_size": res[0]["partition_size"],
                                                "variant": res[0]["variant"], "grid": res[0]["grid"]},
                                  "us_median": us, "best": best, "automatic_over_best": round(us["0"] / us[best], 3)}),
                      flush=True)
                del inp, res
                torch.cuda.empty_cache()
        return 0

    if args.append:
        cfg, inp = make_workload(args.config, dev, args.batch)
        print(json.dumps(time_append(cfg, inp, dev, args.steps, args.warmup, peak)), flush=True)
        return 0

    if args.sweep:
        parts = [int(x) for x in args.sweep_partitions.split(",") if x.strip()] or [None]
        pds = [int(x) for x in args.sweep_pd.split(",") if x.strip()] or [args.prefetch_distance]
        combos = [(p_, d_) for p_ in parts for d_ in pds]
        for name in args.sweep_configs.split(","):
            cfg, inp = make_workload(name, dev, args.batch)
            for variant in args.sweep_variants.split(","):
                for part, pdist in combos:
                    args.partition_size = part
                    args.prefetch_distance = pdist
                    r = time_gpu(args, cfg, variant, dev, inp, min(args.steps, 200), args.warmup,
                                 with_e2e=False, with_clocks=False)
                    gbs = r["algo_bytes"] / (r["mean_ms"] * 1e-3) / 1e9
                    print(json.dumps({"workload": name, "variant": variant,
                                      "us_per_call": round(r["mean_ms"] * 1e3, 2),
                                      "us_min": round(r["min_ms"] * 1e3, 2), "GB_s": round(gbs, 1),
                                      "frac_of_peak": round(gbs / peak, 4),
                                      "partition_size": r["partition_size"],
                                      "prefetch_distance": r["prefetch_distance"],
                                      "prefetch_requested": pdist if pdist else "model",
                                      "launches_per_call": r["launches_per_call"],
                                      "device_error": r["device_error"]}), flush=True)
            del inp
            torch.cuda.empty_cache()
        return 0

    cfg, inp = make_workload(args.config, dev, args.batch)
    variant = args.variant
    r = time_gpu(args, cfg, variant, dev, inp, args.steps, args.warmup, with_e2e=not args.no_e2e)
    mean_ms, value = aggregate_over_ranks(r["mean_ms"], r["algo_bytes"], ws, dev)
    achieved = r["algo_bytes"] / (r["mean_ms"] * 1e-3) / 1e9
    resolved = r["variant"]
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(mean_ms, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": dtype_label(resolved, args.kv_fp8),
        "data": "synthetic",
        "config": {"workload": describe(cfg) + (f", q_len={args.q_len} (causal)" if args.q_len > 1 else "")
                   + (", KV in E4M3 (1 byte/element)" if args.kv_fp8 else ""),
                   "variant": resolved,
                   "partition_size": r["partition_size"],
                   "prefetch_distance": r["prefetch_distance"],
                   "us_per_call": round(mean_ms * 1e3, 2), "us_per_call_median": round(r["median_ms"] * 1e3, 2),
                   "us_per_call_min": round(r["min_ms"] * 1e3, 2),
                   "algorithmic_bytes_per_call": r["algo_bytes"],
                   "l2": r["l2"],
                   "parallelism": f"replicas x{ws} (no collective)"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_kind": peak_kind,
                     "frac_of_nominal": round(achieved / NOMINAL_HBM_GBS, 4), "nominal_peak": NOMINAL_HBM_GBS,
                     "traffic": ncu_traffic(cfg.name, resolved),
                     "kernel": kernel_name(cfg, resolved, args.kv_fp8,
                                           wide=args.q_len == 1 and r["grid"] >= 3 * 4 * torch.cuda.get_device_properties(dev).multi_processor_count,
                                           q_len=args.q_len)},
        "gpu_launches": r["launches_per_call"] * args.steps,
        "clocks": r["clocks"],
        "e2e": r.get("e2e"),
        "device_error_bits": r["device_error"],
    }
    cpu_ref = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline and args.q_len == 1 and not args.kv_fp8:
        v, cores, sample, _, cpu_ref = cpu_oracle_rate(inp)
        v1, sample1 = cpu_oracle_rate_1thread(inp)
        line["cpu_baseline"] = {"value": round(v, 3), "unit": "GB/s", "cores": cores, "kind": "oracle",
                                "value_1_thread": round(v1, 3), "sample_1_thread": sample1,
                                "sample": sample}
    ok = True
    if not args.no_parity:
        # every output element of the last timed call against the oracle (each rank checks its own)
        ref = cpu_ref if cpu_ref is not None else r["oracle_ref"](os.cpu_count() or 1)
        line["parity"] = parity(r["out"], ref)
        ok = line["parity"]["ok"]
        del ref, cpu_ref
    del r, inp
    torch.cuda.empty_cache()
    if (rank == 0 and ws == 1 and args.config == DEFAULT_CONFIG and args.batch is None and args.q_len == 1
            and not args.kv_fp8 and not args.no_extra_configs):
        line["other_configs"] = {}
        for name in EXTRA_CONFIGS:
            extra = time_extra_config(args, name, dev, peak)
            line["other_configs"][name] = extra
            ok = ok and extra["parity"]["ok"] and extra["device_error_bits"] == 0
    ok = ok and line["device_error_bits"] == 0
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    if not ok:
        sys.stderr.write("bench: parity or device-error check failed (see the line's parity keys)\n")
        return 1
    return 0


if __name__ == "__main__":
    sys.exit(main())
