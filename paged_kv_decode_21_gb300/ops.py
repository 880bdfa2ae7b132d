"""ctypes binding of libpaged_decode.so (argument marshalling only).

Every function here has the name of the C entry point it calls (see
``include/paged_decode.h``) and takes torch tensors for device buffers; the
work itself runs in the library's CUDA kernels on the current (or given)
stream.  There is no fallback: if the library is missing, loading fails.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpaged_decode.so")

PKD_OK = 0
STATUS_NAMES = {0: "PKD_OK", 1: "PKD_ERR_NULL", 2: "PKD_ERR_SHAPE", 3: "PKD_ERR_UNSUPPORTED",
                4: "PKD_ERR_ALIGN", 5: "PKD_ERR_WORKSPACE", 6: "PKD_ERR_LAUNCH",
                7: "PKD_ERR_DEVICE", 8: "PKD_ERR_CUDA"}
VARIANTS = {"auto": 0, "no_prefetch": 1, "l2_prefetch": 2, "tma_staged": 3, "tma_mma": 4, "tcgen05": 5}
DEVERR_BAD_BLOCK = 1
DEVERR_TIMEOUT = 2
DEVERR_LAYOUT = 4

_lock = threading.Lock()
_lib = None


class PagedDecodeError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        msg = lib().pkd_status_string(status).decode()
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)} ({msg})")


def lib():
    """The loaded library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m paged_kv_decode_21_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        P, I, F, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        attn = [P, P, P, P, P, P, I, I, I, I, I, I, I, I, F]
        L.paged_decode_attention.argtypes = attn + [P]
        L.paged_decode_attention.restype = I
        L.paged_decode_attention_ex.argtypes = attn + [I, I, I, P, S, P, P]
        L.paged_decode_attention_ex.restype = I
        L.paged_decode_auto_partition_size.argtypes = [I, I, I, I, I, I, I]
        L.paged_decode_auto_partition_size.restype = I
        L.paged_decode_auto_variant.argtypes = [I, I, I, I, I, I, I]
        L.paged_decode_auto_variant.restype = I
        L.paged_decode_workspace_size.argtypes = [I, I, I, I, I, I, I, I]
        L.paged_decode_workspace_size.restype = S
        L.paged_decode_partitions.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, I, F, I, I, I,
                                              P, P, P, I, P, P]
        L.paged_decode_partitions.restype = I
        L.paged_decode_reduce.argtypes = [P, P, P, P, P, I, I, I, I, I, I, P]
        L.paged_decode_reduce.restype = I
        L.paged_decode_validate_tables.argtypes = [P, P, I, I, I, I, P, P]
        L.paged_decode_validate_tables.restype = I
        L.paged_decode_attention_multi.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, I, I, I, F, I, P, S,
                                                   P, P]
        L.paged_decode_attention_multi.restype = I
        L.paged_decode_attention_multi_ex.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, I, I, I, F, I, I, P, S,
                                                      P, P]
        L.paged_decode_attention_multi_ex.restype = I
        L.paged_decode_call_plan.argtypes = [I] * 10 + [ctypes.POINTER(ctypes.c_int)] * 3 + [
            ctypes.POINTER(ctypes.c_longlong), ctypes.POINTER(ctypes.c_int)]
        L.paged_decode_call_plan.restype = I
        LLP = ctypes.POINTER(ctypes.c_longlong)
        D_ = ctypes.c_double
        L.pkd_l2_prefetch_model.argtypes = [ctypes.c_longlong, I, I, ctypes.c_longlong, I, ctypes.c_longlong,
                                            ctypes.c_longlong, D_, D_, D_, I, LLP, LLP, LLP]
        L.pkd_l2_prefetch_model.restype = I
        L.paged_decode_prefetch_model.argtypes = [I] * 11 + [ctypes.c_longlong, D_, LLP, LLP, LLP]
        L.paged_decode_prefetch_model.restype = I
        L.paged_decode_attention_host.argtypes = [P] * 12 + [I] * 8 + [F, I, P, S, P, P]
        L.paged_decode_attention_host.restype = I
        L.paged_decode_auto_plan.argtypes = [I, I, I, I, I, I, I, I, ctypes.POINTER(ctypes.c_int),
                                             ctypes.POINTER(ctypes.c_int)]
        L.paged_decode_auto_plan.restype = I
        L.paged_decode_multi_workspace_size.argtypes = [I, I, I, I, I, I, I, I]
        L.paged_decode_multi_workspace_size.restype = S
        L.paged_decode_attention_fp8.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, I, I, I, F, F, F, I, P, S,
                                                 P, P]
        L.paged_decode_attention_fp8.restype = I
        L.paged_decode_attention_fp8_ex.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, I, I, I, F, F, F, I, I, P,
                                                    S, P, P]
        L.paged_decode_attention_fp8_ex.restype = I
        L.paged_kv_append_fp8.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, F, F, P, P]
        L.paged_kv_append_fp8.restype = I
        L.paged_kv_append.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, P, P]
        L.paged_kv_append.restype = I
        L.pkd_selftest_bounded_wait.argtypes = [P, ctypes.c_ulonglong, P]
        L.pkd_selftest_bounded_wait.restype = I
        L.pkd_read_device_error.argtypes = [P, ctypes.POINTER(ctypes.c_uint), I, P]
        L.pkd_read_device_error.restype = I
        L.paged_decode_attention_static_scratch.argtypes = attn + [I, I, I, P, P]
        L.paged_decode_attention_static_scratch.restype = I
        L.pkd_status_string.argtypes = [I]
        L.pkd_status_string.restype = ctypes.c_char_p
        L.pkd_version.argtypes = []
        L.pkd_version.restype = I
        _lib = L
        return L


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _check(status: int, what: str):
    if status != PKD_OK:
        raise PagedDecodeError(status, what)


def _want(t: torch.Tensor, name: str, dtype, dim=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dim is not None and t.dim() != dim:
        raise ValueError(f"{name} must have {dim} dimensions")


def _shape(q, k_cache, v_cache, block_tables, context_lens):
    _want(q, "q", torch.float16, 3)
    _want(k_cache, "k_cache", torch.float16, 4)
    _want(v_cache, "v_cache", torch.float16, 4)
    _want(block_tables, "block_tables", torch.int32, 2)
    _want(context_lens, "context_lens", torch.int32, 1)
    B, Hq, D = q.shape
    NB, Hkv, BS, D2 = k_cache.shape
    if D2 != D or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("k_cache / v_cache shape mismatch")
    if block_tables.shape[0] != B or context_lens.shape[0] != B:
        raise ValueError("block_tables / context_lens batch mismatch")
    return B, Hq, Hkv, D, BS, NB, block_tables.shape[1]


def _max_len(context_lens, max_context_len):
    if max_context_len is not None:
        return int(max_context_len)
    return int(context_lens.max().item()) if context_lens.numel() else 0


def paged_decode_attention(q, k_cache, v_cache, block_tables, context_lens, scale, out=None,
                           max_context_len=None, stream=None) -> torch.Tensor:
    """Unsplit decode attention (no workspace); returns ``out``."""
    B, Hq, Hkv, D, BS, NB, MB = _shape(q, k_cache, v_cache, block_tables, context_lens)
    if out is None:
        out = torch.empty_like(q)
    _want(out, "out", torch.float16, 3)
    st = lib().paged_decode_attention(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                      _ptr(context_lens), _ptr(out), B, Hq, Hkv, D, BS, NB, MB,
                                      _max_len(context_lens, max_context_len), float(scale),
                                      _stream(stream))
    _check(st, "paged_decode_attention")
    return out


FLAG_L2_EVICT_HINTS = 0x100
FLAG_LONGEST_FIRST = 0x200


FLAGS = {"l2_hints": FLAG_L2_EVICT_HINTS, "longest_first": FLAG_LONGEST_FIRST}


def _variant(variant) -> int:
    """A data-path name ("tma_staged", optionally "+l2_hints", "+longest_first") or its integer code."""
    if isinstance(variant, str):
        name, *flags = variant.split("+")
        code = VARIANTS[name]
        for flag in flags:
            if flag not in FLAGS:
                raise ValueError(f"unknown variant flag {flag!r}")
            code |= FLAGS[flag]
        return code
    return int(variant)


def paged_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                                max_context_len, partition_size=0, variant="auto") -> int:
    return int(lib().paged_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                                 block_size, max_context_len, partition_size,
                                                 _variant(variant)))


def paged_decode_auto_partition_size(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                                     max_context_len, variant="auto") -> int:
    return int(lib().paged_decode_auto_partition_size(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                                      block_size, max_context_len, _variant(variant)))


def paged_decode_auto_variant(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                              max_context_len, partition_size=0) -> int:
    """The variant value (path | flags) that "auto" runs for this shape."""
    v = lib().paged_decode_auto_variant(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                                        max_context_len, partition_size)
    if v < 0:
        raise PagedDecodeError(2, "paged_decode_auto_variant")
    return v


def paged_decode_auto_plan(num_seqs, q_len, num_q_heads, num_kv_heads, head_dim, block_size, max_context_len,
                           kv_fp8=False):
    """What a call with partition_size 0 runs: (launches, partition or -1, longest_first)."""
    part, order = ctypes.c_int(0), ctypes.c_int(0)
    n = lib().paged_decode_auto_plan(num_seqs, q_len, num_q_heads, num_kv_heads, head_dim, block_size,
                                     max_context_len, int(bool(kv_fp8)), ctypes.byref(part), ctypes.byref(order))
    if n < 0:
        raise PagedDecodeError(2, "paged_decode_auto_plan")
    return n, part.value, bool(order.value)


def paged_decode_call_plan(num_seqs, q_len, num_q_heads, num_kv_heads, head_dim, block_size, max_context_len,
                           kv_fp8=False, partition_size=0, variant="auto"):
    """The launch plan of a call: (launches, partition or -1, longest_first,
    variant name it runs, decode CTAs, default L2 prefetch distance)."""
    part, order, var, grid = ctypes.c_int(0), ctypes.c_int(0), ctypes.c_int(0), ctypes.c_longlong(0)
    pd = ctypes.c_int(0)
    n = lib().paged_decode_call_plan(num_seqs, q_len, num_q_heads, num_kv_heads, head_dim, block_size,
                                     max_context_len, int(bool(kv_fp8)), int(partition_size), _variant(variant),
                                     ctypes.byref(part), ctypes.byref(order), ctypes.byref(var), ctypes.byref(grid),
                                     ctypes.byref(pd))
    if n < 0:
        raise PagedDecodeError(2, "paged_decode_call_plan")
    return n, part.value, bool(order.value), variant_name(var.value), grid.value, pd.value


def pkd_l2_prefetch_model(resident_ctas, sm_count, streams_per_cta, m_block, tiles_per_step, ahead_bytes_per_cta,
                          l2_bytes, l2_fraction, hbm_bytes_per_s, latency_s, max_distance):
    """The prefetch-distance rule: (distance, footprint bytes, in-flight bytes per SM, need bytes per SM)."""
    fp, inf, need = ctypes.c_longlong(0), ctypes.c_longlong(0), ctypes.c_longlong(0)
    d = lib().pkd_l2_prefetch_model(int(resident_ctas), int(sm_count), int(streams_per_cta), int(m_block),
                                    int(tiles_per_step), int(ahead_bytes_per_cta), int(l2_bytes), float(l2_fraction),
                                    float(hbm_bytes_per_s), float(latency_s), int(max_distance), ctypes.byref(fp),
                                    ctypes.byref(inf), ctypes.byref(need))
    if d < 0:
        raise PagedDecodeError(2, "pkd_l2_prefetch_model")
    return d, fp.value, inf.value, need.value


def paged_decode_prefetch_model(num_seqs, q_len, num_q_heads, num_kv_heads, head_dim, block_size, max_context_len,
                                sm_count, l2_bytes, hbm_bytes_per_s, kv_fp8=False, partition_size=0,
                                variant="auto"):
    """Default L2 prefetch distance of a call on a described GPU:
    (distance, footprint bytes, in-flight bytes per SM, need bytes per SM)."""
    fp, inf, need = ctypes.c_longlong(0), ctypes.c_longlong(0), ctypes.c_longlong(0)
    d = lib().paged_decode_prefetch_model(num_seqs, q_len, num_q_heads, num_kv_heads, head_dim, block_size,
                                          max_context_len, int(bool(kv_fp8)), int(partition_size),
                                          _variant(variant), int(sm_count), int(l2_bytes), float(hbm_bytes_per_s),
                                          ctypes.byref(fp), ctypes.byref(inf), ctypes.byref(need))
    if d < 0:
        raise PagedDecodeError(2, "paged_decode_prefetch_model")
    return d, fp.value, inf.value, need.value


def variant_name(v: int) -> str:
    """Name of a variant value, e.g. 'tma_staged+l2_hints'."""
    names = {n: k for k, n in VARIANTS.items()}
    return names[v & 0xff] + "".join("+" + f for f, bit in FLAGS.items() if v & bit)


def alloc_workspace(nbytes: int, device) -> Optional[torch.Tensor]:
    """A 256-byte aligned device buffer of at least ``nbytes`` (None for 0)."""
    if nbytes <= 0:
        return None
    buf = torch.empty(nbytes + 256, dtype=torch.uint8, device=device)
    off = (-buf.data_ptr()) % 256
    return buf[off:off + nbytes]


def paged_decode_attention_ex(q, k_cache, v_cache, block_tables, context_lens, scale, out=None,
                              max_context_len=None, partition_size=0, variant="auto",
                              prefetch_distance=0, workspace=None, error_word=None,
                              stream=None) -> torch.Tensor:
    """Decode attention with split-K and data-path control; returns ``out``.

    ``workspace`` (uint8 CUDA tensor, 256-byte aligned) is allocated here when
    None and a split is needed."""
    B, Hq, Hkv, D, BS, NB, MB = _shape(q, k_cache, v_cache, block_tables, context_lens)
    if out is None:
        out = torch.empty_like(q)
    _want(out, "out", torch.float16, 3)
    ml = _max_len(context_lens, max_context_len)
    var = _variant(variant)
    if workspace is None:
        need = paged_decode_workspace_size(B, Hq, Hkv, D, BS, ml, partition_size, var)
        workspace = alloc_workspace(need, q.device)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib().paged_decode_attention_ex(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                         _ptr(context_lens), _ptr(out), B, Hq, Hkv, D, BS, NB, MB,
                                         ml, float(scale), int(partition_size), var,
                                         int(prefetch_distance), _ptr(workspace), wbytes,
                                         _ptr(error_word), _stream(stream))
    _check(st, "paged_decode_attention_ex")
    return out


def paged_decode_attention_host(q, k_cache, v_cache, block_tables, context_lens, out, dev, scale,
                                max_context_len=None, used_blocks_only=True, workspace=None, error_word=None,
                                stream=None) -> torch.Tensor:
    """The whole operation from host tensors (page-locked for asynchronous copies): inputs are
    copied into the device tensors of ``dev`` (a DecodeInputs-like object with q, k_cache,
    v_cache, block_tables, context_lens) and ``out`` (host) receives the result once the stream
    has run.  Returns ``out``."""
    B, Hq, D = q.shape
    NB, Hkv, BS, _ = k_cache.shape
    MB = block_tables.shape[1]
    ml = int(max_context_len) if max_context_len is not None else (int(context_lens.max()) if B else 0)
    out_dev = dev.out if getattr(dev, "out", None) is not None else torch.empty_like(dev.q)
    if workspace is None:
        workspace = alloc_workspace(paged_decode_workspace_size(B, Hq, Hkv, D, BS, ml, 0, "auto"), dev.q.device)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib().paged_decode_attention_host(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), _ptr(context_lens), _ptr(out),
        _ptr(dev.q), _ptr(dev.k_cache), _ptr(dev.v_cache), _ptr(dev.block_tables), _ptr(dev.context_lens),
        _ptr(out_dev), B, Hq, Hkv, D, BS, NB, MB, ml, float(scale), int(bool(used_blocks_only)),
        _ptr(workspace), wbytes, _ptr(error_word), _stream(stream))
    _check(st, "paged_decode_attention_host")
    return out


def paged_decode_partitions(q, k_cache, v_cache, block_tables, context_lens, scale, partition_size,
                            tmp_out, max_logits, exp_sums, max_context_len=None, variant="auto",
                            prefetch_distance=0, error_word=None, stream=None):
    """First split-K kernel alone: per-partition (max_logits, exp_sums, tmp_out)."""
    B, Hq, Hkv, D, BS, NB, MB = _shape(q, k_cache, v_cache, block_tables, context_lens)
    for t, n in ((tmp_out, "tmp_out"), (max_logits, "max_logits"), (exp_sums, "exp_sums")):
        _want(t, n, torch.float32)
    npmax = max_logits.shape[-1]
    var = _variant(variant)
    st = lib().paged_decode_partitions(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                       _ptr(context_lens), B, Hq, Hkv, D, BS, NB, MB,
                                       _max_len(context_lens, max_context_len), float(scale),
                                       int(partition_size), var, int(prefetch_distance),
                                       _ptr(tmp_out), _ptr(max_logits), _ptr(exp_sums), npmax,
                                       _ptr(error_word), _stream(stream))
    _check(st, "paged_decode_partitions")


def paged_decode_reduce(tmp_out, max_logits, exp_sums, context_lens, out, partition_size,
                        min_partitions_to_merge=0, stream=None):
    """Split-K merge of per-partition statistics into ``out``."""
    B, Hq, NP, D = tmp_out.shape
    st = lib().paged_decode_reduce(_ptr(tmp_out), _ptr(max_logits), _ptr(exp_sums),
                                   _ptr(context_lens), _ptr(out), B, Hq, D, int(partition_size),
                                   NP, int(min_partitions_to_merge), _stream(stream))
    _check(st, "paged_decode_reduce")
    return out


def paged_decode_validate_tables(block_tables, context_lens, block_size, num_blocks, error_word,
                                 stream=None):
    B, MB = block_tables.shape
    st = lib().paged_decode_validate_tables(_ptr(block_tables), _ptr(context_lens), B, MB,
                                            int(block_size), int(num_blocks), _ptr(error_word),
                                            _stream(stream))
    _check(st, "paged_decode_validate_tables")


def paged_decode_multi_workspace_size(num_seqs, q_len, num_q_heads, num_kv_heads, head_dim, block_size,
                                      max_context_len, partition_size=0) -> int:
    return int(lib().paged_decode_multi_workspace_size(num_seqs, q_len, num_q_heads, num_kv_heads, head_dim,
                                                       block_size, max_context_len, partition_size))


def paged_decode_attention_multi(q, k_cache, v_cache, block_tables, context_lens, scale, out=None,
                                 max_context_len=None, partition_size=0, workspace=None,
                                 error_word=None, stream=None, variant="auto") -> torch.Tensor:
    """q_len new tokens per sequence, q [B][q_len][Hq][D]; causal among them.
    variant: "auto", "tma_mma" or "tcgen05" (paged_decode_attention_multi_ex)."""
    _want(q, "q", torch.float16, 4)
    B, QL, Hq, D = q.shape
    _, _, Hkv, _, BS, NB, MB = _shape(q.view(B, QL * Hq, D), k_cache, v_cache, block_tables, context_lens)
    if out is None:
        out = torch.empty_like(q)
    _want(out, "out", torch.float16, 4)
    maxlen = _max_len(context_lens, max_context_len)
    need = paged_decode_multi_workspace_size(B, QL, Hq, Hkv, D, BS, maxlen, partition_size)
    if workspace is None:
        workspace = alloc_workspace(need, q.device)
    wsb = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib().paged_decode_attention_multi_ex(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                               _ptr(context_lens), _ptr(out), B, QL, Hq, Hkv, D, BS, NB, MB,
                                               maxlen, float(scale), int(partition_size), _variant(variant),
                                               _ptr(workspace), wsb, _ptr(error_word), _stream(stream))
    _check(st, "paged_decode_attention_multi_ex")
    return out


def _want_fp8_cache(t: torch.Tensor, name: str):
    if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dim() != 4 or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous 4-D CUDA tensor")
    if t.element_size() != 1:
        raise ValueError(f"{name} must hold one byte per element (uint8 or float8_e4m3fn)")


def paged_decode_attention_fp8(q, k_cache, v_cache, block_tables, context_lens, scale, k_scale, v_scale,
                               out=None, max_context_len=None, partition_size=0, workspace=None,
                               error_word=None, stream=None, variant=None) -> torch.Tensor:
    """Decode over E4M3 caches (value = code * k_scale / v_scale); q is
    [B][Hq][D] (single query) or [B][q_len][Hq][D] (causal multi-token).
    With ``variant`` (auto, tma_mma, tcgen05) this calls
    paged_decode_attention_fp8_ex."""
    single = q.dim() == 3
    qm = q.unsqueeze(1) if single else q
    _want(qm, "q", torch.float16, 4)
    _want_fp8_cache(k_cache, "k_cache")
    _want_fp8_cache(v_cache, "v_cache")
    _want(block_tables, "block_tables", torch.int32, 2)
    _want(context_lens, "context_lens", torch.int32, 1)
    B, QL, Hq, D = qm.shape
    NB, Hkv, BS, D2 = k_cache.shape
    if D2 != D or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("k_cache / v_cache shape mismatch")
    if block_tables.shape[0] != B or context_lens.shape[0] != B:
        raise ValueError("block_tables / context_lens batch mismatch")
    if out is None:
        out = torch.empty_like(q)
    _want(out, "out", torch.float16, q.dim())
    maxlen = _max_len(context_lens, max_context_len)
    need = paged_decode_multi_workspace_size(B, QL, Hq, Hkv, D, BS, maxlen, partition_size)
    if workspace is None:
        workspace = alloc_workspace(need, q.device)
    wsb = 0 if workspace is None else workspace.numel() * workspace.element_size()
    if variant is None:
        st = lib().paged_decode_attention_fp8(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                              _ptr(context_lens), _ptr(out), B, QL, Hq, Hkv, D, BS, NB,
                                              block_tables.shape[1], maxlen, float(scale), float(k_scale),
                                              float(v_scale), int(partition_size), _ptr(workspace), wsb,
                                              _ptr(error_word), _stream(stream))
    else:
        st = lib().paged_decode_attention_fp8_ex(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                                 _ptr(context_lens), _ptr(out), B, QL, Hq, Hkv, D, BS, NB,
                                                 block_tables.shape[1], maxlen, float(scale), float(k_scale),
                                                 float(v_scale), int(partition_size), _variant(variant),
                                                 _ptr(workspace), wsb, _ptr(error_word), _stream(stream))
    _check(st, "paged_decode_attention_fp8")
    return out


def paged_kv_append_fp8(k_new, v_new, block_tables, context_lens, k_cache, v_cache, k_scale, v_scale,
                        error_word=None, stream=None):
    """Quantize each sequence's new K/V row (fp16 [B][Hkv][D]) to E4M3 and write it
    at logical position context_lens[b] of the byte caches, in place."""
    _want(k_new, "k_new", torch.float16, 3)
    _want(v_new, "v_new", torch.float16, 3)
    _want_fp8_cache(k_cache, "k_cache")
    _want_fp8_cache(v_cache, "v_cache")
    _want(block_tables, "block_tables", torch.int32, 2)
    _want(context_lens, "context_lens", torch.int32, 1)
    NB, Hkv, BS, D = k_cache.shape
    B = context_lens.shape[0]
    if tuple(k_new.shape) != (B, Hkv, D) or tuple(v_new.shape) != (B, Hkv, D):
        raise ValueError("k_new / v_new must be [num_seqs][num_kv_heads][head_dim]")
    st = lib().paged_kv_append_fp8(_ptr(k_new), _ptr(v_new), _ptr(block_tables), _ptr(context_lens),
                                   _ptr(k_cache), _ptr(v_cache), B, Hkv, D, BS, NB, block_tables.shape[1],
                                   float(k_scale), float(v_scale), _ptr(error_word), _stream(stream))
    _check(st, "paged_kv_append_fp8")


def paged_kv_append(k_new, v_new, block_tables, context_lens, k_cache, v_cache, error_word=None,
                    stream=None):
    """Write each sequence's new K/V row ([B][Hkv][D]) into the paged caches,
    in place, at logical position context_lens[b]."""
    _want(k_new, "k_new", torch.float16, 3)
    _want(v_new, "v_new", torch.float16, 3)
    _want(k_cache, "k_cache", torch.float16, 4)
    _want(v_cache, "v_cache", torch.float16, 4)
    _want(block_tables, "block_tables", torch.int32, 2)
    _want(context_lens, "context_lens", torch.int32, 1)
    NB, Hkv, BS, D = k_cache.shape
    B = context_lens.shape[0]
    if tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("k_cache / v_cache shape mismatch")
    if tuple(k_new.shape) != (B, Hkv, D) or tuple(v_new.shape) != (B, Hkv, D):
        raise ValueError("k_new / v_new must be [num_seqs][num_kv_heads][head_dim]")
    if block_tables.shape[0] != B:
        raise ValueError("block_tables / context_lens batch mismatch")
    st = lib().paged_kv_append(_ptr(k_new), _ptr(v_new), _ptr(block_tables), _ptr(context_lens),
                               _ptr(k_cache), _ptr(v_cache), B, Hkv, D, BS, NB,
                               block_tables.shape[1], _ptr(error_word), _stream(stream))
    _check(st, "paged_kv_append")


def pkd_read_device_error(error_word, clear=True, stream=None) -> int:
    """Synchronise and return the device error bits (0 = none)."""
    bits = ctypes.c_uint(0)
    st = lib().pkd_read_device_error(_ptr(error_word), ctypes.byref(bits), int(bool(clear)),
                                     _stream(stream))
    if st not in (PKD_OK, 7):
        _check(st, "pkd_read_device_error")
    return int(bits.value)


def pkd_selftest_bounded_wait(error_word, budget_ns=1_000_000, stream=None):
    """Launch the bounded-wait self-test (a wait that can only time out)."""
    _check(lib().pkd_selftest_bounded_wait(_ptr(error_word), int(budget_ns), _stream(stream)),
           "pkd_selftest_bounded_wait")


def pkd_version() -> int:
    return int(lib().pkd_version())


def paged_decode_attention_static_scratch(q, k_cache, v_cache, block_tables, context_lens, scale,
                                          out=None, max_context_len=None, partition_size=0,
                                          variant="auto", prefetch_distance=0, error_word=None,
                                          stream=None) -> torch.Tensor:
    """Split-K decode attention whose partials live in the library's own
    fixed device array, for callers that cannot allocate device memory; the
    caller still provides the inputs and ``out``.  Calls must not overlap on
    the GPU (they share the array)."""
    B, Hq, Hkv, D, BS, NB, MB = _shape(q, k_cache, v_cache, block_tables, context_lens)
    if out is None:
        out = torch.empty_like(q)
    _want(out, "out", torch.float16, 3)
    st = lib().paged_decode_attention_static_scratch(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), _ptr(context_lens), _ptr(out),
        B, Hq, Hkv, D, BS, NB, MB, _max_len(context_lens, max_context_len), float(scale),
        int(partition_size), _variant(variant), int(prefetch_distance), _ptr(error_word),
        _stream(stream))
    _check(st, "paged_decode_attention_static_scratch")
    return out
