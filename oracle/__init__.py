"""CPU oracle for paged single-query decode attention (fp64).

TEST INFRASTRUCTURE ONLY: the tests, the package's smoke check and the
benchmark's CPU-baseline leg are the only callers.  The library's own code
never imports this package, and this package imports nothing from the library.

The arithmetic lives in ``pkd_oracle.c`` (plain C, IEEE double, compiled with
floating-point contraction off); this module compiles it with gcc on first use
and marshals numpy / torch-CPU arrays into it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pkd_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_lock = threading.Lock()
_libs = {}


def lib_path(mutant: int = 0) -> str:
    name = "libpkd_oracle.so" if mutant == 0 else f"libpkd_oracle_mutant{mutant}.so"
    return os.path.join(_BUILD, name)


def build(mutant: int = 0, force: bool = False) -> str:
    """Compile the oracle (optionally with a planted mistake) and return the .so path."""
    out = lib_path(mutant)
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(_SRC):
        return out
    os.makedirs(_BUILD, exist_ok=True)
    tmp = out + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-ffp-contract=off",
           "-fno-fast-math", f"-DPKD_ORACLE_MUTANT={int(mutant)}", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _load(mutant: int = 0):
    with _lock:
        if mutant in _libs:
            return _libs[mutant]
        lib = ctypes.CDLL(build(mutant))
        P, I, D = ctypes.c_void_p, ctypes.c_int, ctypes.c_double
        common = [P, P, P, P, P, I, I, I, I, I, I, I, D]
        lib.pkd_oracle_attention.argtypes = common + [P, I, P, I]
        lib.pkd_oracle_attention.restype = I
        lib.pkd_oracle_attention_multi.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, I, D, P, I, P, I]
        lib.pkd_oracle_attention_multi.restype = I
        lib.pkd_oracle_weights.argtypes = common + [I, I, P]
        lib.pkd_oracle_weights.restype = I
        lib.pkd_oracle_partitions.argtypes = common + [I, I, P, P, P]
        lib.pkd_oracle_partitions.restype = I
        lib.pkd_oracle_merge.argtypes = [P, P, P, P, I, I, I, I, I, P]
        lib.pkd_oracle_merge.restype = I
        lib.pkd_oracle_append.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I]
        lib.pkd_oracle_append.restype = I
        lib.pkd_oracle_attention_fp8.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, I, D, D, D, P, I, P, I]
        lib.pkd_oracle_attention_fp8.restype = I
        lib.pkd_oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
        lib.pkd_oracle_e4m3_to_double.restype = D
        lib.pkd_oracle_float_to_e4m3.argtypes = [ctypes.c_float]
        lib.pkd_oracle_float_to_e4m3.restype = ctypes.c_uint8
        lib.pkd_oracle_quantize_e4m3.argtypes = [P, I, ctypes.c_float, P]
        lib.pkd_oracle_quantize_e4m3.restype = None
        lib.pkd_oracle_append_fp8.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, ctypes.c_float, ctypes.c_float]
        lib.pkd_oracle_append_fp8.restype = I
        lib.pkd_oracle_half_to_double.argtypes = [ctypes.c_uint16]
        lib.pkd_oracle_half_to_double.restype = D
        lib.pkd_oracle_mutant.argtypes = []
        lib.pkd_oracle_mutant.restype = I
        _libs[mutant] = lib
        return lib


def _np(x, dtype):
    """numpy view/copy of a numpy array or CPU torch tensor, C-contiguous."""
    if hasattr(x, "detach"):
        x = x.detach().cpu().contiguous().numpy()
    return np.ascontiguousarray(x, dtype=dtype)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


class OracleError(RuntimeError):
    pass


def _check(rc: int, what: str):
    if rc == -1:
        raise OracleError(f"{what}: a used block-table entry is outside the pool")
    if rc == -2:
        raise OracleError(f"{what}: out of memory")
    if rc != 0:
        raise OracleError(f"{what}: bad argument (rc={rc})")


def _problem(q, k_cache, v_cache, block_tables, context_lens):
    qa = _np(q, np.float16).view(np.uint16)
    ka = _np(k_cache, np.float16).view(np.uint16)
    va = _np(v_cache, np.float16).view(np.uint16)
    bt = _np(block_tables, np.int32)
    cl = _np(context_lens, np.int32)
    B, Hq, D = qa.shape
    NB, Hkv, BS, D2 = ka.shape
    assert D2 == D and va.shape == ka.shape and bt.shape[0] == B and cl.shape == (B,)
    return qa, ka, va, bt, cl, (B, Hq, Hkv, D, BS, NB, bt.shape[1])


def attention(q, k_cache, v_cache, block_tables, context_lens, scale, rows=None,
              threads=None, mutant: int = 0) -> np.ndarray:
    """Exact fp64 attention.  ``rows`` (b*Hq+h ids) selects rows; returns
    [B][Hq][D] when ``rows`` is None, else [len(rows)][D]."""
    lib = _load(mutant)
    qa, ka, va, bt, cl, (B, Hq, Hkv, D, BS, NB, MB) = _problem(q, k_cache, v_cache,
                                                              block_tables, context_lens)
    if threads is None:
        threads = os.cpu_count() or 1
    if rows is None:
        out = np.empty((B, Hq, D), np.float64)
        rp, nr = None, 0
    else:
        ra = _np(rows, np.int32).reshape(-1)
        out = np.empty((ra.shape[0], D), np.float64)
        rp, nr = _ptr(ra), ra.shape[0]
    rc = lib.pkd_oracle_attention(_ptr(qa), _ptr(ka), _ptr(va), _ptr(bt), _ptr(cl), B, Hq, Hkv, D,
                                  BS, NB, MB, float(scale), rp, nr, _ptr(out), int(threads))
    _check(rc, "attention")
    return out


def attention_multi(q, k_cache, v_cache, block_tables, context_lens, scale, rows=None,
                    threads=None, mutant: int = 0) -> np.ndarray:
    """Exact fp64 attention of q_len new tokens per sequence, q [B][q_len][Hq][D]:
    query jq sits at position L_b - q_len + jq and sees tokens up to and including
    itself.  ``rows`` ((b*q_len + jq)*Hq + h ids) selects rows; returns
    [B][q_len][Hq][D] when ``rows`` is None, else [len(rows)][D]."""
    lib = _load(mutant)
    qm = _np(q, np.float16)
    B, QL, Hq, D = qm.shape
    qa, ka, va, bt, cl, (_, _, Hkv, _, BS, NB, MB) = _problem(qm.reshape(B, QL * Hq, D), k_cache,
                                                              v_cache, block_tables, context_lens)
    if threads is None:
        threads = os.cpu_count() or 1
    if rows is None:
        out = np.empty((B, QL, Hq, D), np.float64)
        rp, nr = None, 0
    else:
        ra = _np(rows, np.int32).reshape(-1)
        out = np.empty((ra.shape[0], D), np.float64)
        rp, nr = _ptr(ra), ra.shape[0]
    rc = lib.pkd_oracle_attention_multi(_ptr(qa), _ptr(ka), _ptr(va), _ptr(bt), _ptr(cl), B, QL, Hq, Hkv,
                                        D, BS, NB, MB, float(scale), rp, nr, _ptr(out), int(threads))
    _check(rc, "attention_multi")
    return out


def weights(q, k_cache, v_cache, block_tables, context_lens, scale, b, h, mutant: int = 0):
    """Softmax weights of row (b, h) over its L_b tokens (fp64)."""
    lib = _load(mutant)
    qa, ka, va, bt, cl, (B, Hq, Hkv, D, BS, NB, MB) = _problem(q, k_cache, v_cache,
                                                              block_tables, context_lens)
    w = np.zeros(max(1, int(cl[b])), np.float64)
    rc = lib.pkd_oracle_weights(_ptr(qa), _ptr(ka), _ptr(va), _ptr(bt), _ptr(cl), B, Hq, Hkv, D,
                                BS, NB, MB, float(scale), int(b), int(h), _ptr(w))
    _check(rc, "weights")
    return w[: int(cl[b])]


def partitions(q, k_cache, v_cache, block_tables, context_lens, scale, partition_size,
               max_partitions=None, mutant: int = 0):
    """Per-partition (m, l, o): [B][Hq][NP], [B][Hq][NP], [B][Hq][NP][D] (fp64)."""
    lib = _load(mutant)
    qa, ka, va, bt, cl, (B, Hq, Hkv, D, BS, NB, MB) = _problem(q, k_cache, v_cache,
                                                              block_tables, context_lens)
    if max_partitions is None:
        max_partitions = max(1, int(-(-int(cl.max(initial=0)) // partition_size)))
    m = np.empty((B, Hq, max_partitions), np.float64)
    l = np.empty((B, Hq, max_partitions), np.float64)
    o = np.empty((B, Hq, max_partitions, D), np.float64)
    rc = lib.pkd_oracle_partitions(_ptr(qa), _ptr(ka), _ptr(va), _ptr(bt), _ptr(cl), B, Hq, Hkv,
                                   D, BS, NB, MB, float(scale), int(partition_size),
                                   int(max_partitions), _ptr(m), _ptr(l), _ptr(o))
    _check(rc, "partitions")
    return m, l, o


def merge(m, l, o, context_lens, partition_size, mutant: int = 0) -> np.ndarray:
    """Log-sum-exp merge of partition statistics into [B][Hq][D] (fp64)."""
    lib = _load(mutant)
    ma, la, oa = (np.ascontiguousarray(x, np.float64) for x in (m, l, o))
    cl = _np(context_lens, np.int32)
    B, Hq, NP, D = oa.shape
    out = np.empty((B, Hq, D), np.float64)
    rc = lib.pkd_oracle_merge(_ptr(ma), _ptr(la), _ptr(oa), _ptr(cl), B, Hq, D,
                              int(partition_size), NP, _ptr(out))
    _check(rc, "merge")
    return out


def append(k_new, v_new, block_tables, context_lens, k_cache, v_cache, mutant: int = 0,
           check: bool = True):
    """Write each sequence's new K/V row at logical position context_lens[b];
    returns new (k_cache, v_cache) arrays (float16) and leaves the inputs alone."""
    lib = _load(mutant)
    kn = _np(k_new, np.float16).view(np.uint16)
    vn = _np(v_new, np.float16).view(np.uint16)
    bt = _np(block_tables, np.int32)
    cl = _np(context_lens, np.int32)
    kc = _np(k_cache, np.float16).copy().view(np.uint16)
    vc = _np(v_cache, np.float16).copy().view(np.uint16)
    NB, Hkv, BS, D = kc.shape
    B = cl.shape[0]
    assert kn.shape == (B, Hkv, D) and vn.shape == (B, Hkv, D)
    rc = lib.pkd_oracle_append(_ptr(kn), _ptr(vn), _ptr(bt), _ptr(cl), _ptr(kc), _ptr(vc), B, Hkv, D, BS,
                               NB, bt.shape[1])
    if check:
        _check(rc, "append")
    return kc.view(np.float16), vc.view(np.float16)


def e4m3_to_double(bits, mutant: int = 0) -> np.ndarray:
    """Decode E4M3 bytes (the format's definition) to float64."""
    lib = _load(mutant)
    b = np.asarray(bits, dtype=np.uint8).reshape(-1)
    return np.array([lib.pkd_oracle_e4m3_to_double(int(x)) for x in b], np.float64)


def float_to_e4m3(x, mutant: int = 0) -> np.ndarray:
    """Round float32 values to E4M3 bytes (nearest-even, saturating at 448)."""
    lib = _load(mutant)
    f = np.asarray(x, dtype=np.float32).reshape(-1)
    return np.array([lib.pkd_oracle_float_to_e4m3(float(v)) for v in f], np.uint8)


def quantize_e4m3(x_fp16, scale: float, mutant: int = 0) -> np.ndarray:
    """E4M3 bytes of fp16 values: e4m3(fp32(x) / scale), the division in fp32."""
    lib = _load(mutant)
    xa = _np(x_fp16, np.float16)
    flat = np.ascontiguousarray(xa.reshape(-1)).view(np.uint16)
    out = np.empty(flat.shape[0], np.uint8)
    lib.pkd_oracle_quantize_e4m3(_ptr(flat), int(flat.shape[0]), float(scale), _ptr(out))
    return out.reshape(xa.shape)


def attention_fp8(q, k_cache8, v_cache8, block_tables, context_lens, scale, k_scale, v_scale, rows=None,
                  threads=None, mutant: int = 0) -> np.ndarray:
    """Exact fp64 attention over E4M3 caches (value = e4m3(byte) * k_scale / v_scale).
    q is [B][Hq][D] (single query) or [B][q_len][Hq][D] (causal multi-token)."""
    lib = _load(mutant)
    qm = _np(q, np.float16)
    single = qm.ndim == 3
    if single:
        qm = qm[:, None]
    B, QL, Hq, D = qm.shape
    k8 = _np(k_cache8, np.uint8)
    v8 = _np(v_cache8, np.uint8)
    bt = _np(block_tables, np.int32)
    cl = _np(context_lens, np.int32)
    NB, Hkv, BS, D2 = k8.shape
    assert D2 == D and v8.shape == k8.shape and bt.shape[0] == B and cl.shape == (B,)
    qa = np.ascontiguousarray(qm).view(np.uint16)
    if threads is None:
        threads = os.cpu_count() or 1
    if rows is None:
        out = np.empty((B, QL, Hq, D), np.float64)
        rp, nr = None, 0
    else:
        ra = _np(rows, np.int32).reshape(-1)
        out = np.empty((ra.shape[0], D), np.float64)
        rp, nr = _ptr(ra), ra.shape[0]
    rc = lib.pkd_oracle_attention_fp8(_ptr(qa), _ptr(k8), _ptr(v8), _ptr(bt), _ptr(cl), B, QL, Hq, Hkv, D, BS,
                                      NB, bt.shape[1], float(scale), float(k_scale), float(v_scale), rp, nr,
                                      _ptr(out), int(threads))
    _check(rc, "attention_fp8")
    if rows is None and single:
        return out[:, 0]
    return out


def append_fp8(k_new, v_new, block_tables, context_lens, k_cache8, v_cache8, k_scale, v_scale,
               mutant: int = 0, check: bool = True):
    """FP8 cache write: returns new (k_cache8, v_cache8) with each sequence's new row
    quantized into position context_lens[b]; the inputs are left alone."""
    lib = _load(mutant)
    kn = _np(k_new, np.float16).view(np.uint16)
    vn = _np(v_new, np.float16).view(np.uint16)
    bt = _np(block_tables, np.int32)
    cl = _np(context_lens, np.int32)
    kc = _np(k_cache8, np.uint8).copy()
    vc = _np(v_cache8, np.uint8).copy()
    NB, Hkv, BS, D = kc.shape
    B = cl.shape[0]
    rc = lib.pkd_oracle_append_fp8(_ptr(kn), _ptr(vn), _ptr(bt), _ptr(cl), _ptr(kc), _ptr(vc), B, Hkv, D, BS,
                                   NB, bt.shape[1], float(k_scale), float(v_scale))
    if check:
        _check(rc, "append_fp8")
    return kc, vc


def half_to_double(bits) -> np.ndarray:
    """Decode uint16 binary16 bit patterns with the oracle's own decoder."""
    lib = _load(0)
    b = np.asarray(bits, np.uint16).reshape(-1)
    return np.array([lib.pkd_oracle_half_to_double(int(x)) for x in b], np.float64)


def mutant_id(mutant: int) -> int:
    return _load(mutant).pkd_oracle_mutant()
