"""The C-ABI library: it loads without a GPU, exports every declared entry
point, and its host-side argument checks return the documented statuses
before any CUDA call."""
import ctypes
import os
import re

import pytest

from paged_kv_decode_21_gb300 import build as pkd_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "paged_decode.h")


@pytest.fixture(scope="module")
def L():
    pkd_build.build()
    from paged_kv_decode_21_gb300 import ops
    return ops.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*"
                                 r"([a-z][a-z0-9_]+)\s*\(", text, flags=re.M)))


def test_header_declares_entry_points():
    names = declared_functions()
    for n in ["paged_decode_attention", "paged_decode_attention_ex", "paged_decode_reduce",
              "paged_decode_partitions", "paged_decode_workspace_size", "pkd_status_string"]:
        assert n in names


def test_library_exports_every_declared_symbol(L):
    for n in declared_functions():
        assert hasattr(L, n), n


def test_version_and_status_strings(L):
    assert L.pkd_version() >= 10000
    for s in range(9):
        assert L.pkd_status_string(s)
    assert L.pkd_status_string(99) == b"unknown status"


FAKE = ctypes.c_void_p(1 << 20)          # aligned, never dereferenced on the failing paths
MISALIGNED = ctypes.c_void_p((1 << 20) + 2)


def call_ex(L, q=FAKE, k=FAKE, v=FAKE, bt=FAKE, cl=FAKE, out=FAKE, B=2, Hq=8, Hkv=2, D=128, BS=16,
            NB=64, MB=8, maxlen=100, scale=0.1, P=-1, var=0, pd=0, ws=None, wsb=0, err=None):
    return L.paged_decode_attention_ex(q, k, v, bt, cl, out, B, Hq, Hkv, D, BS, NB, MB, maxlen,
                                       ctypes.c_float(scale), P, var, pd, ws, wsb, err, None)


def test_null_pointer_rejected(L):
    assert call_ex(L, q=None) == 1
    assert call_ex(L, out=None) == 1


def test_shape_checks(L):
    assert call_ex(L, Hq=7, Hkv=2) == 2             # heads not divisible
    assert call_ex(L, maxlen=8 * 16 + 1) == 2       # longer than a table row
    assert call_ex(L, B=-1) == 2
    assert call_ex(L, scale=float("nan")) == 2
    assert call_ex(L, P=48) == 2                    # not a multiple of 32
    assert call_ex(L, var=9) == 2


def test_variant_flags(L):
    assert call_ex(L, var=0x100 | 3, D=96) == 3        # flag accepted; fails later on head_dim
    assert call_ex(L, var=0x200 | 3) == 2              # unknown flag bit
    assert L.paged_decode_workspace_size(2, 8, 2, 128, 16, 100, 32, 0x100 | 2) > 0


def test_unsupported_shapes(L):
    assert call_ex(L, D=96) == 3
    assert call_ex(L, BS=8) == 3
    assert call_ex(L, Hq=18, Hkv=2) == 3            # group of 9


def test_alignment_checks(L):
    assert call_ex(L, q=MISALIGNED) == 4
    assert call_ex(L, out=MISALIGNED) == 4


def test_split_needs_workspace(L):
    assert call_ex(L, P=32, maxlen=100) == 5
    small = ctypes.c_void_p(1 << 20)
    assert call_ex(L, P=32, maxlen=100, ws=small, wsb=16) == 5


def test_selftest_argument_checks(L):
    assert L.pkd_selftest_bounded_wait(None, 1000000, None) == 1
    assert L.pkd_selftest_bounded_wait(MISALIGNED, 1000000, None) == 4
    assert L.pkd_selftest_bounded_wait(FAKE, 10, None) == 2           # budget too short
    assert L.pkd_selftest_bounded_wait(FAKE, 10**9, None) == 2        # budget too long


def test_empty_batch_is_a_no_op(L):
    assert call_ex(L, B=0) == 0


def test_workspace_size_formula(L):
    # B=2, Hq=8, D=128, maxlen=100, P=32 -> NP=4: partials 2*8*4*128*4 B, m/l 2*8*4*4 B each
    n = L.paged_decode_workspace_size(2, 8, 2, 128, 16, 100, 32, 0)
    rows = 2 * 8 * 4
    def ru(x):
        return (x + 255) // 256 * 256
    assert n == ru(rows * 128 * 4) + 2 * ru(rows * 4)
    assert L.paged_decode_workspace_size(2, 8, 2, 128, 16, 32, 32, 0) == 0      # nothing splits
    assert L.paged_decode_workspace_size(2, 8, 2, 96, 16, 100, 32, 0) == 0      # unsupported


def test_auto_partition_policy(L):
    # many (sequence, kv head) units: no split
    assert L.paged_decode_auto_partition_size(256, 32, 32, 128, 16, 8192, 0) == -1
    # few units and long contexts: a split into multiples of 32
    p = L.paged_decode_auto_partition_size(2, 8, 1, 128, 16, 32768, 0)
    assert p > 0 and p % 32 == 0 and p < 32768
    assert L.paged_decode_auto_partition_size(2, 8, 3, 128, 16, 100, 0) == -2
    assert L.paged_decode_auto_partition_size(2, 8, 1, 128, 16, 32768, 7) == -2
    for variant in (1, 2, 3):
        p1 = L.paged_decode_auto_partition_size(2, 8, 1, 128, 16, 32768, variant)
        assert 0 < p1 and p1 % 32 == 0
