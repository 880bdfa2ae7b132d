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
              "paged_decode_partitions", "paged_decode_workspace_size", "paged_kv_append",
              "pkd_status_string"]:
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
    assert call_ex(L, var=0x400 | 3) == 2              # unknown flag bit
    assert call_ex(L, var=0x200 | 4, D=96) == 3        # the longest-first flag is known
    # the order (one int32 per sequence, 256-byte aligned) follows the split partials
    base = L.paged_decode_workspace_size(2, 8, 2, 128, 16, 100, 32, 4)
    assert L.paged_decode_workspace_size(2, 8, 2, 128, 16, 100, 32, 0x200 | 4) == base + 256
    assert L.paged_decode_workspace_size(300, 8, 2, 128, 16, 100, -1, 0x200 | 4) == 1280
    assert call_ex(L, var=4, D=96) == 3                # the tensor-core path is a known variant
    assert call_ex(L, var=5, D=96) == 3                # tcgen05 path: head_dim 64 or 128
    assert call_ex(L, var=0x200 | 5, D=96) == 3        # ... and a known variant with flags
    assert call_ex(L, var=6) == 2                      # past the last variant
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


def test_multi_query_argument_checks(L):
    # (q, k, v, bt, cl, out, B, q_len, Hq, Hkv, D, BS, NB, MB, maxlen, scale, P, ws, wsb, err, stream)
    def call(*, ptrs=(FAKE,) * 6, B=2, QL=3, Hq=8, Hkv=2, D=128, BS=16, NB=64, MB=8, maxlen=100, P=-1,
             ws=None, wsb=0):
        return L.paged_decode_attention_multi(*ptrs, B, QL, Hq, Hkv, D, BS, NB, MB, maxlen,
                                              ctypes.c_float(0.1), P, ws, wsb, None, None)
    assert call(B=0) == 0                                     # empty batch: a no-op
    assert call(QL=0) == 2                                    # at least one query token
    assert call(ptrs=(None,) + (FAKE,) * 5) == 1
    assert call(D=96) == 3 and call(Hq=18) == 3               # head_dim; group of 9
    assert call(P=64, maxlen=100) == 5                        # split without a workspace
    assert call(ptrs=(FAKE,) * 5 + (MISALIGNED,)) == 4
    # partials are (sequence, query token, head) rows
    ws = L.paged_decode_multi_workspace_size(2, 3, 8, 2, 128, 16, 100, 64)
    one = L.paged_decode_workspace_size(6, 8, 2, 128, 16, 100, 64, 4)
    assert ws == one > 0
    assert L.paged_decode_multi_workspace_size(2, 3, 8, 2, 128, 16, 100, -1) == 0
    assert L.paged_decode_multi_workspace_size(2, 0, 8, 2, 128, 16, 100, 64) == 0


def test_append_argument_checks(L):
    # (k_new, v_new, bt, cl, kc, vc, B, Hkv, D, BS, NB, MB, err, stream); nothing is launched
    def call(*, ptrs=(FAKE,) * 6, B=2, Hkv=2, D=64, BS=16, NB=4, MB=2, err=None):
        return L.paged_kv_append(*ptrs, B, Hkv, D, BS, NB, MB, err, None)
    assert call(B=0) == 0                                      # empty batch: a no-op
    assert call(ptrs=(FAKE, None, FAKE, FAKE, FAKE, FAKE)) == 1
    assert call(D=12) == 2                                     # head_dim not a multiple of 8
    assert call(BS=0) == 2 and call(NB=0) == 2 and call(MB=0) == 2 and call(B=-1) == 2
    assert call(ptrs=(FAKE, FAKE, FAKE, FAKE, MISALIGNED, FAKE)) == 4
    assert call(err=MISALIGNED) == 4


def test_auto_variant_policy(L):
    from paged_kv_decode_21_gb300 import ops
    # no GPU here: the library assumes 148 SMs; the cases sit far from the
    # thresholds, so they hold for 152 as well
    av = ops.paged_decode_auto_variant
    staged = ops.VARIANTS["tma_mma"]
    # the tensor-core path at every shape, short CTAs included
    assert av(64, 32, 32, 128, 16, 2048) == staged      # long CTAs
    assert av(64, 32, 32, 128, 16, 512) == staged       # 2048 CTAs of 512 tokens
    assert av(16, 32, 32, 128, 16, 2048) == staged      # split at 512: 2048 CTAs
    assert av(256, 32, 32, 128, 16, 512) == staged      # 8192 CTAs: many waves
    assert av(1, 32, 32, 128, 16, 1024) == staged       # fewer CTAs than SMs
    assert av(64, 32, 8, 128, 16, 512) == staged
    assert av(64, 32, 32, 128, 16, 512, -1) == staged
    assert av(64, 32, 32, 128, 16, 4096, 256) == staged  # 16384 CTAs
    # unsplit grids of one to six waves of units walk the batch longest first
    ordered = staged | ops.FLAG_LONGEST_FIRST
    assert av(128, 32, 8, 128, 16, 4096) == ordered      # 1024 units: 3.5 waves
    assert av(128, 32, 8, 128, 16, 4096, -1) == staged   # an explicit partition keeps the grid order
    assert av(128, 32, 8, 128, 16, 512) == staged        # short contexts: the order is not paid back
    assert av(1024, 32, 8, 128, 16, 4096) == staged      # 8192 units: many waves
    assert ops.variant_name(ordered) == "tma_mma+longest_first"
    assert ops.variant_name(staged) == "tma_mma"
    assert ops.variant_name(ops.VARIANTS["tma_staged"] | ops.FLAG_L2_EVICT_HINTS) == "tma_staged+l2_hints"
    with pytest.raises(ops.PagedDecodeError):
        av(64, 32, 32, 128, 16, 512, 100)               # partition not a multiple of 32


def test_auto_plan_matches_policy(L):
    from paged_kv_decode_21_gb300 import ops
    plan = ops.paged_decode_auto_plan
    assert plan(64, 1, 32, 32, 128, 16, 2048) == (1, -1, False)      # MHA bench shape: one launch
    assert plan(128, 1, 32, 8, 128, 16, 4096) == (2, -1, True)       # order + decode
    assert plan(128, 1, 32, 8, 128, 16, 4096, kv_fp8=True) == (2, -1, True)
    n, part, order = plan(32, 1, 40, 8, 128, 16, 32768)              # 256 units: split + merge
    assert n == 2 and part > 0 and not order
    n, part, order = plan(256, 1, 28, 4, 128, 16, 8192)              # long contexts below six waves split
    assert n == 2 and part == 2048 and not order
    # multi-token queries count query chunks as units: 16 / G tokens per CTA
    assert plan(128, 4, 32, 8, 128, 16, 4096)[0] in (2, 3)
    assert plan(0, 1, 32, 8, 128, 16, 4096) == (0, -1, False)
    with pytest.raises(ops.PagedDecodeError):
        plan(2, 0, 8, 2, 128, 16, 100)


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


def test_small_grid_split_fills_one_wave():
    # Calls on a tensor-core path whose (sequence, kv head) units cover less than one resident
    # wave take the shortest power-of-two partition whose grid still fits one wave: single query
    # on mma.sync, 128..2048 tokens, three CTAs per SM (148 SMs without a GPU).
    from paged_kv_decode_21_gb300 import ops
    slots = 148 * 3
    for B, Hq, Hkv, L, want in [(1, 32, 32, 2048, 256), (4, 32, 32, 2048, 1024), (1, 32, 8, 2048, 128),
                                (16, 32, 8, 2048, 1024), (16, 28, 4, 8192, 2048), (4, 28, 4, 8192, 512),
                                (1, 28, 4, 8192, 128)]:
        n, P, _, var, grid, _ = ops.paged_decode_call_plan(B, 1, Hq, Hkv, 128, 16, L)
        assert var == "tma_mma" and P == want, (B, Hq, Hkv, L, P)
        assert grid == B * Hkv * -(-L // P) <= slots
        assert P == 128 or B * Hkv * -(-L // (P // 2)) > slots
    # the tcgen05 path (multi-token queries): two CTAs per SM, partitions of 256..8192 tokens
    for B, Hq, Hkv, L, want in [(1, 32, 8, 2048, 256), (16, 32, 8, 2048, 1024), (16, 32, 8, 8192, 4096),
                                (16, 28, 4, 8192, 2048), (4, 28, 4, 8192, 512)]:
        for fp8 in (False, True):
            n, P, _, var, grid, _ = ops.paged_decode_call_plan(B, 8, Hq, Hkv, 128, 16, L, kv_fp8=fp8)
            assert var.startswith("tcgen05") and P == want, (B, Hq, Hkv, L, fp8, P)
            assert grid == B * Hkv * -(-L // P) <= 148 * 2
            assert P == 256 or B * Hkv * -(-L // (P // 2)) > 148 * 2
    # more units than a wave: the waves-based split (512 at least), unchanged
    assert ops.paged_decode_call_plan(16, 1, 32, 32, 128, 16, 2048)[1] == 512
    assert ops.paged_decode_call_plan(16, 1, 32, 32, 128, 16, 8192)[1] == 2048
    # the CUDA-core paths keep the waves-based split
    assert ops.paged_decode_call_plan(1, 1, 32, 32, 128, 16, 2048, variant="tma_staged")[1] == 512


def test_tcgen05_tail_split_plan():
    # An unsplit, longest-first tcgen05 grid whose last round of resident CTAs (two per SM,
    # 148 SMs without a GPU) is at most half full sizes its grid for splitting its K shortest
    # sequences in two, K = ceil(CTAs of the last round / CTAs per sequence): grid (B + K) x kv
    # heads x query chunks (the order kernel splits those of them at least half as long as the
    # longest sequence; the other slots exit at once).
    from paged_kv_decode_21_gb300 import ops
    slots = 2 * 148
    for B, Hq, Hkv, q_len, L in [(160, 28, 4, 8, 2048), (256, 28, 4, 8, 8192), (128, 32, 8, 8, 4096),
                                 (300, 28, 4, 8, 2048), (76, 32, 8, 8, 2048)]:
        for fp8 in (False, True):
            n, part, ordered, var, grid, _ = ops.paged_decode_call_plan(B, q_len, Hq, Hkv, 128, 16, L, kv_fp8=fp8)
            units = B * Hkv
            last = units - (units - 1) // slots * slots
            k = -(-last // Hkv) if units > slots and 2 * last <= slots else 0
            assert var.startswith("tcgen05") and part == -1 and ordered, (B, L, var, part)
            assert grid == (B + k) * Hkv and n == (3 if k else 2), (B, L, fp8, grid, k)
            ws = ops.paged_decode_multi_workspace_size(B, q_len, Hq, Hkv, 128, 16, L, 0)
            rows = B * q_len * Hq
            if k:  # partials of two partitions per row, the order of B + K pieces and its tail record
                assert ws >= rows * 2 * 128 * 4 + 2 * rows * 2 * 4 + (B + k) * 4 + 8
    # an explicit partition, short contexts, or a path other than tcgen05: no tail split
    assert ops.paged_decode_call_plan(256, 8, 28, 4, 128, 16, 8192, partition_size=-1)[4] == 1024
    assert ops.paged_decode_call_plan(256, 8, 28, 4, 128, 16, 512)[4] == 1024
    assert ops.paged_decode_call_plan(256, 1, 28, 4, 128, 16, 8192, variant="tma_mma")[4] == 1024 * 4


def test_tcgen05_partition_runs_plan():
    # Explicit partitions of up to 1024 tokens on the tcgen05 path at head_dim 128: a CTA takes
    # a run of up to 4096 tokens of consecutive partitions while the grid keeps four waves of
    # CTAs (two per SM, 148 SMs without a GPU); every other path and shape keeps one partition
    # per CTA.
    from paged_kv_decode_21_gb300 import ops
    floor = 4 * 148 * 2
    for B, Hq, Hkv, L, P, want_runs in [(32, 40, 8, 32768, 512, 8), (16, 40, 8, 16384, 512, 2),
                                        (64, 40, 8, 16384, 256, 16), (32, 40, 8, 32768, 1024, 4),
                                        (4, 40, 8, 8192, 512, 1), (32, 40, 8, 32768, 2048, 1),
                                        (64, 40, 8, 32768, 2048, 1)]:
        for fp8 in (False, True):
            n, part, order, var, grid, _ = ops.paged_decode_call_plan(B, 8, Hq, Hkv, 128, 16, L, kv_fp8=fp8,
                                                                      partition_size=P)
            units, npart = B * Hkv, -(-L // P)
            assert var == "tcgen05" and part == P and not order, (B, L, P, fp8)
            assert grid == units * -(-npart // want_runs), (B, L, P, fp8, grid)
            assert want_runs == 1 or grid >= floor
            assert P > 1024 or want_runs * 2 > 4096 // P or units * -(-npart // (want_runs * 2)) < floor
    # single query (mma.sync) and head_dim 64 keep one partition per CTA
    assert ops.paged_decode_call_plan(32, 1, 40, 8, 128, 16, 32768, partition_size=512)[4] == 32 * 8 * 64
    assert ops.paged_decode_call_plan(32, 8, 40, 8, 64, 16, 32768, partition_size=512,
                                      variant="tcgen05")[4] == 32 * 8 * 64
    # a partition that is not a multiple of the 64-token tile keeps one partition per CTA
    assert ops.paged_decode_call_plan(32, 8, 40, 8, 128, 16, 32768, partition_size=480)[4] == 32 * 8 * 69


def test_workspace_sizes_cover_every_plan(L):
    # For random shapes, partitions and flags, a workspace of exactly the reported size is
    # never refused (PKD_ERR_WORKSPACE = 5); without a GPU the call then fails at launch
    # (PKD_ERR_LAUNCH = 6) or on the device query (PKD_ERR_CUDA = 8), after every host check.
    import random
    rng = random.Random(7)
    ws_ptr = ctypes.c_void_p(1 << 20)
    for _ in range(300):
        Hkv = rng.choice([1, 2, 4, 8])
        G = rng.randint(1, 8)
        D = rng.choice([64, 128])
        BS = rng.choice([16, 32])
        B = rng.randint(1, 300)
        maxlen = rng.randint(1, 20000)
        MB = -(-maxlen // BS) + rng.randint(0, 3)
        P = rng.choice([0, 0, -1, 32 * BS // 16 * rng.randint(1, 64)])
        var = rng.choice([0, 4, 4 | 0x200, 3, 0x100 | 4, 5, 5 | 0x200])
        need = L.paged_decode_workspace_size(B, G * Hkv, Hkv, D, BS, maxlen, P, var)
        st = L.paged_decode_attention_ex(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, B, G * Hkv, Hkv, D, BS, 64, MB, maxlen,
                                         ctypes.c_float(0.1), P, var, 0, ws_ptr if need else None, need, None, None)
        assert st in (6, 8), (B, G, Hkv, D, BS, maxlen, P, var, need, st)
        q_len = rng.randint(1, 9)
        needm = L.paged_decode_multi_workspace_size(B, q_len, G * Hkv, Hkv, D, BS, maxlen, P)
        stm = L.paged_decode_attention_multi(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, B, q_len, G * Hkv, Hkv, D, BS, 64, MB,
                                             maxlen, ctypes.c_float(0.1), P, ws_ptr if needm else None, needm, None, None)
        assert stm in (6, 8), (B, q_len, G, Hkv, D, BS, maxlen, P, needm, stm)
        # the multi-token entry with each tensor-core path forced (tcgen05: head_dim 128 only)
        for mvar in (4, 5, 5 | 0x200):
            stx = L.paged_decode_attention_multi_ex(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, B, q_len, G * Hkv, Hkv, D, BS,
                                                    64, MB, maxlen, ctypes.c_float(0.1), P, mvar,
                                                    ws_ptr if needm else None, needm, None, None)
            assert stx in (6, 8), (B, q_len, G, Hkv, D, BS, maxlen, P, mvar, needm, stx)
        stf = L.paged_decode_attention_fp8(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, B, q_len, G * Hkv, Hkv, D, BS, 64, MB,
                                           maxlen, ctypes.c_float(0.1), ctypes.c_float(0.5), ctypes.c_float(0.5), P,
                                           ws_ptr if needm else None, needm, None, None)
        assert stf in (6, 8), (B, q_len, G, Hkv, D, BS, maxlen, P, needm, stf)


def test_multi_ex_argument_checks(L):
    # (q, k, v, bt, cl, out, B, q_len, Hq, Hkv, D, BS, NB, MB, maxlen, scale, P, variant, ws, wsb, err, stream)
    def call(*, QL=3, D=128, var=5, P=-1):
        return L.paged_decode_attention_multi_ex(*(FAKE,) * 6, 2, QL, 8, 2, D, 16, 64, 8, 100, ctypes.c_float(0.1),
                                                 P, var, None, 0, None, None)
    assert call(var=5, D=96) == 3            # tcgen05: head_dim 64 or 128
    assert call(var=1) == 3 and call(var=3) == 3   # CUDA-core paths: single query only
    assert call(var=6) == 2                  # not a variant
    assert call(var=5, P=64) == 5            # split without a workspace
    assert call(var=5, QL=0) == 2
    assert call(var=5) in (6, 8)             # passes every host check (no GPU here)
    assert call(var=4) in (6, 8) and call(var=0) in (6, 8)


def test_host_entry_argument_checks(L):
    def call(*, ptrs=(FAKE,) * 12, B=2, D=128, ws=None, wsb=0):
        return L.paged_decode_attention_host(*ptrs, B, 8, 2, D, 16, 64, 8, 100, ctypes.c_float(0.1), 1, ws, wsb,
                                             None, None)
    assert call(B=0) == 0                                   # empty batch: a no-op
    assert call(ptrs=(None,) + (FAKE,) * 11) == 1           # a host buffer missing
    assert call(ptrs=(FAKE,) * 6 + (None,) + (FAKE,) * 5) == 1  # a device buffer missing
    assert call(ptrs=(MISALIGNED,) + (FAKE,) * 11) == 4
    assert call(D=96) == 3


def test_call_plan_picks_the_tensor_core_path(L):
    from paged_kv_decode_21_gb300 import ops
    # two or more 16-row mma.sync tiles of q_len x G rows, fp16 caches, head_dim 128: tcgen05
    assert ops.paged_decode_call_plan(4, 8, 28, 4, 128, 16, 1000)[3] == "tcgen05"   # 4 tiles
    assert ops.paged_decode_call_plan(4, 4, 28, 4, 128, 16, 1000)[3] == "tcgen05"   # 2 tiles
    assert ops.paged_decode_call_plan(4, 8, 32, 8, 128, 16, 1000)[3] == "tcgen05"   # 2 tiles
    assert ops.paged_decode_call_plan(4, 17, 4, 4, 128, 16, 1000)[3] == "tcgen05"   # G=1: 2 tiles
    # E4M3 caches: the same rule
    assert ops.paged_decode_call_plan(4, 8, 28, 4, 128, 16, 1000, kv_fp8=True)[3] == "tcgen05"   # 4 tiles
    assert ops.paged_decode_call_plan(4, 8, 40, 8, 128, 16, 1000, kv_fp8=True)[3] == "tcgen05"   # 3 tiles
    assert ops.paged_decode_call_plan(4, 4, 28, 4, 128, 16, 1000, kv_fp8=True)[3] == "tcgen05"   # 2 tiles
    assert ops.paged_decode_call_plan(4, 8, 32, 8, 128, 16, 1000, kv_fp8=True)[3] == "tcgen05"   # 2 tiles
    # one tile, head_dim 64 or a single query: the mma.sync path
    assert ops.paged_decode_call_plan(4, 2, 28, 4, 128, 16, 1000)[3] == "tma_mma"
    assert ops.paged_decode_call_plan(4, 4, 32, 8, 128, 16, 1000)[3] == "tma_mma"
    assert ops.paged_decode_call_plan(4, 16, 4, 4, 128, 16, 1000)[3] == "tma_mma"
    assert ops.paged_decode_call_plan(4, 8, 28, 4, 64, 16, 1000)[3] == "tcgen05"                # head_dim 64
    assert ops.paged_decode_call_plan(4, 8, 28, 4, 64, 16, 1000, kv_fp8=True)[3] == "tma_mma"   # E4M3 at 64
    assert ops.paged_decode_call_plan(4, 2, 28, 4, 128, 16, 1000, kv_fp8=True)[3] == "tma_mma"
    assert ops.paged_decode_call_plan(4, 1, 28, 4, 128, 16, 1000, kv_fp8=True)[3] == "tma_mma"
    assert ops.paged_decode_call_plan(4, 1, 28, 4, 128, 16, 1000)[3] == "tma_mma"
    # grid: (sequence, kv head, chunk of 64 / G query tokens, partition)
    n, part, ordered, var, grid, _ = ops.paged_decode_call_plan(4, 10, 28, 4, 128, 16, 1000, partition_size=256,
                                                             variant="tcgen05")
    assert (n, part, var, grid) == (2, 256, "tcgen05", 4 * 4 * 2 * 4)
    n, part, ordered, var, grid, _ = ops.paged_decode_call_plan(4, 10, 28, 4, 128, 16, 1000, partition_size=-1,
                                                             variant="tma_mma")
    assert (n, part, grid) == (1, -1, 4 * 4 * 5)
    # refused: tcgen05 with head_dim 64, CUDA-core paths for several queries
    with pytest.raises(ops.PagedDecodeError):
        ops.paged_decode_call_plan(4, 8, 28, 4, 128, 16, 1000, variant="tma_staged")
    with pytest.raises(ops.PagedDecodeError):  # E4M3 at head_dim 64
        ops.paged_decode_call_plan(4, 8, 28, 4, 64, 16, 1000, kv_fp8=True, variant="tcgen05")


def test_multi_workspace_covers_both_tensor_core_paths(L):
    from paged_kv_decode_21_gb300 import ops
    # with partition 0 the split depends on the path; the size covers either
    import random
    rng = random.Random(5)
    for _ in range(200):
        G = rng.choice([1, 2, 4, 5, 7, 8])
        Hkv = rng.choice([1, 2, 4, 8])
        B = rng.choice([1, 2, 7, 32, 100, 300])
        q_len = rng.choice([2, 3, 5, 8, 9, 17, 33])
        maxlen = rng.choice([16, 100, 1000, 5000, 20000])
        ws = L_size = ops.paged_decode_multi_workspace_size(B, q_len, G * Hkv, Hkv, 128, 16, maxlen, 0)
        for variant in ("auto", "tma_mma", "tcgen05"):
            n, part, ordered, var, grid, _ = ops.paged_decode_call_plan(B, q_len, G * Hkv, Hkv, 128, 16, maxlen,
                                                                     partition_size=0, variant=variant)
            need = 0
            if part > 0:
                rows = B * q_len * G * Hkv * (-(-maxlen // part))
                need = -(-rows * 128 * 4 // 256) * 256 + 2 * (-(-rows * 4 // 256) * 256)
            assert ws >= need, (B, q_len, G, Hkv, maxlen, variant)
        assert L_size == ws


def test_tcgen05_split_policy(L):
    # the tcgen05 path splits only below two waves of units (two CTAs per SM), into
    # partitions of up to 8192 tokens (per rounded up to a power of two); the mma.sync path also splits long contexts
    # below six waves, into partitions of at most 2048 tokens
    from paged_kv_decode_21_gb300 import ops
    sms = 148  # no device here: the library's default SM count
    # GQA 7:1, 256 x 8192 tokens, q_len 8: 1024 units, three waves and more, unsplit and walked
    # longest first; the last round of 296 slots holds 1024 - 3 * 296 = 136 CTAs, so the order
    # splits the 34 shortest sequences in two (three launches: order, decode, merge)
    n, part, ordered, var, grid, _ = ops.paged_decode_call_plan(256, 8, 28, 4, 128, 16, 8192)
    assert var.startswith("tcgen05") and part == -1 and ordered and n == 3 and grid == (256 + 34) * 4
    n, part, ordered, var, grid, _ = ops.paged_decode_call_plan(256, 8, 28, 4, 128, 16, 8192, variant="tma_mma")
    assert part == -1 and grid == 256 * 4 * 4  # four 16-row chunks: many waves, unsplit too
    n, part, ordered, var, grid, _ = ops.paged_decode_call_plan(256, 1, 28, 4, 128, 16, 8192)
    assert var == "tma_mma" and part == 2048  # single query: 1024 units, long context, split
    # GQA 5:1, 32 x 32768 tokens, q_len 8: 256 units, below two waves: split
    n, part, ordered, var, grid, _ = ops.paged_decode_call_plan(32, 8, 40, 8, 128, 16, 32768)
    want = 6 * 2 * sms
    np_ = -(-want // 256)
    per = -(-32768 // np_)
    p = 512  # the smallest power of two covering per (at most 8192)
    while p < per and p * 2 <= 8192:
        p *= 2
    assert var == "tcgen05" and part == p and part > 2048
    # a longest context just below 32768 takes the same partition (per just below a power of
    # two rounds up to it, not down to half of it)
    assert ops.paged_decode_call_plan(32, 8, 40, 8, 128, 16, 32700)[1] == p
