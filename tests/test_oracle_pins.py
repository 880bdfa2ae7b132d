"""Pins of the CPU oracle against facts fixed outside it.

Each ``pin_*`` function checks the oracle (optionally a build with a planted
mistake, ``mutant``) against something the pages or the mathematics fix:
numpy's binary16 decoding, torch's scaled_dot_product_attention over
contiguous K/V, closed forms (mean of V, a single token, a one-token spike),
invariants (block permutation, weights summing to one, GQA == repeated MHA,
masking), and the log-sum-exp identity for the partition merge.  The mutation
test at the bottom requires every planted mistake to fail at least one pin.
"""
import math

import numpy as np
import pytest
import torch

import oracle

TOL = 1e-12


# ---------------------------------------------------------------------------
# Input construction independent of the oracle's gather: logical per-sequence
# K/V rows are scattered into a pool through an explicit block permutation.
# ---------------------------------------------------------------------------
def scatter_problem(seed, lens, Hq, Hkv, D, BS, extra_blocks=3, mbps=None, logical_k=None,
                    logical_v=None, q=None, pool_fill=None):
    rng = np.random.default_rng(seed)
    B = len(lens)
    nbs = [-(-L // BS) for L in lens]
    needed = sum(nbs)
    NB = needed + extra_blocks
    mbps = mbps or max(1, max(nbs) if nbs else 1)
    perm = rng.permutation(NB)[:needed]
    if pool_fill is None:
        kp = rng.standard_normal((NB, Hkv, BS, D)).astype(np.float16)
        vp = rng.standard_normal((NB, Hkv, BS, D)).astype(np.float16)
    else:
        kp = np.full((NB, Hkv, BS, D), pool_fill, np.float16)
        vp = np.full((NB, Hkv, BS, D), pool_fill, np.float16)
    if logical_k is None:
        logical_k = [rng.standard_normal((Hkv, L, D)).astype(np.float16) for L in lens]
    if logical_v is None:
        logical_v = [rng.standard_normal((Hkv, L, D)).astype(np.float16) for L in lens]
    if q is None:
        q = rng.standard_normal((B, Hq, D)).astype(np.float16)
    bt = np.full((B, mbps), -1, np.int32)
    pos = 0
    for b, L in enumerate(lens):
        for i in range(nbs[b]):
            p = int(perm[pos]); pos += 1
            bt[b, i] = p
            t0, t1 = i * BS, min(L, (i + 1) * BS)
            kp[p, :, : t1 - t0, :] = logical_k[b][:, t0:t1, :]
            vp[p, :, : t1 - t0, :] = logical_v[b][:, t0:t1, :]
    cl = np.array(lens, np.int32)
    return dict(q=q, k=kp, v=vp, bt=bt, cl=cl, lk=logical_k, lv=logical_v, perm=perm, NB=NB)


def run(pr, scale, mutant=0, **kw):
    return oracle.attention(pr["q"], pr["k"], pr["v"], pr["bt"], pr["cl"], scale, mutant=mutant, **kw)


def sdpa_reference(pr, scale, Hq, Hkv):
    """torch's scaled_dot_product_attention in fp64 over contiguous K/V."""
    G = Hq // Hkv
    outs = []
    for b, L in enumerate(pr["cl"]):
        D = pr["q"].shape[2]
        if L == 0:
            outs.append(np.zeros((Hq, D)))
            continue
        q = torch.from_numpy(pr["q"][b].astype(np.float64)).view(1, Hq, 1, D)
        k = torch.from_numpy(pr["lk"][b].astype(np.float64)).repeat_interleave(G, 0).view(1, Hq, L, D)
        v = torch.from_numpy(pr["lv"][b].astype(np.float64)).repeat_interleave(G, 0).view(1, Hq, L, D)
        o = torch.nn.functional.scaled_dot_product_attention(q, k, v, scale=scale)
        outs.append(o.view(Hq, D).numpy())
    return np.stack(outs)


# ---------------------------------------------------------------------------
# Pins
# ---------------------------------------------------------------------------
def pin_half_decoder(mutant=0):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = oracle.half_to_double(bits)
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(ref[~nan], got[~nan])


def pin_sdpa_contiguous(mutant=0):
    for seed, (lens, Hq, Hkv, D, BS) in enumerate([
        ((37, 100), 4, 4, 64, 16),
        ((1, 5, 16, 33), 8, 2, 32, 4),
        ((70, 9, 48), 14, 2, 16, 8),
        ((17,), 6, 3, 8, 16),
    ]):
        pr = scatter_problem(100 + seed, list(lens), Hq, Hkv, D, BS)
        scale = 1.0 / math.sqrt(D)
        got = run(pr, scale, mutant)
        ref = sdpa_reference(pr, scale, Hq, Hkv)
        assert np.max(np.abs(got - ref)) <= TOL * max(1.0, np.max(np.abs(ref)))


def pin_permutation_invariance(mutant=0):
    lens, Hq, Hkv, D, BS = [23, 64, 50], 6, 2, 16, 8
    base = scatter_problem(7, lens, Hq, Hkv, D, BS)
    other = scatter_problem(8, lens, Hq, Hkv, D, BS, logical_k=base["lk"], logical_v=base["lv"],
                            q=base["q"])
    assert not np.array_equal(base["bt"], other["bt"])
    a = run(base, 0.25, mutant)
    b = run(other, 0.25, mutant)
    assert np.array_equal(a, b)


def pin_weights_sum_to_one(mutant=0):
    lens, Hq, Hkv, D, BS = [45, 3], 4, 2, 16, 16
    pr = scatter_problem(11, lens, Hq, Hkv, D, BS)
    for b, L in enumerate(lens):
        for h in range(Hq):
            w = oracle.weights(pr["q"], pr["k"], pr["v"], pr["bt"], pr["cl"], 0.25, b, h,
                               mutant=mutant)
            assert w.shape == (L,)
            assert np.all(w >= 0)
            assert abs(w.sum() - 1.0) <= TOL


def pin_identical_keys_mean_of_v(mutant=0):
    lens, Hq, Hkv, D, BS = [29, 64, 7], 4, 2, 16, 8
    rng = np.random.default_rng(5)
    row = rng.standard_normal(D).astype(np.float16)
    lk = [np.broadcast_to(row, (Hkv, L, D)).copy() for L in lens]
    pr = scatter_problem(12, lens, Hq, Hkv, D, BS, logical_k=lk)
    got = run(pr, 0.3, mutant)
    G = Hq // Hkv
    for b in range(len(lens)):
        for h in range(Hq):
            ref = pr["lv"][b][h // G].astype(np.float64).mean(axis=0)
            assert np.max(np.abs(got[b, h] - ref)) <= TOL


def pin_scale_zero_mean_of_v(mutant=0):
    lens, Hq, Hkv, D, BS = [31, 16], 4, 4, 8, 16
    pr = scatter_problem(13, lens, Hq, Hkv, D, BS)
    got = run(pr, 0.0, mutant)
    for b in range(len(lens)):
        for h in range(Hq):
            ref = pr["lv"][b][h].astype(np.float64).mean(axis=0)
            assert np.max(np.abs(got[b, h] - ref)) <= TOL


def pin_single_token(mutant=0):
    lens, Hq, Hkv, D, BS = [1, 1, 1], 6, 3, 16, 16
    pr = scatter_problem(14, lens, Hq, Hkv, D, BS)
    got = run(pr, 0.25, mutant)
    G = Hq // Hkv
    for b in range(3):
        for h in range(Hq):
            assert np.array_equal(got[b, h], pr["lv"][b][h // G][0].astype(np.float64))


def pin_spike_every_position(mutant=0):
    L, Hq, Hkv, D, BS = 37, 2, 1, 16, 16
    for t_star in range(L):
        q = np.ones((1, Hq, D), np.float16)
        rng = np.random.default_rng(1000 + t_star)
        lk = [rng.standard_normal((Hkv, L, D)).astype(np.float16)]
        lk[0][:, t_star, :] = 1000.0
        pr = scatter_problem(15 + t_star, [L], Hq, Hkv, D, BS, logical_k=lk, q=q)
        got = run(pr, 0.25, mutant)
        ref = pr["lv"][0][0, t_star].astype(np.float64)
        for h in range(Hq):
            assert np.array_equal(got[0, h], ref), t_star


def pin_gqa_equals_repeated_mha(mutant=0):
    lens, Hq, Hkv, D, BS = [40, 19], 14, 2, 16, 8
    pr = scatter_problem(16, lens, Hq, Hkv, D, BS)
    G = Hq // Hkv
    mha = dict(pr)
    mha["k"] = np.repeat(pr["k"], G, axis=1)
    mha["v"] = np.repeat(pr["v"], G, axis=1)
    a = run(pr, 0.25, mutant)
    b = run(mha, 0.25, mutant)
    assert np.array_equal(a, b)


def pin_context_zero(mutant=0):
    pr = scatter_problem(17, [0, 5], 2, 2, 8, 4, mbps=2)
    got = run(pr, 0.5, mutant)
    assert np.array_equal(got[0], np.zeros((2, 8)))


def pin_nan_poison_ignored(mutant=0):
    lens, Hq, Hkv, D, BS = [21, 9], 4, 2, 16, 8
    clean = scatter_problem(18, lens, Hq, Hkv, D, BS)
    poison = scatter_problem(18, lens, Hq, Hkv, D, BS, logical_k=clean["lk"], logical_v=clean["lv"],
                             q=clean["q"], pool_fill=np.nan)
    # unused pool blocks and tail slots hold NaN, used rows are identical
    assert np.isnan(poison["k"]).any()
    a = run(clean, 0.25, mutant)
    b = run(poison, 0.25, mutant)
    assert np.all(np.isfinite(b))
    assert np.array_equal(a, b)


def pin_partition_merge(mutant=0):
    lens, Hq, Hkv, D, BS, P = [100, 33, 64, 1, 0], 6, 2, 16, 16, 32
    pr = scatter_problem(19, lens, Hq, Hkv, D, BS, mbps=8)
    full = run(pr, 0.25, mutant)
    m, l, o = oracle.partitions(pr["q"], pr["k"], pr["v"], pr["bt"], pr["cl"], 0.25, P,
                                mutant=mutant)
    merged = oracle.merge(m, l, o, pr["cl"], P, mutant=mutant)
    assert np.max(np.abs(merged - full)) <= TOL


def pin_partition_counts_scale_zero(mutant=0):
    lens, Hq, Hkv, D, BS, P = [100, 32, 1, 64, 0], 2, 1, 8, 16, 32
    pr = scatter_problem(20, lens, Hq, Hkv, D, BS, mbps=8)
    m, l, o = oracle.partitions(pr["q"], pr["k"], pr["v"], pr["bt"], pr["cl"], 0.0, P,
                                max_partitions=4, mutant=mutant)
    for b, L in enumerate(lens):
        for j in range(4):
            expect = max(0, min(P, L - j * P))
            assert np.all(l[b, :, j] == expect), (b, j, l[b, :, j])
            if expect == 0:
                assert np.all(np.isneginf(m[b, :, j]))
            else:
                assert np.all(m[b, :, j] == 0.0)


def pin_partition_max_is_max_score(mutant=0):
    lens, Hq, Hkv, D, BS, P = [70], 2, 2, 16, 16, 32
    pr = scatter_problem(21, lens, Hq, Hkv, D, BS)
    m, l, o = oracle.partitions(pr["q"], pr["k"], pr["v"], pr["bt"], pr["cl"], 0.25, P,
                                mutant=mutant)
    for h in range(Hq):
        q = pr["q"][0, h].astype(np.float64)
        k = pr["lk"][0][h].astype(np.float64)
        s = 0.25 * (k @ q)
        for j in range(m.shape[2]):
            seg = s[j * P: (j + 1) * P]
            assert abs(m[0, h, j] - seg.max()) <= TOL
            assert abs(l[0, h, j] - np.exp(seg - seg.max()).sum()) <= TOL * len(seg)


def pin_append_then_attend(mutant=0):
    # the first L tokens are scattered independently; the oracle appends token L;
    # attention over L+1 tokens must equal SDPA over the grown logical sequence
    for seed, (lens, Hq, Hkv, D, BS) in enumerate([((15, 16, 17, 0, 31), 6, 3, 16, 16),
                                                   ((7, 8, 1), 4, 4, 8, 8)]):
        rng = np.random.default_rng(300 + seed)
        full = [L + 1 for L in lens]
        grown = scatter_problem(400 + seed, full, Hq, Hkv, D, BS, mbps=4)
        before = dict(grown)
        # the pool as it was before the append: the new slot holds noise
        k_old, v_old = grown["k"].copy(), grown["v"].copy()
        for b, L in enumerate(lens):
            p = grown["bt"][b, L // BS]
            k_old[p, :, L % BS, :] = rng.standard_normal((Hkv, D)).astype(np.float16)
            v_old[p, :, L % BS, :] = rng.standard_normal((Hkv, D)).astype(np.float16)
        k_new = np.stack([grown["lk"][b][:, L, :] for b, L in enumerate(lens)])
        v_new = np.stack([grown["lv"][b][:, L, :] for b, L in enumerate(lens)])
        kc, vc = oracle.append(k_new, v_new, grown["bt"], np.array(lens, np.int32), k_old, v_old,
                               mutant=mutant)
        after = dict(before, k=kc, v=vc)
        scale = 1.0 / math.sqrt(D)
        got = run(after, scale, mutant)
        ref = sdpa_reference(grown, scale, Hq, Hkv)
        assert np.max(np.abs(got - ref)) <= TOL * max(1.0, np.max(np.abs(ref)))


def pin_append_changes_one_row_per_head(mutant=0):
    lens, Hkv, D, BS = [5, 16, 0], 2, 8, 16
    pr = scatter_problem(500, [L + 1 for L in lens], 2, Hkv, D, BS, mbps=3)
    rng = np.random.default_rng(501)
    k_new = rng.standard_normal((3, Hkv, D)).astype(np.float16)
    v_new = rng.standard_normal((3, Hkv, D)).astype(np.float16)
    kc, vc = oracle.append(k_new, v_new, pr["bt"], np.array(lens, np.int32), pr["k"], pr["v"],
                           mutant=mutant)
    changed = np.zeros(pr["k"].shape[:3], bool)
    for b, L in enumerate(lens):
        p = pr["bt"][b, L // BS]
        changed[p, :, L % BS] = True
        assert np.array_equal(kc[p, :, L % BS], k_new[b])
        assert np.array_equal(vc[p, :, L % BS], v_new[b])
    assert np.array_equal(kc[~changed], pr["k"][~changed])
    assert np.array_equal(vc[~changed], pr["v"][~changed])


def multi_problem(seed, lens, q_len, Hq, Hkv, D, BS):
    pr = scatter_problem(seed, lens, Hq, Hkv, D, BS)
    rng = np.random.default_rng(seed + 1)
    pr["qm"] = rng.standard_normal((len(lens), q_len, Hq, D)).astype(np.float16)
    return pr


def causal_sdpa_reference(pr, scale, Hq, Hkv):
    """SDPA in fp64 with an explicit boolean mask: query jq of a sequence of
    length L sits at position L - q_len + jq and sees keys t <= that position;
    rows that see no key are zero."""
    G = Hq // Hkv
    B, QL, _, D = pr["qm"].shape
    out = np.zeros((B, QL, Hq, D))
    for b, L in enumerate(pr["cl"]):
        L = int(L)
        if L == 0:
            continue
        q = torch.from_numpy(pr["qm"][b].astype(np.float64)).permute(1, 0, 2).reshape(1, Hq, QL, D)
        k = torch.from_numpy(pr["lk"][b].astype(np.float64)).repeat_interleave(G, 0).view(1, Hq, L, D)
        v = torch.from_numpy(pr["lv"][b].astype(np.float64)).repeat_interleave(G, 0).view(1, Hq, L, D)
        pos = torch.arange(QL).view(QL, 1) + (L - QL)
        mask = torch.arange(L).view(1, L) <= pos
        o = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=mask, scale=scale)
        o = o.view(Hq, QL, D).permute(1, 0, 2).numpy()
        seen = mask.any(dim=1).numpy()
        out[b][seen] = o[seen]
    return out


def pin_multi_query_causal_sdpa(mutant=0):
    for seed, (lens, q_len, Hq, Hkv, D, BS) in enumerate([
        ((37, 100, 4), 4, 8, 2, 32, 16),
        ((16, 17, 9), 7, 7, 1, 16, 8),
        ((2, 30), 4, 4, 4, 8, 4),          # the first sequence is shorter than q_len
        ((50,), 2, 6, 3, 16, 16),
    ]):
        pr = multi_problem(600 + seed, list(lens), q_len, Hq, Hkv, D, BS)
        scale = 1.0 / math.sqrt(D)
        got = oracle.attention_multi(pr["qm"], pr["k"], pr["v"], pr["bt"], pr["cl"], scale, mutant=mutant)
        ref = causal_sdpa_reference(pr, scale, Hq, Hkv)
        assert np.max(np.abs(got - ref)) <= TOL * max(1.0, np.max(np.abs(ref)))


def pin_multi_query_ignores_the_future(mutant=0):
    # query jq's output cannot depend on tokens after its position; the next
    # query (which sees one more token) does
    lens, q_len, Hq, Hkv, D, BS = [40], 5, 4, 2, 16, 8
    base = multi_problem(700, lens, q_len, Hq, Hkv, D, BS)
    scale = 0.3
    a = oracle.attention_multi(base["qm"], base["k"], base["v"], base["bt"], base["cl"], scale, mutant=mutant)
    L = lens[0]
    for jq in range(q_len - 1):
        pos = L - q_len + jq
        lk = [base["lk"][0].copy()]
        lv = [base["lv"][0].copy()]
        lk[0][:, pos + 1:, :] = np.float16(3.0)
        lv[0][:, pos + 1:, :] = np.float16(-2.0)
        other = scatter_problem(700, lens, Hq, Hkv, D, BS, logical_k=lk, logical_v=lv, q=base["q"])
        b = oracle.attention_multi(base["qm"], other["k"], other["v"], other["bt"], other["cl"], scale,
                                   mutant=mutant)
        assert np.array_equal(a[0, : jq + 1], b[0, : jq + 1])
        assert not np.allclose(a[0, jq + 1], b[0, jq + 1])


def pin_multi_query_last_is_single_query(mutant=0):
    # the last new token sees the whole context: plain decode of that query
    lens, q_len, Hq, Hkv, D, BS = [33, 64, 5], 3, 6, 2, 16, 16
    pr = multi_problem(800, lens, q_len, Hq, Hkv, D, BS)
    got = oracle.attention_multi(pr["qm"], pr["k"], pr["v"], pr["bt"], pr["cl"], 0.25, mutant=mutant)
    single = oracle.attention(np.ascontiguousarray(pr["qm"][:, -1]), pr["k"], pr["v"], pr["bt"], pr["cl"],
                              0.25, mutant=mutant)
    assert np.array_equal(got[:, -1], single)


def torch_e4m3_to_f64(codes):
    t = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8))
    return t.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def pin_e4m3_decoder(mutant=0):
    codes = np.arange(256, dtype=np.uint8)
    got = oracle.e4m3_to_double(codes, mutant=mutant)
    ref = torch_e4m3_to_f64(codes)
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got)) and nan.sum() == 2      # 0x7f and 0xff
    assert np.array_equal(ref[~nan], got[~nan])
    assert got[0x7e] == 448.0 and got[0x01] == 2.0 ** -9 and got[0x38] == 1.0


def pin_e4m3_rounding(mutant=0):
    # every finite binary16 value, at two scales: nearest-even rounding of the
    # fp32 quotient onto the E4M3 grid, compared with torch's conversion where
    # it does not overflow; beyond, the oracle saturates to +-448
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    x = bits.view(np.float16)
    fin = np.isfinite(x)
    x = x[fin]
    for scale in (1.0, 0.0625, 3.0):
        got = oracle.quantize_e4m3(x, scale, mutant=mutant)
        qf = torch.from_numpy(x.astype(np.float32)) / torch.tensor(scale, dtype=torch.float32)
        inr = (qf.abs() < 464.0).numpy()
        ref = qf.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert np.array_equal(got[inr], ref[inr])
        big = ~inr
        assert np.all(got[big] == np.where(qf.numpy()[big] < 0, 0xFE, 0x7E))
    # ties to even at the smallest step: 0.5 and 1.5 units of 2^-9
    t = oracle.float_to_e4m3(np.array([2.0 ** -10, 1.5 * 2.0 ** -9, 2.5 * 2.0 ** -9], np.float32), mutant=mutant)
    assert t.tolist() == [0x00, 0x02, 0x02]


def fp8_problem(seed, lens, q_len, Hq, Hkv, D, BS):
    rng = np.random.default_rng(seed)
    B = len(lens)
    nbs = [-(-L // BS) for L in lens]
    NB = sum(nbs) + 2
    perm = rng.permutation(NB)[:sum(nbs)]
    def codes(shape):  # any finite E4M3 code
        c = rng.integers(0, 0x7f, size=shape, dtype=np.uint8)
        return (c | (rng.integers(0, 2, size=shape, dtype=np.uint8) << 7)).astype(np.uint8)
    k8 = codes((NB, Hkv, BS, D))
    v8 = codes((NB, Hkv, BS, D))
    lk = [codes((Hkv, L, D)) for L in lens]
    lv = [codes((Hkv, L, D)) for L in lens]
    bt = np.full((B, max(1, max(nbs))), -1, np.int32)
    pos = 0
    for b, L in enumerate(lens):
        for i in range(nbs[b]):
            p = int(perm[pos]); pos += 1
            bt[b, i] = p
            t0, t1 = i * BS, min(L, (i + 1) * BS)
            k8[p, :, : t1 - t0] = lk[b][:, t0:t1]
            v8[p, :, : t1 - t0] = lv[b][:, t0:t1]
    q = rng.standard_normal((B, q_len, Hq, D)).astype(np.float16)
    return dict(q=q, k8=k8, v8=v8, bt=bt, cl=np.array(lens, np.int32), lk=lk, lv=lv)


def pin_fp8_attention_sdpa(mutant=0):
    for seed, (lens, q_len, Hq, Hkv, D, BS, ks, vs) in enumerate([
        ((37, 100, 5), 1, 8, 2, 32, 16, 0.05, 0.11),
        ((20, 64), 3, 4, 4, 16, 8, 0.02, 0.3),
    ]):
        pr = fp8_problem(900 + seed, list(lens), q_len, Hq, Hkv, D, BS)
        scale = 1.0 / math.sqrt(D)
        got = oracle.attention_fp8(pr["q"], pr["k8"], pr["v8"], pr["bt"], pr["cl"], scale, ks, vs, mutant=mutant)
        # reference: torch decodes the logical codes; SDPA with the causal mask
        fp = dict(qm=pr["q"], cl=pr["cl"],
                  lk=[torch_e4m3_to_f64(k) * ks for k in pr["lk"]],
                  lv=[torch_e4m3_to_f64(v) * vs for v in pr["lv"]])
        ref = causal_sdpa_reference(fp, scale, Hq, Hkv)
        assert np.max(np.abs(got - ref)) <= TOL * max(1.0, np.max(np.abs(ref)))


def pin_fp8_append(mutant=0):
    lens, Hkv, D, BS = [5, 16, 0], 2, 16, 16
    pr = fp8_problem(950, [L + 1 for L in lens], 1, 2, Hkv, D, BS)
    rng = np.random.default_rng(951)
    k_new = (rng.standard_normal((3, Hkv, D)) * 3).astype(np.float16)
    v_new = (rng.standard_normal((3, Hkv, D)) * 3).astype(np.float16)
    ks, vs = 0.03, 0.5
    kc, vc = oracle.append_fp8(k_new, v_new, pr["bt"], np.array(lens, np.int32), pr["k8"], pr["v8"], ks, vs,
                               mutant=mutant)
    q = lambda x, sc: (torch.from_numpy(x.astype(np.float32)) / torch.tensor(sc, dtype=torch.float32)
                       ).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    changed = np.zeros(kc.shape[:3], bool)
    for b, L in enumerate(lens):
        p = pr["bt"][b, L // BS]
        changed[p, :, L % BS] = True
        assert np.array_equal(kc[p, :, L % BS], q(k_new[b], ks))
        assert np.array_equal(vc[p, :, L % BS], q(v_new[b], vs))
    assert np.array_equal(kc[~changed], pr["k8"][~changed])
    assert np.array_equal(vc[~changed], pr["v8"][~changed])


PINS = [pin_half_decoder, pin_sdpa_contiguous, pin_permutation_invariance, pin_weights_sum_to_one,
        pin_identical_keys_mean_of_v, pin_scale_zero_mean_of_v, pin_single_token,
        pin_spike_every_position, pin_gqa_equals_repeated_mha, pin_context_zero,
        pin_nan_poison_ignored, pin_partition_merge, pin_partition_counts_scale_zero,
        pin_partition_max_is_max_score, pin_append_then_attend, pin_append_changes_one_row_per_head,
        pin_multi_query_causal_sdpa, pin_multi_query_ignores_the_future, pin_multi_query_last_is_single_query,
        pin_e4m3_decoder, pin_e4m3_rounding, pin_fp8_attention_sdpa, pin_fp8_append]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_oracle_pin(pin):
    pin(0)


def test_threads_do_not_change_result():
    pr = scatter_problem(30, [77, 5, 130], 8, 2, 32, 16)
    a = run(pr, 0.2, threads=1)
    b = run(pr, 0.2, threads=7)
    assert np.array_equal(a, b)


def test_row_selection_matches_full():
    pr = scatter_problem(31, [40, 12], 4, 2, 16, 8)
    full = run(pr, 0.3)
    rows = np.array([5, 0, 7, 2], np.int32)
    sel = run(pr, 0.3, rows=rows)
    for i, r in enumerate(rows):
        assert np.array_equal(sel[i], full[r // 4, r % 4])


def test_append_without_room_is_reported():
    pr = scatter_problem(33, [32], 2, 2, 8, 16, mbps=2)
    k_new = np.zeros((1, 2, 8), np.float16)
    with pytest.raises(oracle.OracleError):
        oracle.append(k_new, k_new, pr["bt"], np.array([32], np.int32), pr["k"], pr["v"])


def test_bad_block_id_is_reported():
    pr = scatter_problem(32, [20], 2, 2, 8, 16)
    pr["bt"][0, 1] = pr["NB"] + 5
    with pytest.raises(oracle.OracleError):
        run(pr, 0.3)


MUTANTS = list(range(1, 12))


@pytest.mark.parametrize("mutant", MUTANTS)
def test_planted_mistake_fails_a_pin(mutant):
    assert oracle.mutant_id(mutant) == mutant
    failed = []
    for pin in PINS:
        if pin is pin_half_decoder:
            continue
        try:
            pin(mutant)
        except (AssertionError, oracle.OracleError):
            failed.append(pin.__name__)
    assert failed, f"planted mistake {mutant} passed every pin"
