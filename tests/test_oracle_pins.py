"""Pins for the CPU oracle: each test checks it against something other than
itself -- the pages' worked examples (tests/golden), closed forms, invariants
the pages state, library routines (scipy / torch) on special cases, and brute
force on tiny inputs laid out contiguously instead of through a block table.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch
from scipy.special import logsumexp, softmax

import oracle
import workloads
from tests._util import bf16_values, bits, golden


def rand_case(seed, B, Hq, Hkv, D, bs, lens, dv=None, extra_blocks=3):
    """Random small paged cache: per sequence, blocks drawn from a shuffled pool."""
    dv = dv or D
    rng = np.random.default_rng(seed)
    counts = [-(-n // bs) for n in lens]
    nb = sum(counts) + extra_blocks
    perm = rng.permutation(nb)
    width = max(max(counts), 1)
    tables = np.full((B, width), -1, dtype=np.int32)
    at = 0
    for b, c in enumerate(counts):
        tables[b, :c] = perm[at:at + c]
        at += c
    k = bits(torch.from_numpy(rng.standard_normal((nb, Hkv, bs, D))).to(torch.bfloat16))
    v = bits(torch.from_numpy(rng.standard_normal((nb, Hkv, bs, dv))).to(torch.bfloat16))
    q = rng.standard_normal((B, Hq, D)).astype(np.float32)
    return q, k, v, tables, np.array(lens, dtype=np.int32)


def brute_force(q, k_bits, v_bits, tables, lens, scale):
    """Contiguous attention: rebuild each sequence's K/V in logical order with
    numpy fancy indexing, then softmax / logsumexp from scipy."""
    B, Hq, D = q.shape
    nb, Hkv, bs, _ = k_bits.shape
    dv = v_bits.shape[3]
    K = bf16_values(k_bits)
    V = bf16_values(v_bits)
    out = np.zeros((B, Hq, dv))
    lse = np.full((B, Hq), -np.inf)
    for b in range(B):
        L = int(lens[b])
        if L == 0:
            continue
        idx = np.arange(L)
        phys = tables[b][idx // bs]
        off = idx % bs
        for h in range(Hq):
            g = h // (Hq // Hkv)
            Kc = K[phys, g, off, :]            # [L, D] logical order
            Vc = V[phys, g, off, :]
            s = scale * (Kc @ q[b, h].astype(np.float64))
            out[b, h] = softmax(s) @ Vc
            lse[b, h] = logsumexp(s)
    return out, lse


# ---------------------------------------------------------------- bf16 decode

def test_bf16_decode_all_patterns_match_torch():
    allbits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = bf16_values(allbits)
    got = np.array([oracle.bf16_to_double(int(b)) for b in allbits[::97]])
    r = ref[::97]
    nan = np.isnan(r)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], r[~nan])
    assert oracle.bf16_to_double(0x3F80) == 1.0
    assert oracle.bf16_to_double(0xC000) == -2.0
    assert oracle.bf16_to_double(0x0001) == 2.0 ** -133
    assert oracle.bf16_to_double(0x7F80) == math.inf


# ------------------------------------------------------ pages' worked examples

def test_block_accounting_example():
    gd = golden("block_accounting.txt")
    bs = gd["block_size"]
    a = oracle.blocks_needed(gd["tokens_A"], bs)
    b = oracle.blocks_needed(gd["tokens_B"], bs)
    assert (a, b) == (gd["blocks_A"], gd["blocks_B"])
    assert gd["tokens_A"] + gd["tokens_B"] == gd["total_tokens"]
    assert (a + b) * bs == gd["total_slots"]
    assert (a + b) * bs - gd["total_tokens"] == gd["slack_slots"]
    assert oracle.blocks_needed(gd["B_grown_tokens"], bs) == gd["B_grown_blocks"]
    assert oracle.blocks_needed(gd["B_next_tokens"], bs) == gd["B_next_blocks"]
    assert oracle.blocks_needed(0, bs) == 0


def test_block_accounting_slots_follow_table():
    """B's 9 tokens in 3 scattered blocks: token j sits in logical block j // 4."""
    gd = golden("block_accounting.txt")
    bs = gd["block_size"]
    table_b = np.array([5, 0, 6], dtype=np.int32)   # scattered physical blocks
    slots = [oracle.slot_of(table_b, j, bs) for j in range(gd["tokens_B"])]
    assert slots == [20, 21, 22, 23, 0, 1, 2, 3, 24]


def test_kv_bytes_per_token_example():
    gd = golden("kv_bytes_per_token.txt")
    n = oracle.kv_bytes_per_token(gd["layers"], gd["kv_heads"], gd["head_dim"],
                                  gd["bytes_per_number"])
    assert n == gd["bytes_per_token"] == gd["kib_per_token"] * 1024
    assert gd["conversation_tokens"] * n == gd["conversation_mib"] * 2 ** 20


@pytest.mark.parametrize("interleave", [1, 16])
def test_interleave_200k_over_4(interleave):
    gd = golden("dcp_interleave.txt")
    N, P = gd["num_tokens"], gd["dcp_size"]
    part, local = oracle.interleave(N, P, interleave)
    counts = np.bincount(part, minlength=P)
    assert counts.tolist() == [gd["tokens_per_partition"]] * P
    # not contiguous ranges: every partition appears within the first P*I tokens
    assert set(part[:P * interleave].tolist()) == set(range(P))
    # order kept inside each partition: local positions run 0..n-1 in token order
    for r in range(P):
        assert np.array_equal(local[part == r], np.arange(counts[r]))


def test_interleave_size_one_is_token_mod_p():
    """The page's interleave-1 statement: token i goes to GPU i mod DCP size."""
    part, _ = oracle.interleave(1000, 4, 1)
    assert np.array_equal(part, np.arange(1000) % 4)


def test_interleave_groups_rotate():
    """Interleave I: runs of I consecutive tokens share a partition and
    successive runs go to successive partitions (mod P); ragged last run."""
    N, P, I = 1000, 3, 7
    part, local = oracle.interleave(N, P, I)
    runs = [part[s:s + I] for s in range(0, N, I)]
    for c, run in enumerate(runs):
        assert (run == run[0]).all()
        if c:
            assert run[0] == (runs[c - 1][0] + 1) % P
    assert runs[0][0] == 0
    assert sum(np.bincount(part, minlength=P)) == N


# ------------------------------------------------------- attention values

@pytest.mark.parametrize("seed,B,Hq,Hkv,D,bs,lens", [
    (0, 2, 4, 2, 64, 4, [7, 10]),
    (1, 3, 8, 8, 16, 16, [1, 17, 33]),
    (2, 4, 6, 2, 8, 3, [5, 0, 9, 2]),
    (3, 1, 8, 1, 12, 5, [23]),
])
def test_attention_matches_contiguous_brute_force(seed, B, Hq, Hkv, D, bs, lens):
    q, k, v, tables, L = rand_case(seed, B, Hq, Hkv, D, bs, lens)
    scale = 1.0 / math.sqrt(D)
    out, lse = oracle.paged_decode_attn(q, k, v, tables, L, scale)
    ref_o, ref_l = brute_force(q, k, v, tables, L, scale)
    np.testing.assert_allclose(out, ref_o, rtol=0, atol=1e-12)
    finite = np.isfinite(ref_l)
    np.testing.assert_allclose(lse[finite], ref_l[finite], rtol=0, atol=1e-12)
    assert np.array_equal(np.isneginf(lse), ~finite)


def test_attention_tiny_workload_matches_brute_force():
    w = workloads.tiny()
    q = w.q.numpy()
    k, v = bits(w.k_pool), bits(w.v_pool)
    t, L = w.block_tables.numpy(), w.seq_lens.numpy()
    out, lse = oracle.paged_decode_attn(q, k, v, t, L, w.scale)
    ro, rl = brute_force(q, k, v, t, L, w.scale)
    np.testing.assert_allclose(out, ro, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, rl, rtol=0, atol=1e-12)


def test_attention_distinct_value_dim():
    q, k, v, tables, L = rand_case(9, 2, 4, 1, 24, 8, [13, 30], dv=10)
    out, lse = oracle.paged_decode_attn(q, k, v, tables, L, 0.3)
    ro, rl = brute_force(q, k, v, tables, L, 0.3)
    assert out.shape == (2, 4, 10)
    np.testing.assert_allclose(out, ro, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, rl, rtol=0, atol=1e-12)


def test_physical_placement_does_not_change_result():
    """Relabel every physical block (pool and tables together): identical bits."""
    q, k, v, tables, L = rand_case(4, 3, 8, 2, 32, 4, [9, 22, 14])
    out, lse = oracle.paged_decode_attn(q, k, v, tables, L, 0.2)
    rng = np.random.default_rng(44)
    nb = k.shape[0]
    new_of_old = rng.permutation(nb)
    k2 = np.empty_like(k)
    v2 = np.empty_like(v)
    k2[new_of_old] = k
    v2[new_of_old] = v
    t2 = np.where(tables >= 0, new_of_old[np.maximum(tables, 0)], -1).astype(np.int32)
    out2, lse2 = oracle.paged_decode_attn(q, k2, v2, t2, L, 0.2)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def _small_int_bf16(vals):
    return bits(torch.tensor(vals, dtype=torch.float64).to(torch.bfloat16))


def test_single_token_returns_its_value_and_score():
    D = 8
    k = _small_int_bf16(np.arange(D).reshape(1, 1, 1, D) - 3.0)
    v = _small_int_bf16(np.arange(D).reshape(1, 1, 1, D) * 0.5 + 1.0)
    q = np.ones((1, 1, D), dtype=np.float32)
    out, lse = oracle.paged_decode_attn(q, k, v, np.array([[0]], np.int32),
                                        np.array([1], np.int32), 0.5)
    assert np.array_equal(out[0, 0], np.arange(D) * 0.5 + 1.0)
    assert lse[0, 0] == 0.5 * float(np.sum(np.arange(D) - 3.0))


def test_identical_keys_give_mean_value_and_log_count():
    L, D, bs = 11, 4, 4
    nb = 3
    krow = np.array([1.0, -2.0, 0.5, 3.0])
    k = _small_int_bf16(np.broadcast_to(krow, (nb, 1, bs, D)).copy())
    rng = np.random.default_rng(5)
    v = bits(torch.from_numpy(rng.standard_normal((nb, 1, bs, D))).to(torch.bfloat16))
    q = np.array([[[0.25, 1.0, -2.0, 0.5]]], dtype=np.float32)
    tables = np.array([[2, 0, 1]], np.int32)
    out, lse = oracle.paged_decode_attn(q, k, v, tables, np.array([L], np.int32), 1.0)
    V = bf16_values(v)
    rows = [V[tables[0, j // bs], 0, j % bs] for j in range(L)]
    mean = np.array([math.fsum(r[d] for r in rows) / L for d in range(D)])
    s = float(np.dot(q[0, 0].astype(np.float64), krow))
    np.testing.assert_allclose(out[0, 0], mean, rtol=0, atol=1e-15)
    assert abs(lse[0, 0] - (s + math.log(L))) < 1e-14


def test_dominant_key_selects_its_value():
    D, bs, L = 4, 2, 6
    kvals = np.zeros((3, 1, bs, D))
    kvals[1, 0, 1, 0] = 64.0           # logical token 3 (table [2, 1, 0])
    k = _small_int_bf16(kvals)
    rng = np.random.default_rng(6)
    v = bits(torch.from_numpy(rng.standard_normal((3, 1, bs, D))).to(torch.bfloat16))
    q = np.array([[[1.0, 0, 0, 0]]], dtype=np.float32)
    out, lse = oracle.paged_decode_attn(q, k, v, np.array([[2, 1, 0]], np.int32),
                                        np.array([L], np.int32), 1.0)
    V = bf16_values(v)
    np.testing.assert_allclose(out[0, 0], V[1, 0, 1], rtol=0, atol=1e-25)
    assert abs(lse[0, 0] - (64.0 + math.log1p(5 * math.exp(-64.0)))) < 1e-14


def test_two_tokens_closed_form():
    D = 2
    k = _small_int_bf16(np.array([[[[1.0, 0.0], [0.0, 2.0]]]]))
    v = _small_int_bf16(np.array([[[[1.0, 2.0], [-4.0, 8.0]]]]))
    q = np.array([[[0.5, 0.25]]], dtype=np.float32)
    out, lse = oracle.paged_decode_attn(q, k, v, np.array([[0]], np.int32),
                                        np.array([2], np.int32), 1.0)
    s0, s1 = 0.5, 0.5
    assert lse[0, 0] == pytest.approx(math.log(math.exp(s0) + math.exp(s1)), abs=1e-15)
    np.testing.assert_allclose(out[0, 0], [-1.5, 5.0], rtol=0, atol=1e-15)


def test_query_group_mapping():
    """Hq=6 over Hkv=3: heads 0,1 read KV head 0; 2,3 head 1; 4,5 head 2."""
    D, bs = 4, 4
    k = np.zeros((1, 3, bs, D))
    v = np.zeros((1, 3, bs, D))
    for g in range(3):
        k[0, g, 0, g] = 4.0        # token 0 scores high only on head-group g
        v[0, g, :, :] = g + 1.0    # every value of KV head g is g + 1
    q = np.ones((1, 6, D), dtype=np.float32)
    out, _ = oracle.paged_decode_attn(q, _small_int_bf16(k), _small_int_bf16(v),
                                      np.array([[0]], np.int32), np.array([3], np.int32), 1.0)
    assert out[0, :, 0].tolist() == [1.0, 1.0, 2.0, 2.0, 3.0, 3.0]


def test_empty_sequence_gives_zero_and_minus_inf():
    q, k, v, tables, _ = rand_case(7, 2, 2, 1, 8, 4, [5, 3])
    out, lse = oracle.paged_decode_attn(q, k, v, tables, np.array([0, 3], np.int32), 1.0)
    assert (out[0] == 0).all() and np.isneginf(lse[0]).all()
    assert np.isfinite(lse[1]).all()


def test_token_range_restricts_attention():
    """A range [b, e) equals attention over a table that starts at token b."""
    bs = 4
    q, k, v, tables, L = rand_case(8, 1, 2, 1, 8, bs, [14])
    out, lse = oracle.paged_decode_attn(q, k, v, tables, L, 1.0,
                                        tok_begin=np.array([4]), tok_end=np.array([11]))
    t2 = tables[:, 1:].copy()            # tokens 4.. are logical blocks 1..
    ro, rl = brute_force(q, k, v, t2, np.array([7]), 1.0)
    np.testing.assert_allclose(out, ro, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, rl, rtol=0, atol=1e-12)


# ------------------------------------------------------------------- merge

def test_merge_of_contiguous_splits_equals_whole():
    q, k, v, tables, L = rand_case(10, 3, 4, 2, 16, 4, [37, 5, 20])
    whole_o, whole_l = oracle.paged_decode_attn(q, k, v, tables, L, 0.25)
    cuts = [0, 6, 13, 13, 40]            # includes an empty split and splits past L
    parts_o, parts_l = [], []
    for s in range(len(cuts) - 1):
        b = np.full(3, cuts[s], np.int32)
        e = np.full(3, cuts[s + 1], np.int32)
        o, l = oracle.paged_decode_attn(q, k, v, tables, L, 0.25, tok_begin=b, tok_end=e)
        parts_o.append(o)
        parts_l.append(l)
    mo, ml = oracle.lse_merge(np.stack(parts_o), np.stack(parts_l))
    np.testing.assert_allclose(mo, whole_o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(ml, whole_l, rtol=0, atol=1e-12)


@pytest.mark.parametrize("interleave", [1, 3, 4])
def test_merge_of_interleaved_partitions_equals_whole(interleave):
    """DCP on paper: partition the tokens by the interleave rule, give each
    partition its own table over its own blocks, attend per partition, merge."""
    rng = np.random.default_rng(11 + interleave)
    N, P, Hq, Hkv, D, bs = 45, 4, 4, 2, 8, 4
    K = rng.standard_normal((N, Hkv, D))
    V = rng.standard_normal((N, Hkv, D))
    q = rng.standard_normal((1, Hq, D)).astype(np.float32)
    # unsplit: tokens in order through an identity table
    nbw = -(-N // bs)
    kw = np.zeros((nbw, Hkv, bs, D), np.uint16)
    vw = np.zeros((nbw, Hkv, bs, D), np.uint16)
    slots = np.arange(N)
    oracle.kv_append(kw, vw, _small_int_bf16(K), _small_int_bf16(V), slots, bs)
    whole_o, whole_l = oracle.paged_decode_attn(q, kw, vw, np.arange(nbw, dtype=np.int32)[None],
                                                np.array([N], np.int32), 0.4)
    part, local = oracle.interleave(N, P, interleave)
    parts_o, parts_l = [], []
    for r in range(P):
        toks = np.nonzero(part == r)[0]
        nbr = max(1, -(-len(toks) // bs))
        kr = np.zeros((nbr, Hkv, bs, D), np.uint16)
        vr = np.zeros((nbr, Hkv, bs, D), np.uint16)
        oracle.kv_append(kr, vr, _small_int_bf16(K[toks]), _small_int_bf16(V[toks]),
                         local[toks], bs)
        o, l = oracle.paged_decode_attn(q, kr, vr, np.arange(nbr, dtype=np.int32)[None],
                                        np.array([len(toks)], np.int32), 0.4)
        parts_o.append(o)
        parts_l.append(l)
    mo, ml = oracle.lse_merge(np.stack(parts_o), np.stack(parts_l))
    np.testing.assert_allclose(mo, whole_o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(ml, whole_l, rtol=0, atol=1e-12)


def test_merge_closed_forms():
    out = np.array([[[1.0, 2.0]], [[3.0, -2.0]]])          # P=2, rows=1, dv=2
    lse = np.array([[5.0], [5.0]])
    mo, ml = oracle.lse_merge(out, lse)
    assert mo.tolist() == [[2.0, 0.0]] and ml[0] == pytest.approx(5.0 + math.log(2), abs=1e-15)
    # an empty partial contributes nothing
    mo, ml = oracle.lse_merge(np.array([[[1.0, 2.0]], [[0.0, 0.0]]]),
                              np.array([[0.7], [-np.inf]]))
    assert mo.tolist() == [[1.0, 2.0]] and ml[0] == 0.7
    # the first partial empty, the others far apart: the exact result is the
    # dominant partial's output, with no overflow from e^(1000)
    mo, ml = oracle.lse_merge(np.array([[[0.0, 0.0]], [[3.0, -1.0]], [[7.0, 9.0]]]),
                              np.array([[-np.inf], [-1000.0], [1000.0]]))
    assert mo.tolist() == [[7.0, 9.0]] and ml[0] == 1000.0
    # all empty
    mo, ml = oracle.lse_merge(np.zeros((3, 1, 2)), np.full((3, 1), -np.inf))
    assert mo.tolist() == [[0.0, 0.0]] and np.isneginf(ml[0])
    # weights e^(lse) in general: compare with scipy's logsumexp
    rng = np.random.default_rng(3)
    o = rng.standard_normal((5, 4, 3))
    l = rng.standard_normal((5, 4)) * 30
    mo, ml = oracle.lse_merge(o, l)
    w = softmax(l, axis=0)
    np.testing.assert_allclose(mo, np.einsum("pr,prd->rd", w, o), rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(ml, logsumexp(l, axis=0), rtol=0, atol=1e-12)


# ------------------------------------------------------- append and copy

def test_kv_append_matches_fancy_index_scatter():
    rng = np.random.default_rng(12)
    nb, Hkv, bs, Dk, Dv, T = 6, 3, 4, 8, 5, 9
    k = rng.integers(0, 1 << 16, (nb, Hkv, bs, Dk), dtype=np.uint16)
    v = rng.integers(0, 1 << 16, (nb, Hkv, bs, Dv), dtype=np.uint16)
    kn = rng.integers(0, 1 << 16, (T, Hkv, Dk), dtype=np.uint16)
    vn = rng.integers(0, 1 << 16, (T, Hkv, Dv), dtype=np.uint16)
    slots = rng.choice(nb * bs, T, replace=False).astype(np.int64)
    slots[2] = -1
    slots[5] = nb * bs + 3            # out of range: skipped and counted
    ek, ev = k.copy(), v.copy()
    for t in range(T):
        s = slots[t]
        if 0 <= s < nb * bs:
            ek[s // bs, :, s % bs, :] = kn[t]
            ev[s // bs, :, s % bs, :] = vn[t]
    bad = oracle.kv_append(k, v, kn, vn, slots, bs)
    assert bad == 1
    assert np.array_equal(k, ek) and np.array_equal(v, ev)


def test_copy_blocks_copies_every_head():
    rng = np.random.default_rng(13)
    k = rng.integers(0, 1 << 16, (7, 2, 4, 6), dtype=np.uint16)
    v = rng.integers(0, 1 << 16, (7, 2, 4, 3), dtype=np.uint16)
    ek, ev = k.copy(), v.copy()
    ek[[5, 0]] = k[[1, 3]]
    ev[[5, 0]] = v[[1, 3]]
    assert oracle.copy_blocks(k, v, [1, 3, 2], [5, 0, 9]) == 1
    assert np.array_equal(k, ek) and np.array_equal(v, ev)


def test_copy_on_write_leaves_other_sequence_unchanged():
    """Two sequences share all blocks including a partly filled tail; the
    second copies the tail to a free block, repoints its table, then appends.
    The first sequence's view and attention are bit-identical to before."""
    bs, Hkv, D = 4, 2, 8
    q, k, v, _, _ = rand_case(14, 2, 4, Hkv, D, bs, [10, 10], extra_blocks=0)
    k = np.concatenate([k, np.zeros_like(k[:2])])   # blocks 6 and 7 are free
    v = np.concatenate([v, np.zeros_like(v[:2])])
    shared = np.array([[3, 0, 5]], np.int32)          # 10 tokens, tail block 5 holds 2
    tables = np.repeat(shared, 2, axis=0)
    L = np.array([10, 10], np.int32)
    before_o, before_l = oracle.paged_decode_attn(q, k, v, tables, L, 0.3)
    # copy-on-write for sequence 1 into block 6
    assert oracle.copy_blocks(k, v, [5], [6]) == 0
    assert np.array_equal(k[6], k[5]) and np.array_equal(v[6], v[5])
    tables[1, 2] = 6
    mid_o, mid_l = oracle.paged_decode_attn(q, k, v, tables, L, 0.3)
    assert np.array_equal(mid_o, before_o) and np.array_equal(mid_l, before_l)
    rng = np.random.default_rng(15)
    kn = rng.integers(0x3000, 0x4000, (1, Hkv, D), dtype=np.uint16)
    vn = rng.integers(0x3000, 0x4000, (1, Hkv, D), dtype=np.uint16)
    slot = oracle.slot_of(tables[1], 10, bs)
    assert slot == 6 * bs + 2
    k5, v5 = k[5].copy(), v[5].copy()
    oracle.kv_append(k, v, kn, vn, [slot], bs)
    assert np.array_equal(k[5], k5) and np.array_equal(v[5], v5)      # original block intact
    assert np.array_equal(k[6, :, 2], kn[0]) and np.array_equal(v[6, :, 2], vn[0])
    after_o, after_l = oracle.paged_decode_attn(q, k, v, tables, np.array([10, 11], np.int32), 0.3)
    assert np.array_equal(after_o[0], before_o[0]) and np.array_equal(after_l[0], before_l[0])
    assert not np.array_equal(after_o[1], before_o[1])


# ------------------------------------------------------- multi-token decode

@pytest.mark.parametrize("T", [1, 2, 5])
def test_multi_token_matches_causal_mask_brute_force(T):
    """Query t of T new tokens sees the context and new tokens 0..t: one
    causal mask over the whole [T x L] score matrix, softmax row by row."""
    B, Hq, Hkv, D, bs = 3, 4, 2, 16, 4
    _, k, v, tables, L = rand_case(41 + T, B, Hq, Hkv, D, bs, [9, 14, 5])
    q = np.random.default_rng(7 + T).standard_normal((B, T, Hq, D)).astype(np.float32)
    out, lse = oracle.paged_decode_attn_multi(q, k, v, tables, L, 0.25)
    K, V = bf16_values(k), bf16_values(v)
    for b in range(B):
        n = int(L[b])
        idx = np.arange(n)
        phys, off = tables[b][idx // bs], idx % bs
        for h in range(Hq):
            g = h // (Hq // Hkv)
            Kc, Vc = K[phys, g, off], V[phys, g, off]
            S = 0.25 * (q[b, :, h].astype(np.float64) @ Kc.T)          # [T, n]
            future = idx[None, :] > (n - T + np.arange(T))[:, None]
            S = np.where(future, -np.inf, S)
            for t in range(T):
                np.testing.assert_allclose(out[b, t, h], softmax(S[t]) @ Vc, rtol=0, atol=1e-12)
                assert abs(lse[b, t, h] - logsumexp(S[t])) < 1e-12


def test_multi_token_special_cases():
    """T = 1 is ordinary decode; the last new token sees every stored token;
    a sequence holding fewer tokens than T leaves its first queries empty."""
    q1, k, v, tables, L = rand_case(5, 2, 4, 4, 8, 4, [7, 12])
    o1, l1 = oracle.paged_decode_attn(q1, k, v, tables, L, 0.5)
    om, lm = oracle.paged_decode_attn_multi(q1[:, None], k, v, tables, L, 0.5)
    assert np.array_equal(om[:, 0], o1) and np.array_equal(lm[:, 0], l1)
    q3 = np.random.default_rng(9).standard_normal((2, 3, 4, 8)).astype(np.float32)
    o3, l3 = oracle.paged_decode_attn_multi(q3, k, v, tables, L, 0.5)
    of, lf = oracle.paged_decode_attn(q3[:, 2], k, v, tables, L, 0.5)
    assert np.array_equal(o3[:, 2], of) and np.array_equal(l3[:, 2], lf)
    short = np.array([1, 12], dtype=np.int32)
    os_, ls_ = oracle.paged_decode_attn_multi(q3, k, v, tables, short, 0.5)
    assert np.all(np.isneginf(ls_[0, :2])) and np.all(os_[0, :2] == 0)
    assert np.isfinite(ls_[0, 2]).all()
