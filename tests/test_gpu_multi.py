"""Multi-token decode (several new tokens per sequence, causal among them):
pkv_paged_decode_attn_multi against the oracle, after each side's own
append of the step's new tokens."""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests._steps import assert_attention_close, oracle_cache

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    import __graft_entry__
    __graft_entry__.build()
    import paged_kv_cache_93_gb300 as m
    m.device_status(reset=True)
    return m


def multi_case(seed, cached, T, hq, hkv, dk, dv, bs, extra_blocks=3):
    """Sequences holding `cached` tokens, then T new tokens each."""
    g = torch.Generator().manual_seed(seed)
    B = len(cached)
    lens = [c + T for c in cached]
    counts = [-(-n // bs) for n in lens]
    nb = sum(counts) + extra_blocks
    perm = torch.randperm(nb, generator=g)
    tables = torch.full((B, max(counts)), -1, dtype=torch.int32)
    at = 0
    for b, c in enumerate(counts):
        tables[b, :c] = perm[at:at + c].to(torch.int32)
        at += c
    bf = torch.bfloat16
    k = torch.randn(nb, hkv, bs, dk, generator=g).to(bf)
    v = torch.randn(nb, hkv, bs, dv, generator=g).to(bf)
    q = torch.randn(B, T, hq, dk, generator=g)
    new_seq = torch.arange(B, dtype=torch.int32).repeat_interleave(T)
    new_pos = torch.cat([torch.arange(c, c + T, dtype=torch.int64) for c in cached])
    k_new = torch.randn(B * T, hkv, dk, generator=g).to(bf)
    v_new = torch.randn(B * T, hkv, dv, generator=g).to(bf)
    w = workloads.Workload("multi", hq, hkv, dk, dv, bs, q, k, v, tables,
                           torch.tensor(lens, dtype=torch.int32), 1.0 / math.sqrt(dk),
                           new_seq, new_pos, k_new, v_new)
    w.tokens_per_seq = T
    return w


def gpu_multi(pkv, w, splits, flags=0):
    dev = "cuda"
    k, v, bt = w.k_pool.to(dev), w.v_pool.to(dev), w.block_tables.to(dev)
    slots = pkv.slot_mapping(k, v, bt, w.new_seq.to(dev), w.new_pos.to(dev))
    pkv.kv_append(k, v, w.k_new.to(dev), w.v_new.to(dev), slots)
    out, lse = pkv.paged_decode_attn_multi(w.q.to(dev), k, v, bt, w.seq_lens.to(dev), w.scale,
                                           num_splits=splits, flags=flags)
    torch.cuda.synchronize()
    return out.cpu().numpy(), lse.cpu().numpy()


def oracle_multi(w):
    k, v, _ = oracle_cache(w)
    return oracle.paged_decode_attn_multi(w.q.numpy(), k, v, w.block_tables.numpy(),
                                          w.seq_lens.numpy(), w.scale)


# (cached, Hq, Hkv, Dk, Dv, block size): GQA TMA kernel (G 4 and 8, D 128 and
# 64), the tcgen05 GQA kernel (G x T of 16, or 32 as two head groups: G 8 with
# T 4, G 16 with T 2), the tcgen05 MLA kernel (128 heads over 576/512), the
# generic kernel (G 3).
SHAPES = [
    ([300, 7, 64], 32, 8, 128, 128, 16),
    ([129, 40], 64, 8, 128, 128, 16),
    ([90, 260, 2], 32, 2, 128, 128, 32),
    ([77, 5], 8, 2, 64, 64, 8),
    ([200, 3], 128, 1, 576, 512, 64),
    ([50, 9], 6, 2, 64, 64, 16),
]


@pytest.mark.parametrize("shape", SHAPES,
                         ids=lambda s: f"G{s[1]//s[2]}_Dk{s[3]}_Dv{s[4]}_bs{s[5]}")
@pytest.mark.parametrize("T", [1, 2, 4])
@pytest.mark.parametrize("splits", [1, 3, 0])
@pytest.mark.parametrize("flags", ["auto", "no_tcgen05"])
def test_multi_token_decode(pkv, shape, T, splits, flags):
    """G*T = 16 or 32 rows with head dim 128 run on the tcgen05 GQA kernel
    (32 as two head groups), other foldable shapes on the warp-level-MMA one;
    no_tcgen05 checks the latter on the 16-row shapes too."""
    cached, hq, hkv, dk, dv, bs = shape
    w = multi_case(500 + T + dk, cached, T, hq, hkv, dk, dv, bs)
    f = pkv.DECODE_NO_TCGEN05 if flags == "no_tcgen05" else 0
    out, lse = gpu_multi(pkv, w, splits, flags=f)
    ro, rl = oracle_multi(w)
    assert_attention_close(out, lse, ro, rl, f"{shape}/T{T}/S{splits}")
    assert pkv.device_status() == 0


@pytest.mark.parametrize("T,hq", [(3, 8), (4, 8), (2, 16)],
                         ids=["rows12_per_token", "rows16_folded", "rows16_folded_G8"])
@pytest.mark.parametrize("splits", [1, 2])
@pytest.mark.parametrize("dk", [64, 128])
@pytest.mark.parametrize("held", ["one", "T-1"])
def test_multi_token_short_sequence_is_flagged(pkv, T, hq, splits, dk, held):
    """A sequence holding fewer tokens than T (one, or T - 1: then no row is
    of negative length): the queries with no token are empty (out 0, lse
    -inf), the others attend to what there is, and the device flags the
    length -- through the per-token rows (G*T = 12) and through the GQA
    kernel's folded rows (G*T = 16)."""
    n = 1 if held == "one" else T - 1
    w = multi_case(3, [20, 0], T, hq, 2, dk, dk, 16)
    w.seq_lens = torch.tensor([20 + T, n], dtype=torch.int32)  # sequence 1 holds n < T tokens
    pkv.device_status(reset=True)
    out, lse = gpu_multi(pkv, w, splits)
    assert np.isneginf(lse[1, :T - n]).all() and (out[1, :T - n] == 0).all()
    assert np.isfinite(lse[1, T - n:]).all() and np.isfinite(lse[0]).all()
    ro, rl = oracle_multi(w)
    assert_attention_close(out, lse, ro, rl, f"short T{T}")
    assert pkv.device_status() & pkv.DEV_SEQ_LEN


def test_multi_token_full_size_sampled_rows(pkv):
    """Speculative verification at 8 x 32K (4 new tokens per sequence, at
    the benchmark's split count), sampled (sequence, token, head) rows
    against the oracle."""
    from bench import DEFAULT_SPLITS
    w = workloads.spec_verify()
    out, lse = gpu_multi(pkv, w, DEFAULT_SPLITS["spec4_32k"])
    assert pkv.device_status() == 0
    k, v, _ = oracle_cache(w)
    T = w.tokens_per_seq
    for b, t, heads in [(0, 0, [0, 31]), (3, 2, [5]), (7, 3, [17, 30])]:
        qb = w.q.numpy()[b:b + 1, t]
        end = np.array([int(w.seq_lens[b]) - (T - 1) + t], dtype=np.int32)
        ro, rl = oracle.paged_decode_attn(qb, k, v, w.block_tables.numpy()[b:b + 1],
                                          w.seq_lens.numpy()[b:b + 1], w.scale, tok_end=end)
        assert_attention_close(out[b, t][None, heads], lse[b, t][None, heads],
                               ro[:, heads], rl[:, heads], f"row {b}/{t}")
