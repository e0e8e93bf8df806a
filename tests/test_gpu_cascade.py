"""The shared-prefix cascade, pkv_paged_decode_attn_cascade ([PA] shared
blocks through every sequence's table; [AX] long shared prefixes): the
prefix part (all sequences' rows over the shared blocks as one sequence), the
suffix part (each sequence over the rest of its table) and their merge must
equal plain attention over the whole tables, which the oracle computes
directly.  Covered: the one-launch tcgen05 path (128 and 64 heads per KV
head), the two-launch path of other shapes (GQA with several KV heads, whose
rows are regrouped KV-head-major for the prefix part), no shared part,
nothing past the prefix but the decode token, the latent layout, explicit
and chosen split counts, the full-size shared-prefix MLA step, and the two
conditions the device flags (a table that does not begin with the shared
blocks, a sequence shorter than the prefix)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import workloads
from bench import DEFAULT_SPLITS
from tests._steps import (agent_rows, assert_attention_close, oracle_cache, oracle_rows,
                          oracle_step)
from tests._util import bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    import __graft_entry__
    __graft_entry__.build()
    import paged_kv_cache_93_gb300 as m
    m.device_status(reset=True)
    return m


def cascade_step(pkv, w, prefix_table, prefix_splits=0, suffix_splits=0, flags=0, dev="cuda"):
    """copy-on-write pairs -> slot mapping -> append -> cascade attention."""
    k = w.k_pool.to(dev)
    v = pkv.ValuesInKeys(w.head_dim_v) if w.v_pool is None else w.v_pool.to(dev)
    bt = w.block_tables.to(dev)
    if w.cow_src.numel():
        pkv.copy_blocks(k, v, w.cow_src.to(dev), w.cow_dst.to(dev))
    slots = pkv.slot_mapping(k, v, bt, w.new_seq.to(dev), w.new_pos.to(dev))
    pkv.kv_append(k, v, w.k_new.to(dev), None if w.v_new is None else w.v_new.to(dev), slots)
    out, lse = pkv.paged_decode_attn_cascade(w.q.to(dev), k, v, prefix_table.to(dev), bt,
                                             w.seq_lens.to(dev), w.scale,
                                             prefix_splits=prefix_splits,
                                             suffix_splits=suffix_splits, flags=flags)
    torch.cuda.synchronize()
    return out, lse, k, v


# (seed, prefix blocks, tokens cached past the prefix, Hq, Hkv, Dk, Dv, block size)
CASES = [
    (1, 6, [100, 0, 37, 300], 128, 1, 576, 512, 64),    # one tcgen05 launch, 128 heads
    (2, 3, [513, 5, 130], 64, 1, 192, 256, 128),        # one tcgen05 launch, 64 heads
    (3, 10, [40, 77, 0], 32, 8, 128, 128, 16),          # GQA, 8 KV heads: regrouped rows
    (4, 0, [90, 10], 128, 1, 576, 512, 64),             # no shared part
    (5, 4, [0, 0], 128, 1, 576, 512, 64),               # only the decode token past it
    (6, 5, [200, 31], 16, 2, 64, 64, 16),               # GQA, G 8, head dim 64
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"P{c[1]}_G{c[3]//c[4]}_Hkv{c[4]}_Dk{c[5]}")
@pytest.mark.parametrize("splits", [(0, 0), (3, 2), (1, 1)])
def test_cascade_equals_attention_over_whole_tables(pkv, case, splits):
    seed, pb, cached, hq, hkv, dk, dv, bs = case
    w = workloads.shared_prefix(seed, pb, cached, hq, hkv, dk, dv, bs)
    out, lse, _, _ = cascade_step(pkv, w, w.info["prefix_table"], *splits)
    assert pkv.device_status() == 0
    ro, rl, *_ = oracle_step(w)
    assert_attention_close(out.cpu().numpy(), lse.cpu().numpy(), ro, rl, f"{case}/{splits}")


@pytest.mark.parametrize("flags", ["generic", "no_tcgen05"])
def test_cascade_with_kernel_flags(pkv, flags):
    """The two-launch path on the MLA shape (the flags keep it off the
    tcgen05 kernel)."""
    f = {"generic": pkv.DECODE_GENERIC, "no_tcgen05": pkv.DECODE_NO_TCGEN05}[flags]
    w = workloads.shared_prefix(7, 3, [70, 9], 128, 1, 576, 512, 64)
    out, lse, _, _ = cascade_step(pkv, w, w.info["prefix_table"], 2, 2, flags=f)
    assert pkv.device_status() == 0
    ro, rl, *_ = oracle_step(w)
    assert_attention_close(out.cpu().numpy(), lse.cpu().numpy(), ro, rl, flags)


def test_cascade_latent_layout(pkv):
    """Values inside the keys (v_pool NULL), one tcgen05 launch."""
    w = workloads.shared_prefix(8, 5, [250, 3, 64], 128, 1, 576, 512, 64, latent=True)
    out, lse, k, _ = cascade_step(pkv, w, w.info["prefix_table"], 2, 2)
    assert pkv.device_status() == 0
    kh = bits(k.cpu())
    ro, rl = oracle.paged_decode_attn(w.q.numpy(), kh, np.ascontiguousarray(kh[..., :512]),
                                      w.block_tables.numpy(), w.seq_lens.numpy(), w.scale)
    assert_attention_close(out.cpu().numpy(), lse.cpu().numpy(), ro, rl, "latent")


def test_table_not_beginning_with_the_prefix_is_flagged(pkv):
    w = workloads.shared_prefix(9, 4, [30, 40], 128, 1, 576, 512, 64)
    bt = w.block_tables.clone()
    bt[1, 2] = bt[1, 4]          # a valid block, but not the shared one
    w.block_tables = bt
    cascade_step(pkv, w, w.info["prefix_table"], 1, 1)
    assert pkv.device_status() & pkv.DEV_PREFIX


def test_sequence_shorter_than_the_prefix_is_flagged(pkv):
    w = workloads.shared_prefix(10, 4, [30, 40], 128, 1, 576, 512, 64)
    P = 4 * 64
    dev = "cuda"
    lens = w.seq_lens.clone()
    lens[1] = P - 5
    k, v = w.k_pool.to(dev), w.v_pool.to(dev)
    pkv.paged_decode_attn_cascade(w.q.to(dev), k, v, w.info["prefix_table"].to(dev),
                                  w.block_tables.to(dev), lens.to(dev), w.scale)
    torch.cuda.synchronize()
    assert pkv.device_status() & pkv.DEV_SEQ_LEN


def test_agent_mla_cascade_full_size(pkv):
    """The shared-prefix MLA step at full size (32 sequences, 136,040-token
    prefix: its 2,125 full blocks shared, the tail block copied per
    sequence), the cascade at the benchmark's split counts: every head of
    four sequences and one head of every sequence against the oracle, and
    every row against the plain split path."""
    w = workloads.agent_mla()
    full = w.info["prefix"] // w.block_size
    ptab = w.block_tables[0, :full].clone()
    s1, s2 = DEFAULT_SPLITS["agent_mla_cascade"]
    out, lse, k, v = cascade_step(pkv, w, ptab, s1, s2)
    assert pkv.device_status() == 0
    ok_, ov_, _ = oracle_cache(w)
    assert np.array_equal(bits(k.cpu()), ok_) and np.array_equal(bits(v.cpu()), ov_)
    rows, fullrows = agent_rows(w)
    assert len(fullrows) == 4
    ro, rl = oracle_rows(w.q.numpy(), ok_, ov_, w.block_tables.numpy(), w.seq_lens.numpy(),
                         w.scale, rows)
    go, gl = out.cpu().numpy(), lse.cpu().numpy()
    for b, heads in rows.items():
        assert_attention_close(go[b, heads], gl[b, heads], ro[b, heads], rl[b, heads],
                               f"cascade seq {b}")
    # the plain split path on the same cache: every row
    po, pl = pkv.paged_decode_attn(w.q.cuda(), k, v, w.block_tables.cuda(), w.seq_lens.cuda(),
                                   w.scale, num_splits=DEFAULT_SPLITS["agent_mla"])
    torch.cuda.synchronize()
    assert_attention_close(go, gl, po.cpu().numpy().astype(np.float64),
                           pl.cpu().numpy().astype(np.float64), "cascade vs plain")
