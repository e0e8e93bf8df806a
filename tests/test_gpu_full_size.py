"""Parity at the full workload sizes, in the launch configurations the
benchmark times: the 32K-context GQA batch at the benchmark's headline split
count and at the split count the library picks by itself (every row against
the oracle), the 200,000-token DCP-style partition split (interleave 1 and
16, merged partitions against unsplit attention and the oracle; the
partitions also as the rows of one batched launch at the benchmark's split
count), and the
shared-prefix MLA-shaped step at the benchmark's split count (bit-exact cache
after copy-on-write + append; every head of the first, last, shortest- and
longest-suffix sequences and one head of every sequence against the
oracle)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import workloads
from bench import DEFAULT_SPLITS          # the split counts the benchmark times
from tests._steps import (agent_rows, assert_attention_close, auto_splits, gpu_step,
                          oracle_cache, oracle_step)
from tests._util import bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    import __graft_entry__
    __graft_entry__.build()
    import paged_kv_cache_93_gb300 as m
    m.device_status(reset=True)
    return m


@pytest.mark.parametrize("which", ["headline", "library_auto"])
def test_long32k_all_rows(pkv, which):
    """Every row of the 32K step, at the split count of the benchmark's
    headline line (16, the configuration's own) and at num_splits = 0, the
    library's choice, which the benchmark reports beside it."""
    w = workloads.long32k()
    if which == "headline":
        splits = DEFAULT_SPLITS["long32k"]
        assert splits == 16
    else:
        splits = 0
        auto = auto_splits(pkv, w)
        assert 1 <= auto <= 256
    out, lse, k, v, slots = gpu_step(pkv, w, num_splits=splits)
    ro, rl, ok_, ov_, oslots = oracle_step(w)
    assert np.array_equal(slots.cpu().numpy(), oslots)
    # the appended tokens landed exactly where the oracle put them
    for b, s in enumerate(oslots):
        blk, off = divmod(int(s), w.block_size)
        assert np.array_equal(bits(k[blk, :, off].cpu()), ok_[blk, :, off])
        assert np.array_equal(bits(v[blk, :, off].cpu()), ov_[blk, :, off])
    assert_attention_close(out.cpu().numpy(), lse.cpu().numpy(), ro, rl, "long32k")
    assert pkv.device_status() == 0


@pytest.mark.parametrize("interleave", [1, 16])
def test_dcp200k_partitions_merge_to_unsplit(pkv, interleave):
    w = workloads.dcp200k(interleave=interleave)
    N, P, bs = int(w.seq_lens[0]), w.num_parts, w.block_size
    dev = "cuda"
    k, v = w.k_pool.to(dev), w.v_pool.to(dev)
    table, ptab = w.block_tables.to(dev), w.part_tables.to(dev)
    kt, vt = w.k_tokens.to(dev), w.v_tokens.to(dev)
    # cache before the step: tokens 0..N-2 in both layouts
    seq0 = torch.zeros(N - 1, dtype=torch.int32, device=dev)
    pos = torch.arange(N - 1, dtype=torch.int64, device=dev)
    pkv.kv_append(k, v, kt[:N - 1], vt[:N - 1], pkv.slot_mapping(k, v, table, seq0, pos))
    pkv.kv_append(k, v, kt[:N - 1], vt[:N - 1],
                  pkv.interleave_slot_mapping(k, v, 0, N - 1, P, interleave, ptab))
    # the step: append the decode token to both layouts, then attend
    pkv.kv_append(k, v, w.k_new.to(dev), w.v_new.to(dev),
                  pkv.slot_mapping(k, v, table, w.new_seq.to(dev), w.new_pos.to(dev)))
    pkv.kv_append(k, v, w.k_new.to(dev), w.v_new.to(dev),
                  pkv.interleave_slot_mapping(k, v, N - 1, 1, P, interleave, ptab))
    q = w.q.to(dev)
    out_u, lse_u = pkv.paged_decode_attn(q, k, v, table, w.seq_lens.to(dev), w.scale)
    plen = torch.tensor([pkv.interleave_partition_len(N, P, interleave, r) for r in range(P)],
                        dtype=torch.int32)
    out_p = torch.empty(P, 1, w.num_q_heads, w.head_dim_v, device=dev)
    lse_p = torch.empty(P, 1, w.num_q_heads, device=dev)
    for r in range(P):
        pkv.paged_decode_attn(q, k, v, ptab[r:r + 1].contiguous(), plen[r:r + 1].to(dev), w.scale,
                              out=out_p[r], lse=lse_p[r])
    out_m, lse_m = pkv.lse_merge(out_p, lse_p)
    torch.cuda.synchronize()
    assert pkv.device_status() == 0

    # oracle: its own slots, appends, per-partition attention and merge
    ko, vo = bits(w.k_pool), bits(w.v_pool)
    ktb, vtb = bits(w.k_tokens), bits(w.v_tokens)
    uslots = oracle.slot_mapping(w.block_tables.numpy(), np.zeros(N, np.int32),
                                 np.arange(N), bs)
    part, local = oracle.interleave(N, P, interleave)
    pslots = oracle.slot_mapping(w.part_tables.numpy(), part, local, bs)
    oracle.kv_append(ko, vo, ktb, vtb, uslots, bs)
    oracle.kv_append(ko, vo, ktb, vtb, pslots, bs)
    assert np.array_equal(bits(k.cpu()), ko) and np.array_equal(bits(v.cpu()), vo)
    qn = w.q.numpy()
    ro, rl = oracle.paged_decode_attn(qn, ko, vo, w.block_tables.numpy(), w.seq_lens.numpy(),
                                      w.scale)
    counts = np.bincount(part, minlength=P).astype(np.int32)
    assert counts.tolist() == plen.tolist()
    po, pl = [], []
    for r in range(P):
        o, l = oracle.paged_decode_attn(qn, ko, vo, w.part_tables.numpy()[r:r + 1],
                                        counts[r:r + 1], w.scale)
        po.append(o)
        pl.append(l)
        assert_attention_close(out_p[r].cpu().numpy(), lse_p[r].cpu().numpy(), o, l,
                               f"partition {r}")
    # the benchmark's launch: the P partitions as the P rows of one batch
    # (the query repeated), at its split count, then the merge of the P results
    pq = q.expand(P, w.num_q_heads, w.head_dim_k).contiguous()
    bo, bl = pkv.paged_decode_attn(pq, k, v, ptab, plen.to(dev), w.scale,
                                   num_splits=DEFAULT_SPLITS["dcp200k"])
    bmo, bml = pkv.lse_merge(bo.unsqueeze(1), bl.unsqueeze(1))
    torch.cuda.synchronize()
    assert pkv.device_status() == 0
    for r in range(P):
        assert_attention_close(bo[r:r + 1].cpu().numpy(), bl[r:r + 1].cpu().numpy(), po[r],
                               pl[r], f"batched partition {r}")
    mo, ml = oracle.lse_merge(np.stack(po), np.stack(pl))
    np.testing.assert_allclose(mo, ro, rtol=0, atol=1e-12)     # the oracle agrees with itself
    np.testing.assert_allclose(ml, rl, rtol=0, atol=1e-12)
    assert_attention_close(out_u.cpu().numpy(), lse_u.cpu().numpy(), ro, rl, "unsplit")
    assert_attention_close(out_m.cpu().numpy(), lse_m.cpu().numpy(), ro, rl, "merged partitions")
    assert_attention_close(bmo.cpu().numpy(), bml.cpu().numpy(), ro, rl, "batched, merged")


def test_agent_mla_shared_prefix_step(pkv):
    w = workloads.agent_mla()
    splits = DEFAULT_SPLITS["agent_mla"]
    out, lse, k, v, slots = gpu_step(pkv, w, num_splits=splits)
    assert pkv.device_status() == 0
    rows, full = agent_rows(w)
    assert len(full) == 4
    ro, rl, ok_, ov_, oslots = oracle_step(w, rows)
    assert np.array_equal(slots.cpu().numpy(), oslots)
    assert np.array_equal(bits(k.cpu()), ok_) and np.array_equal(bits(v.cpu()), ov_)
    go, gl = out.cpu().numpy(), lse.cpu().numpy()
    for b, heads in rows.items():
        assert_attention_close(go[b, heads], gl[b, heads], ro[b, heads], rl[b, heads],
                               f"agent_mla seq {b}")
    assert np.isfinite(go).all() and np.isfinite(gl).all()


def test_agent_mla_shared_blocks_unchanged_by_copy_on_write(pkv):
    """The shared tail block keeps its original contents after every
    sequence copied it and appended into its private copy."""
    w = workloads.agent_mla(num_seqs=4, suffix_range=(50, 300))
    _, _, k, v, _ = gpu_step(pkv, w, num_splits=2)
    tail = w.info["shared_tail"]
    assert np.array_equal(bits(k[tail].cpu()), bits(w.k_pool[tail]))
    assert np.array_equal(bits(v[tail].cpu()), bits(w.v_pool[tail]))
    fill = w.info["prefix"] % w.block_size
    for dst in w.cow_dst.tolist():
        assert np.array_equal(bits(k[dst, :, :fill].cpu()), bits(w.k_pool[tail, :, :fill]))
    ok_, ov_, _ = oracle_cache(w)
    assert np.array_equal(bits(k.cpu()), ok_) and np.array_equal(bits(v.cpu()), ov_)
