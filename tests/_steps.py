"""One decode step of a workload, run two independent ways: through the GPU
library (C ABI via the Python binding) and through the CPU oracle.  The two
share only the seeded inputs from `workloads`."""
from __future__ import annotations

import ctypes

import numpy as np
import torch

import oracle
from tests._util import bits

# Tolerances of the contract: elementwise |d| <= 2e-3 or |d| <= 1e-2 |ref| on
# outputs, |d| <= 1e-4 on the LSE; plus a stricter relative-L2 check per row.
OUT_ABS, OUT_REL, LSE_ABS, ROW_REL_L2 = 2e-3, 1e-2, 1e-4, 1e-3


def assert_attention_close(out, lse, ref_out, ref_lse, where=""):
    out = np.asarray(out, dtype=np.float64)
    lse = np.asarray(lse, dtype=np.float64)
    assert out.shape == ref_out.shape and lse.shape == ref_lse.shape, where
    err = np.abs(out - ref_out)
    bad = ~((err <= OUT_ABS) | (err <= OUT_REL * np.abs(ref_out)))
    if bad.any():
        idx = np.argwhere(bad)
        rows = sorted({tuple(r[:-1]) for r in idx.tolist()})
        raise AssertionError(
            f"{where}: out mismatch in {len(idx)} elements of {len(rows)} rows {rows[:12]}, "
            f"last-axis indices {idx[:, -1].min()}..{idx[:, -1].max()}, first at "
            f"{idx[:5].tolist()}, max err {err.max():.3g}")
    empty = np.isneginf(ref_lse)
    assert np.array_equal(np.isneginf(lse), empty), f"{where}: empty rows differ"
    lerr = np.abs(lse[~empty] - ref_lse[~empty])
    assert lerr.size == 0 or lerr.max() <= LSE_ABS, f"{where}: lse max err {lerr.max():.3g}"
    assert (out[empty] == 0).all(), f"{where}: empty rows must give out = 0"
    d = out.reshape(-1, out.shape[-1]) - ref_out.reshape(-1, out.shape[-1])
    rn = np.linalg.norm(ref_out.reshape(-1, out.shape[-1]), axis=1)
    rel = np.linalg.norm(d, axis=1) / np.maximum(rn, 1e-30)
    rel = rel[rn > 0]
    assert rel.size == 0 or rel.max() <= ROW_REL_L2, f"{where}: row rel-L2 {rel.max():.3g}"


def auto_splits(pkv, w):
    """The split count num_splits = 0 resolves to for workload `w` on the
    current device (the library's rule, sized by the table width as the
    decode call sizes it)."""
    desc = pkv.CacheDesc(w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim_k, w.head_dim_v)
    return int(pkv.lib.pkv_decode_auto_splits(ctypes.byref(desc), w.batch, w.num_q_heads,
                                              w.block_tables.shape[1] * w.block_size))


def gpu_step(pkv, w, num_splits=0, flags=0, dev="cuda"):
    """copy-on-write pairs -> slot mapping -> append -> attention, on the GPU."""
    k = w.k_pool.to(dev)
    v = w.v_pool.to(dev)
    bt = w.block_tables.to(dev)
    if w.cow_src.numel():
        pkv.copy_blocks(k, v, w.cow_src.to(dev), w.cow_dst.to(dev))
    slots = pkv.slot_mapping(k, v, bt, w.new_seq.to(dev), w.new_pos.to(dev))
    pkv.kv_append(k, v, w.k_new.to(dev), w.v_new.to(dev), slots)
    out, lse = pkv.paged_decode_attn(w.q.to(dev), k, v, bt, w.seq_lens.to(dev), w.scale,
                                     num_splits=num_splits, flags=flags)
    torch.cuda.synchronize()
    return out, lse, k, v, slots


def oracle_cache(w):
    """The oracle's own copy-on-write + append on host copies of the pools."""
    k, v = bits(w.k_pool), bits(w.v_pool)
    if w.cow_src.numel():
        assert oracle.copy_blocks(k, v, w.cow_src.numpy(), w.cow_dst.numpy()) == 0
    slots = oracle.slot_mapping(w.block_tables.numpy(), w.new_seq.numpy(), w.new_pos.numpy(),
                                w.block_size)
    assert oracle.kv_append(k, v, bits(w.k_new), bits(w.v_new), slots, w.block_size) == 0
    return k, v, slots


def oracle_rows(q, k, v, tables, lens, scale, rows):
    """Oracle attention of the selected {sequence: [query heads]} of a cache
    with one KV head: every (sequence, head) as a one-head row of its own,
    all in one oracle call (its threads take the rows in turn).  Rows not
    selected stay NaN."""
    B, Hq, _ = q.shape
    out = np.full((B, Hq, v.shape[-1]), np.nan)
    lse = np.full((B, Hq), np.nan)
    pairs = [(b, h) for b, heads in rows.items() for h in heads]
    bs_, hs_ = np.array([p[0] for p in pairs]), np.array([p[1] for p in pairs])
    o, l = oracle.paged_decode_attn(np.ascontiguousarray(q[bs_, hs_][:, None, :]), k, v,
                                    np.ascontiguousarray(tables[bs_]),
                                    np.ascontiguousarray(lens[bs_]), scale)
    out[bs_, hs_], lse[bs_, hs_] = o[:, 0], l[:, 0]
    return out, lse


def agent_rows(w):
    """{sequence: [heads]} checked at the shared-prefix workload's full size:
    all heads of the first and last sequences and of those with the shortest
    and longest suffix, and one head of every other sequence (a different
    head each, so that every 64-head group is covered).  Also returns the
    fully checked sequences."""
    lens = w.seq_lens.numpy().astype(np.int64)
    full = {0, len(lens) - 1, int(np.argmin(lens)), int(np.argmax(lens))}
    rows = {b: (list(range(w.num_q_heads)) if b in full else [(37 * b + 11) % w.num_q_heads])
            for b in range(len(lens))}
    return rows, sorted(full)


def oracle_step(w, rows=None):
    """Oracle attention after its own append.  `rows`: optional {sequence:
    [query heads]} to compute (the rest stay NaN); with one KV head the
    selected heads are computed alone, otherwise the whole sequence is."""
    k, v, slots = oracle_cache(w)
    q = w.q.numpy()
    tables, lens = w.block_tables.numpy(), w.seq_lens.numpy()
    if rows is None:
        out, lse = oracle.paged_decode_attn(q, k, v, tables, lens, w.scale)
        return out, lse, k, v, slots
    B, Hq, _ = q.shape
    out = np.full((B, Hq, w.head_dim_v), np.nan)
    lse = np.full((B, Hq), np.nan)
    if w.num_kv_heads == 1:
        o, l = oracle_rows(q, k, v, tables, lens, w.scale, rows)
        return o, l, k, v, slots
    for b, heads in rows.items():
        heads = list(heads)
        o, l = oracle.paged_decode_attn(q[b:b + 1], k, v, tables[b:b + 1], lens[b:b + 1],
                                        w.scale)
        out[b, heads], lse[b, heads] = o[0, heads], l[0, heads]
    return out, lse, k, v, slots
