"""Values inside the keys (the latent layout of multi-head latent attention):
the cache is the K pool alone and a token's value is the first head_dim_v
dims of its key row.  The oracle reads that definition literally: its value
pool is a copy of K[..., :Dv] taken after the step's appends.  Every kernel
that takes the shape is checked against it, and against the same kernel fed
an explicit value pool holding those bytes (which must give identical bits,
since only the address the values are read from differs)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests._steps import agent_rows, assert_attention_close, oracle_rows
from tests._util import bits

pytestmark = pytest.mark.gpu

# (cached lengths, Hq, Hkv, Dk, Dv, block size, flags name)
LATENT_SHAPES = [
    ([200, 1, 77], 128, 1, 576, 512, 64, "auto"),          # tcgen05 kernel
    ([200, 1, 77], 128, 1, 576, 512, 64, "no_tcgen05"),    # warp-level-MMA kernel
    ([130, 9], 32, 1, 576, 512, 64, "auto"),               # G = 32: warp-level-MMA kernel
    ([90, 33], 16, 1, 576, 512, 32, "auto"),               # generic kernel
    ([300, 17], 32, 8, 128, 128, 16, "auto"),              # GQA TMA kernel: V = K
    ([41, 5], 64, 1, 192, 128, 64, "generic"),
]


@pytest.fixture(scope="module")
def pkv():
    import __graft_entry__
    __graft_entry__.build()
    import paged_kv_cache_93_gb300 as m
    m.device_status(reset=True)
    return m


def _flags(pkv, name):
    return {"auto": 0, "no_tcgen05": pkv.DECODE_NO_TCGEN05, "generic": pkv.DECODE_GENERIC}[name]


def _oracle_latent_cache(w):
    """The oracle's own copy-on-write and append on a host copy of the K pool
    (its value arrays are dummies: this cache keeps no values of its own)."""
    k = bits(w.k_pool)
    dummy_v = np.zeros(k.shape[:3] + (8,), dtype=np.uint16)
    if w.cow_src.numel():
        assert oracle.copy_blocks(k, dummy_v, w.cow_src.numpy(), w.cow_dst.numpy()) == 0
    slots = oracle.slot_mapping(w.block_tables.numpy(), w.new_seq.numpy(), w.new_pos.numpy(),
                                w.block_size)
    dummy_new = np.zeros((w.new_pos.numel(), w.num_kv_heads, 8), dtype=np.uint16)
    assert oracle.kv_append(k, dummy_v, bits(w.k_new), dummy_new, slots, w.block_size) == 0
    return k


def _oracle_latent(w):
    """Attention with V = K[..., :Dv] over the oracle's own cache."""
    k = _oracle_latent_cache(w)
    v = np.ascontiguousarray(k[..., :w.head_dim_v])
    out, lse = oracle.paged_decode_attn(w.q.numpy(), k, v, w.block_tables.numpy(),
                                        w.seq_lens.numpy(), w.scale)
    return out, lse, k


@pytest.mark.parametrize("shape", LATENT_SHAPES,
                         ids=lambda s: f"G{s[1]//s[2]}_Dk{s[3]}_Dv{s[4]}_bs{s[5]}_{s[6]}")
@pytest.mark.parametrize("splits", [1, 3])
def test_latent_decode(pkv, shape, splits):
    cached, hq, hkv, dk, dv, bs, fname = shape
    w = workloads.custom(300 + dk + hq, cached, hq, hkv, dk, dv, bs)
    dev = "cuda"
    k = w.k_pool.to(dev)
    latent = pkv.ValuesInKeys(dv)
    bt, lens = w.block_tables.to(dev), w.seq_lens.to(dev)
    slots = pkv.slot_mapping(k, latent, bt, w.new_seq.to(dev), w.new_pos.to(dev))
    pkv.kv_append(k, latent, w.k_new.to(dev), None, slots)
    f = _flags(pkv, fname)
    out, lse = pkv.paged_decode_attn(w.q.to(dev), k, latent, bt, lens, w.scale,
                                     num_splits=splits, flags=f)
    torch.cuda.synchronize()
    ro, rl, k_ref = _oracle_latent(w)
    assert np.array_equal(bits(k.cpu()), k_ref), "K pool after the append"
    assert_attention_close(out.cpu().numpy(), lse.cpu().numpy(), ro, rl,
                           f"latent {shape}/{splits}")
    # the same kernel with an explicit value pool holding K[..., :Dv]
    v = k[..., :dv].contiguous()
    out2, lse2 = pkv.paged_decode_attn(w.q.to(dev), k, v, bt, lens, w.scale,
                                       num_splits=splits, flags=f)
    torch.cuda.synchronize()
    assert torch.equal(out, out2) and torch.equal(lse, lse2)
    assert pkv.device_status() == 0


def test_latent_copy_blocks_copies_keys_only(pkv):
    w = workloads.custom(17, [70, 10], 128, 1, 576, 512, 64, extra_blocks=4)
    dev = "cuda"
    k = w.k_pool.to(dev)
    before = k.clone()
    src = torch.tensor([0, 2], dtype=torch.int32, device=dev)
    dst = torch.tensor([w.k_pool.shape[0] - 1, w.k_pool.shape[0] - 2], dtype=torch.int32,
                       device=dev)
    pkv.copy_blocks(k, pkv.ValuesInKeys(512), src, dst)
    torch.cuda.synchronize()
    expect = before.clone()
    expect[dst.long()] = before[src.long()]
    assert torch.equal(k, expect)
    assert pkv.device_status() == 0


def test_latent_agent_step_full_heads(pkv):
    """The shared-prefix MLA workload in the latent layout (1,152 B per token):
    copy-on-write of the shared tail + append + attention at the benchmark's
    19 splits; every head of four sequences (first, last, shortest and
    longest suffix) and one head of every other sequence against the
    oracle."""
    w = workloads.agent_mla()
    dev = "cuda"
    latent = pkv.ValuesInKeys(w.head_dim_v)
    k = w.k_pool.to(dev)
    bt = w.block_tables.to(dev)
    pkv.copy_blocks(k, latent, w.cow_src.to(dev), w.cow_dst.to(dev))
    slots = pkv.slot_mapping(k, latent, bt, w.new_seq.to(dev), w.new_pos.to(dev))
    pkv.kv_append(k, latent, w.k_new.to(dev), None, slots)
    out, lse = pkv.paged_decode_attn(w.q.to(dev), k, latent, bt, w.seq_lens.to(dev), w.scale,
                                     num_splits=19)
    torch.cuda.synchronize()
    assert pkv.device_status() == 0
    kh = _oracle_latent_cache(w)
    assert np.array_equal(bits(k.cpu()), kh), "K pool after copy-on-write + append"
    v = np.ascontiguousarray(kh[..., :w.head_dim_v])
    rows, full = agent_rows(w)
    assert len(full) == 4
    ro, rl = oracle_rows(w.q.numpy(), kh, v, w.block_tables.numpy(), w.seq_lens.numpy(),
                         w.scale, rows)
    go, gl = out.cpu().numpy(), lse.cpu().numpy()
    for b, heads in rows.items():
        assert_attention_close(go[b, heads], gl[b, heads], ro[b, heads], rl[b, heads],
                               f"latent agent seq {b}")
    assert np.isfinite(go).all() and np.isfinite(gl).all()
