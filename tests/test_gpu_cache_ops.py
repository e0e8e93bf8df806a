"""GPU parity of the integer / copy paths against the oracle: slot mapping,
kv_append, copy_blocks and the interleaved partition slot mapping must be
bit-exact."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests._util import bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    import __graft_entry__
    __graft_entry__.build()
    import paged_kv_cache_93_gb300 as m
    m.device_status(reset=True)
    return m


@pytest.mark.parametrize("name", ["tiny", "mix"])
def test_slot_mapping_and_append_bit_exact(pkv, name):
    w = workloads.make(name)
    k, v = w.k_pool.cuda(), w.v_pool.cuda()
    bt = w.block_tables.cuda()
    slots = pkv.slot_mapping(k, v, bt, w.new_seq.cuda(), w.new_pos.cuda())
    pkv.kv_append(k, v, w.k_new.cuda(), w.v_new.cuda(), slots)
    ok_, ov_ = bits(w.k_pool), bits(w.v_pool)
    oslots = oracle.slot_mapping(w.block_tables.numpy(), w.new_seq.numpy(), w.new_pos.numpy(),
                                 w.block_size)
    oracle.kv_append(ok_, ov_, bits(w.k_new), bits(w.v_new), oslots, w.block_size)
    assert np.array_equal(slots.cpu().numpy(), oslots)
    assert np.array_equal(bits(k.cpu()), ok_) and np.array_equal(bits(v.cpu()), ov_)
    assert pkv.device_status() == 0


def test_bulk_append_with_padding_and_bad_slots(pkv):
    g = torch.Generator().manual_seed(21)
    nb, hkv, bs, dk, dv, T = 64, 4, 16, 128, 64, 700
    k0 = torch.randn(nb, hkv, bs, dk, generator=g).to(torch.bfloat16)
    v0 = torch.randn(nb, hkv, bs, dv, generator=g).to(torch.bfloat16)
    kn = torch.randn(T, hkv, dk, generator=g).to(torch.bfloat16)
    vn = torch.randn(T, hkv, dv, generator=g).to(torch.bfloat16)
    slots = torch.randperm(nb * bs, generator=g)[:T].to(torch.int64)
    slots[::37] = -1                      # padding: skipped silently
    slots[5] = nb * bs + 11               # out of range: skipped, flagged
    k, v = k0.cuda(), v0.cuda()
    pkv.kv_append(k, v, kn.cuda(), vn.cuda(), slots.cuda())
    assert pkv.device_status() == pkv.DEV_SLOT
    ok_, ov_ = bits(k0), bits(v0)
    assert oracle.kv_append(ok_, ov_, bits(kn), bits(vn), slots.numpy(), bs) == 1
    assert np.array_equal(bits(k.cpu()), ok_) and np.array_equal(bits(v.cpu()), ov_)


def test_slot_mapping_range_errors(pkv):
    w = workloads.tiny()
    k, v = w.k_pool.cuda(), w.v_pool.cuda()
    bt = w.block_tables.clone()
    bt[1, 2] = 99                         # block id outside the 8-block pool
    seq = torch.tensor([0, 1, 1, -1, 0], dtype=torch.int32)
    pos = torch.tensor([3, 9, 8, 0, 12], dtype=torch.int64)   # pos 12 -> past table row
    s = pkv.slot_mapping(k, v, bt.cuda(), seq.cuda(), pos.cuda()).cpu().tolist()
    st = pkv.device_status()
    assert st == pkv.DEV_BLOCK_ID | pkv.DEV_TABLE_RANGE
    assert s[0] == oracle.slot_of(w.block_tables[0].numpy(), 3, 4)
    assert s[1:] == [-1, -1, -1, -1]


def test_copy_blocks_bit_exact_and_conflicts(pkv):
    g = torch.Generator().manual_seed(22)
    nb, hkv, bs, dk, dv = 40, 1, 64, 576, 512
    k0 = torch.randn(nb, hkv, bs, dk, generator=g).to(torch.bfloat16)
    v0 = torch.randn(nb, hkv, bs, dv, generator=g).to(torch.bfloat16)
    src = torch.tensor([3, 3, 7, 9, 12], dtype=torch.int32)     # one source, several copies
    dst = torch.tensor([20, 21, 22, 23, 24], dtype=torch.int32)
    k, v = k0.cuda(), v0.cuda()
    pkv.copy_blocks(k, v, src.cuda(), dst.cuda())
    assert pkv.device_status() == 0
    ok_, ov_ = bits(k0), bits(v0)
    assert oracle.copy_blocks(ok_, ov_, src.numpy(), dst.numpy()) == 0
    assert np.array_equal(bits(k.cpu()), ok_) and np.array_equal(bits(v.cpu()), ov_)
    # conflicting pairs are skipped (and flagged); the clean pair still runs
    k, v = k0.cuda(), v0.cuda()
    src = torch.tensor([1, 2, 5, 30], dtype=torch.int32)
    dst = torch.tensor([10, 10, 1, 31], dtype=torch.int32)   # dup dst; dst 1 is a source
    pkv.copy_blocks(k, v, src.cuda(), dst.cuda())
    assert pkv.device_status() == pkv.DEV_COPY_CONFLICT
    kk = bits(k.cpu())
    ok_ = bits(k0)
    assert np.array_equal(kk[31], ok_[30])
    assert np.array_equal(kk[10], ok_[10]) and np.array_equal(kk[1], ok_[1])
    # out-of-range ids
    pkv.copy_blocks(k, v, torch.tensor([0], dtype=torch.int32).cuda(),
                    torch.tensor([nb], dtype=torch.int32).cuda())
    assert pkv.device_status() == pkv.DEV_BLOCK_ID


@pytest.mark.parametrize("N,P,I,bs", [(1000, 4, 1, 16), (1000, 4, 16, 16), (777, 3, 5, 8),
                                      (200_000, 4, 1, 16), (200_000, 4, 16, 16)])
def test_interleave_slot_mapping_bit_exact(pkv, N, P, I, bs):
    cap = -(-(-(-N // P) + I) // bs)
    rng = np.random.default_rng(N + P + I)
    perm = rng.permutation(P * cap).astype(np.int32)
    tables = perm.reshape(P, cap)
    k = torch.empty(P * cap, 1, bs, 8, dtype=torch.bfloat16, device="cuda")
    parts = torch.empty(N, dtype=torch.int32, device="cuda")
    slots = pkv.interleave_slot_mapping(k, k, 0, N, P, I, torch.from_numpy(tables).cuda(),
                                        part_out=parts)
    opart, olocal = oracle.interleave(N, P, I)
    oslots = oracle.slot_mapping(tables, opart, olocal, bs)
    assert np.array_equal(parts.cpu().numpy(), opart)
    assert np.array_equal(slots.cpu().numpy(), oslots)
    # a tail starting mid-sequence (the decode token of a long sequence)
    tail = pkv.interleave_slot_mapping(k, k, N - 3, 3, P, I, torch.from_numpy(tables).cuda())
    assert np.array_equal(tail.cpu().numpy(), oslots[-3:])
    assert pkv.device_status() == 0
