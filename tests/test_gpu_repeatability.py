"""Repeatability: the same decode call, made hundreds of times on the same
inputs, must return identical bits every time.

Every kernel here processes a work item in a fixed order on one CTA, so its
result is a deterministic function of the inputs; a result that changes
between calls exposes a race between the roles of a pipelined kernel (a
stage or accumulator written while another role still uses it) that a
single comparison against the oracle can miss.  The cases are chosen to
keep every pipeline busy: keys that grow along the sequence (the running
max keeps rising, so the accumulators are rescaled in TMEM), ragged tiles,
several splits.  The first call of each case is also checked against the
oracle."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests._steps import assert_attention_close
from tests._util import bits

pytestmark = pytest.mark.gpu
REPEATS = 300


@pytest.fixture(scope="module")
def pkv():
    import __graft_entry__
    __graft_entry__.build()
    import paged_kv_cache_93_gb300 as m
    m.device_status(reset=True)
    return m


def rising(seed, cached, hq, hkv, dk, dv, bs):
    """Keys scaled up along each sequence (x1 .. x7)."""
    w = workloads.custom(seed, cached, hq, hkv, dk, dv, bs)
    k = w.k_pool.float()
    for b in range(w.batch):
        L = int(w.seq_lens[b])
        j = np.arange(L)
        blk = w.block_tables[b, j // bs].long()
        k[blk, :, torch.from_numpy(j % bs)] *= torch.from_numpy(1.0 + 6.0 * j / L).float()[
            :, None, None]
    w.k_pool = k.to(torch.bfloat16)
    return w


def as_e4m3(w):
    w = workloads.e4m3(w)
    w.k_scale *= 7.0                     # keep the grown keys in range
    w.k_codes = (w.k_pool.float() / w.k_scale.view(1, -1, 1, 1)).clamp(-448, 448).to(
        torch.float8_e4m3fn).view(torch.uint8)
    return w


# (name, seed, cached lengths, Hq, Hkv, Dk, Dv, block size): one case per
# tensor-core kernel form and the warp-level GQA kernel
CASES = [
    ("mla_tc", 95, [1500, 700], 128, 1, 576, 512, 64),
    ("gqa_tc_16rows", 96, [1500, 900, 300], 64, 4, 128, 128, 16),
    ("gqa_tma", 97, [1500, 900, 300], 32, 8, 128, 128, 16),
]
E4M3_CASES = [
    ("mla_tc_e4m3", 95, [1500, 700], 128, 1, 576, 512, 64),
    ("gqa_tc_e4m3_4rows", 98, [1500, 900, 300], 32, 8, 128, 128, 16),
    ("gqa_tc_e4m3_16rows", 99, [1500, 900, 300], 64, 4, 128, 128, 16),
]


def _repeat(call, ro, rl, name):
    o0, l0 = call()
    torch.cuda.synchronize()
    first = (o0.cpu().numpy().copy(), l0.cpu().numpy().copy())
    assert_attention_close(first[0], first[1], ro, rl, name)
    differing = 0
    for _ in range(REPEATS):
        o, l = call()
        torch.cuda.synchronize()
        if not (np.array_equal(o.cpu().numpy(), first[0]) and
                np.array_equal(l.cpu().numpy(), first[1])):
            differing += 1
    assert differing == 0, f"{name}: {differing} of {REPEATS} calls differ from the first"


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("splits", [1, 3])
def test_bf16_calls_repeat_bit_for_bit(pkv, case, splits):
    name, seed, cached, hq, hkv, dk, dv, bs = case
    w = rising(seed, cached, hq, hkv, dk, dv, bs)
    dev = "cuda"
    k, v, bt = w.k_pool.to(dev), w.v_pool.to(dev), w.block_tables.to(dev)
    slots = pkv.slot_mapping(k, v, bt, w.new_seq.to(dev), w.new_pos.to(dev))
    pkv.kv_append(k, v, w.k_new.to(dev), w.v_new.to(dev), slots)
    q, lens = w.q.to(dev), w.seq_lens.to(dev)
    ko, vo = bits(w.k_pool), bits(w.v_pool)
    sl = oracle.slot_mapping(w.block_tables.numpy(), w.new_seq.numpy(), w.new_pos.numpy(), bs)
    assert oracle.kv_append(ko, vo, bits(w.k_new), bits(w.v_new), sl, bs) == 0
    ro, rl = oracle.paged_decode_attn(w.q.numpy(), ko, vo, w.block_tables.numpy(),
                                      w.seq_lens.numpy(), w.scale)
    _repeat(lambda: pkv.paged_decode_attn(q, k, v, bt, lens, w.scale, num_splits=splits),
            ro, rl, f"{name}/{splits}")
    assert pkv.device_status() == 0


@pytest.mark.parametrize("case", E4M3_CASES, ids=[c[0] for c in E4M3_CASES])
@pytest.mark.parametrize("splits", [1, 3])
def test_e4m3_calls_repeat_bit_for_bit(pkv, case, splits):
    name, seed, cached, hq, hkv, dk, dv, bs = case
    w = as_e4m3(rising(seed, cached, hq, hkv, dk, dv, bs))
    dev = "cuda"
    k, v, bt = w.k_codes.to(dev), w.v_codes.to(dev), w.block_tables.to(dev)
    ks, vs = w.k_scale.to(dev), w.v_scale.to(dev)
    slots = pkv.slot_mapping(k, v, bt, w.new_seq.to(dev), w.new_pos.to(dev))
    pkv.kv_append_e4m3(k, v, w.k_new.to(dev), w.v_new.to(dev), slots, ks, vs)
    q, lens = w.q.to(dev), w.seq_lens.to(dev)
    kc, vc = w.k_codes.numpy().copy(), w.v_codes.numpy().copy()
    sl = oracle.slot_mapping(w.block_tables.numpy(), w.new_seq.numpy(), w.new_pos.numpy(), bs)
    assert oracle.kv_append_e4m3(kc, vc, bits(w.k_new), bits(w.v_new), w.k_scale.numpy(),
                                 w.v_scale.numpy(), sl, bs) == 0
    ro, rl = oracle.paged_decode_attn_e4m3(w.q.numpy(), kc, vc, w.k_scale.numpy(),
                                           w.v_scale.numpy(), w.block_tables.numpy(),
                                           w.seq_lens.numpy(), w.scale)
    _repeat(lambda: pkv.paged_decode_attn_e4m3(q, k, v, ks, vs, bt, lens, w.scale,
                                               num_splits=splits),
            ro, rl, f"{name}/{splits}")
    assert pkv.device_status() == 0


@pytest.mark.parametrize("splits", [(3, 2), (1, 1)])
def test_cascade_calls_repeat_bit_for_bit(pkv, splits):
    """The cascade's single launch over two problems (all rows over the
    shared prefix, each sequence over the rest) on the tcgen05 kernel."""
    w = workloads.shared_prefix(31, 6, [400, 37, 900], 128, 1, 576, 512, 64)
    dev = "cuda"
    k, v, bt = w.k_pool.to(dev), w.v_pool.to(dev), w.block_tables.to(dev)
    slots = pkv.slot_mapping(k, v, bt, w.new_seq.to(dev), w.new_pos.to(dev))
    pkv.kv_append(k, v, w.k_new.to(dev), w.v_new.to(dev), slots)
    q, lens, ptab = w.q.to(dev), w.seq_lens.to(dev), w.info["prefix_table"].to(dev)
    ko, vo = bits(w.k_pool), bits(w.v_pool)
    sl = oracle.slot_mapping(w.block_tables.numpy(), w.new_seq.numpy(), w.new_pos.numpy(),
                             w.block_size)
    assert oracle.kv_append(ko, vo, bits(w.k_new), bits(w.v_new), sl, w.block_size) == 0
    ro, rl = oracle.paged_decode_attn(w.q.numpy(), ko, vo, w.block_tables.numpy(),
                                      w.seq_lens.numpy(), w.scale)
    _repeat(lambda: pkv.paged_decode_attn_cascade(q, k, v, ptab, bt, lens, w.scale,
                                                  prefix_splits=splits[0],
                                                  suffix_splits=splits[1]),
            ro, rl, f"cascade/{splits}")
    assert pkv.device_status() == 0
