"""FP8 (E4M3) cache on the GPU against the oracle: the quantising append and
the block copy byte for byte, and decode attention over E4M3 pools with
per-KV-head scales within the contract's tolerances (the oracle attends to
the same stored values, decoded and scaled in fp64)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests._steps import agent_rows, assert_attention_close
from tests._util import bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    import __graft_entry__
    __graft_entry__.build()
    import paged_kv_cache_93_gb300 as m
    m.device_status(reset=True)
    return m


def gpu_e4m3_step(pkv, w, splits, dev="cuda", flags=0):
    k, v = w.k_codes.to(dev), w.v_codes.to(dev)
    ks, vs = w.k_scale.to(dev), w.v_scale.to(dev)
    bt = w.block_tables.to(dev)
    slots = pkv.slot_mapping(k, v, bt, w.new_seq.to(dev), w.new_pos.to(dev))
    pkv.kv_append_e4m3(k, v, w.k_new.to(dev), w.v_new.to(dev), slots, ks, vs)
    out, lse = pkv.paged_decode_attn_e4m3(w.q.to(dev), k, v, ks, vs, bt, w.seq_lens.to(dev),
                                          w.scale, num_splits=splits, flags=flags)
    torch.cuda.synchronize()
    return out.cpu().numpy(), lse.cpu().numpy(), k.cpu().numpy(), v.cpu().numpy()


def oracle_e4m3_cache(w):
    k, v = w.k_codes.numpy().copy(), w.v_codes.numpy().copy()
    slots = oracle.slot_mapping(w.block_tables.numpy(), w.new_seq.numpy(), w.new_pos.numpy(),
                                w.block_size)
    assert oracle.kv_append_e4m3(k, v, bits(w.k_new), bits(w.v_new), w.k_scale.numpy(),
                                 w.v_scale.numpy(), slots, w.block_size) == 0
    return k, v


def oracle_e4m3_step(w):
    k, v = oracle_e4m3_cache(w)
    out, lse = oracle.paged_decode_attn_e4m3(w.q.numpy(), k, v, w.k_scale.numpy(),
                                             w.v_scale.numpy(), w.block_tables.numpy(),
                                             w.seq_lens.numpy(), w.scale)
    return out, lse, k, v


# (cached lengths, Hq, Hkv, block size): groups of 4, 8 and 16; ragged tails,
# a sequence holding only the new token, block sizes 16..256
SHAPES = [
    ([300, 7, 64, 0], 32, 8, 16),
    ([129, 40, 255], 16, 2, 32),
    ([600, 65], 64, 4, 64),
    ([700, 5, 130], 8, 2, 128),
    ([200, 1], 16, 1, 256),
    ([250, 3, 90], 64, 2, 16),             # group 32: two head groups of 16
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"G{s[1]//s[2]}_bs{s[3]}")
@pytest.mark.parametrize("splits", [1, 3, 0])
def test_e4m3_step_matches_oracle(pkv, shape, splits):
    cached, hq, hkv, bs = shape
    w = workloads.e4m3(workloads.custom(40 + bs + hq, cached, hq, hkv, 128, 128, bs))
    out, lse, k, v = gpu_e4m3_step(pkv, w, splits)
    ro, rl, rk, rv = oracle_e4m3_step(w)
    assert np.array_equal(k, rk) and np.array_equal(v, rv), "pools after the append"
    assert_attention_close(out, lse, ro, rl, f"e4m3 {shape}/{splits}")
    assert pkv.device_status() == 0


# shapes the tensor-core kernel does not take: the CUDA-core kernel
GENERIC_SHAPES = [
    ([37, 5], 8, 2, 64, 64, 8),            # head dim 64, group 4
    ([90, 1, 33], 6, 2, 64, 64, 16),       # group 3
    ([70, 9], 16, 1, 576, 512, 64),        # MLA-shaped dims
    ([40], 2, 2, 128, 128, 16),            # group 1
]


@pytest.mark.parametrize("shape", GENERIC_SHAPES,
                         ids=lambda s: f"G{s[1]//s[2]}_Dk{s[3]}_Dv{s[4]}_bs{s[5]}")
@pytest.mark.parametrize("splits", [1, 3])
def test_e4m3_generic_shapes(pkv, shape, splits):
    cached, hq, hkv, dk, dv, bs = shape
    w = workloads.e4m3(workloads.custom(60 + dk + hq, cached, hq, hkv, dk, dv, bs))
    out, lse, k, v = gpu_e4m3_step(pkv, w, splits)
    ro, rl, rk, rv = oracle_e4m3_step(w)
    assert np.array_equal(k, rk) and np.array_equal(v, rv)
    assert_attention_close(out, lse, ro, rl, f"e4m3 generic {shape}/{splits}")
    assert pkv.device_status() == 0


# The MLA shape over an FP8 cache: 128 (or 64) query heads over one 576-dim
# key / 512-dim value head, ragged lengths across 128-token tiles.
MLA_SHAPES = [
    ([700, 3, 255, 128], 128, 1, 576, 512, 64),
    ([1000, 65], 64, 1, 576, 512, 128),
    ([300, 129], 256, 2, 576, 512, 64),
]


@pytest.mark.parametrize("shape", MLA_SHAPES,
                         ids=lambda s: f"G{s[1]//s[2]}_Hkv{s[2]}_bs{s[5]}")
@pytest.mark.parametrize("splits", [1, 3, 0])
def test_e4m3_mla_shape_matches_oracle(pkv, shape, splits):
    cached, hq, hkv, dk, dv, bs = shape
    w = workloads.e4m3(workloads.custom(90 + hq + bs, cached, hq, hkv, dk, dv, bs))
    out, lse, k, v = gpu_e4m3_step(pkv, w, splits)
    ro, rl, rk, rv = oracle_e4m3_step(w)
    assert np.array_equal(k, rk) and np.array_equal(v, rv), "pools after the append"
    assert_attention_close(out, lse, ro, rl, f"e4m3 MLA {shape}/{splits}")
    assert pkv.device_status() == 0


# (cached tokens, Hq, Hkv, Dk, Dv, block size): the four tcgen05 FP8 GQA
# forms, the large-group (MLA-shaped) form and a CUDA-core shape (head dim
# 64); the last row is made empty
PARTIAL_SHAPES = [
    ([900, 70, 1, 0], 32, 8, 128, 128, 16),
    ([700, 129, 0], 16, 2, 128, 128, 32),
    ([1000, 65, 0], 64, 4, 128, 128, 64),
    ([600, 3, 0], 64, 2, 128, 128, 16),
    ([800, 1, 0], 128, 1, 576, 512, 64),
    ([500, 33, 0], 16, 4, 64, 64, 16),
]


@pytest.mark.parametrize("shape", PARTIAL_SHAPES,
                         ids=lambda s: f"G{s[1]//s[2]}_D{s[3]}_bs{s[5]}")
def test_e4m3_partials_match_oracle_token_ranges(pkv, shape):
    """Split s of row b covers [s*C, min(L, (s+1)*C)), C = 64*ceil(L/(64*S));
    an empty row or chunk gives (0, -inf); the merged partials are the
    attention call's result at the same split count, bit for bit."""
    lens, hq, hkv, dk, dv, bs = shape
    w = workloads.e4m3(workloads.custom(60 + hq + bs, lens, hq, hkv, dk, dv, bs))
    w.seq_lens[-1] = 0                                 # an empty row
    S = 5
    dev = "cuda"
    k, v = w.k_codes.to(dev), w.v_codes.to(dev)
    ks, vs = w.k_scale.to(dev), w.v_scale.to(dev)
    bt, sl, q = w.block_tables.to(dev), w.seq_lens.to(dev), w.q.to(dev)
    op, lp = pkv.paged_decode_attn_partial_e4m3(q, k, v, ks, vs, bt, sl, w.scale, S)
    out, lse = pkv.paged_decode_attn_e4m3(q, k, v, ks, vs, bt, sl, w.scale, num_splits=S)
    mo, ml = pkv.lse_merge(op, lp)
    torch.cuda.synchronize()
    assert pkv.device_status() == 0
    L = w.seq_lens.numpy().astype(np.int64)
    C = 64 * (-(-L // (64 * S)))
    args = (w.q.numpy(), w.k_codes.numpy(), w.v_codes.numpy(), w.k_scale.numpy(),
            w.v_scale.numpy(), w.block_tables.numpy(), L.astype(np.int32), w.scale)
    for s in range(S):
        begin = np.minimum(s * C, L).astype(np.int32)
        end = np.minimum((s + 1) * C, L).astype(np.int32)
        ro, rl = oracle.paged_decode_attn_e4m3(*args, tok_begin=begin, tok_end=end)
        assert_attention_close(op[s].cpu().numpy(), lp[s].cpu().numpy(), ro, rl, f"split {s}")
    assert torch.equal(mo, out) and torch.equal(ml, lse), "merged partials vs the call"
    ro, rl = oracle.paged_decode_attn_e4m3(*args)
    assert_attention_close(mo.cpu().numpy(), ml.cpu().numpy(), ro, rl, "merged partials")


def test_e4m3_mla_nan_codes_in_unused_slots_do_not_leak(pkv):
    """NaN codes in the slots past each sequence's end (and possibly in the
    block whose rows stand in for half tiles past the end): the value rows
    past the end are written as zeros, the scores there are masked."""
    bs = 64
    w = workloads.e4m3(workloads.custom(15, [100, 190, 63], 128, 1, 576, 512, bs,
                                        extra_blocks=0))
    for b in range(w.batch):
        L = int(w.seq_lens[b])
        last = int(w.block_tables[b, (L - 1) // bs])
        w.k_codes[last, :, L % bs or bs:] = 0x7F
        w.v_codes[last, :, L % bs or bs:] = 0xFF
    ro, rl, *_ = oracle_e4m3_step(w)
    for splits in (1, 2):
        out, lse, *_ = gpu_e4m3_step(pkv, w, splits)
        assert np.isfinite(out).all() and np.isfinite(lse).all()
        assert_attention_close(out, lse, ro, rl, f"MLA nan tail/{splits}")
        assert pkv.device_status() == 0


@pytest.mark.parametrize("splits", [1, 3])
def test_e4m3_mla_rising_scores(pkv, splits):
    """MLA shape, keys growing along the sequence: the running max keeps
    rising past the slack and the accumulators are rescaled in TMEM."""
    bs = 64
    w = workloads.custom(95, [1500, 700], 128, 1, 576, 512, bs)
    k = w.k_pool.float()
    for b in range(2):
        L = int(w.seq_lens[b])
        j = np.arange(L)
        blk = w.block_tables[b, j // bs].long()
        k[blk, :, torch.from_numpy(j % bs)] *= torch.from_numpy(1.0 + 6.0 * j / L).float()[:, None,
                                                                                         None]
    w.k_pool = k.to(torch.bfloat16)
    w = workloads.e4m3(w)
    w.k_scale *= 7.0                                      # keep the grown keys in range
    w.k_codes = (w.k_pool.float() / w.k_scale.view(1, -1, 1, 1)).clamp(-448, 448).to(
        torch.float8_e4m3fn).view(torch.uint8)
    out, lse, *_ = gpu_e4m3_step(pkv, w, splits)
    ro, rl, *_ = oracle_e4m3_step(w)
    assert_attention_close(out, lse, ro, rl, f"MLA rising/{splits}")
    assert pkv.device_status() == 0


@pytest.mark.parametrize("factor", [0.0, 1e-3, 8.0])
def test_e4m3_mla_query_magnitudes(pkv, factor):
    """The query is stored as fp16 hi + lo after scaling by a power of two
    chosen per work item from its largest element: a zero, a tiny and a
    large query (the first sequence's; the second stays as drawn) keep the
    tolerances."""
    w = workloads.custom(96, [400, 260], 128, 1, 576, 512, 64)
    w.q[0] *= factor
    w = workloads.e4m3(w)
    ro, rl, *_ = oracle_e4m3_step(w)
    for splits in (1, 3):
        out, lse, *_ = gpu_e4m3_step(pkv, w, splits)
        assert_attention_close(out, lse, ro, rl, f"MLA query x{factor}/{splits}")
        assert pkv.device_status() == 0


def test_e4m3_agent_mla_full_size_sampled_rows(pkv):
    """The shared-prefix MLA step at full size over an FP8 cache (32
    sequences over a 136,040-token shared prefix; copy-on-write of the
    shared tail block's codes, the quantising append of every suffix and
    decode token, attention at the benchmark's split count): the pools byte
    for byte, and every head of four sequences and one head of every other
    sequence against the oracle."""
    from bench import DEFAULT_SPLITS
    w = workloads.make("agent_mla_e4m3")
    dev = "cuda"
    k, v = w.k_codes.to(dev), w.v_codes.to(dev)
    ks, vs = w.k_scale.to(dev), w.v_scale.to(dev)
    bt = w.block_tables.to(dev)
    pkv.copy_blocks_e4m3(k, v, w.cow_src.to(dev), w.cow_dst.to(dev))
    slots = pkv.slot_mapping(k, v, bt, w.new_seq.to(dev), w.new_pos.to(dev))
    pkv.kv_append_e4m3(k, v, w.k_new.to(dev), w.v_new.to(dev), slots, ks, vs)
    out, lse = pkv.paged_decode_attn_e4m3(w.q.to(dev), k, v, ks, vs, bt, w.seq_lens.to(dev),
                                          w.scale, num_splits=DEFAULT_SPLITS["agent_mla_e4m3"])
    torch.cuda.synchronize()
    assert pkv.device_status() == 0
    kc, vc = w.k_codes.numpy().copy(), w.v_codes.numpy().copy()
    # a block copy moves bytes: the oracle's copy over the code pools viewed
    # as 16-bit words
    assert oracle.copy_blocks(kc.view(np.uint16), vc.view(np.uint16), w.cow_src.numpy(),
                              w.cow_dst.numpy()) == 0
    sl = oracle.slot_mapping(w.block_tables.numpy(), w.new_seq.numpy(), w.new_pos.numpy(),
                             w.block_size)
    assert oracle.kv_append_e4m3(kc, vc, bits(w.k_new), bits(w.v_new), w.k_scale.numpy(),
                                 w.v_scale.numpy(), sl, w.block_size) == 0
    assert np.array_equal(k.cpu().numpy(), kc) and np.array_equal(v.cpu().numpy(), vc)
    rows, full = agent_rows(w)
    assert len(full) == 4
    pairs = [(b, h) for b, heads in rows.items() for h in heads]
    bs_, hs_ = np.array([p[0] for p in pairs]), np.array([p[1] for p in pairs])
    # with one KV head every (sequence, head) is a one-head row of its own
    ro, rl = oracle.paged_decode_attn_e4m3(np.ascontiguousarray(w.q.numpy()[bs_, hs_][:, None]),
                                           kc, vc, w.k_scale.numpy(), w.v_scale.numpy(),
                                           np.ascontiguousarray(w.block_tables.numpy()[bs_]),
                                           np.ascontiguousarray(w.seq_lens.numpy()[bs_]),
                                           w.scale)
    go, gl = out.cpu().numpy(), lse.cpu().numpy()
    assert_attention_close(go[bs_, hs_], gl[bs_, hs_], ro[:, 0], rl[:, 0], "agent MLA e4m3")


@pytest.mark.parametrize("shape", SHAPES[:3], ids=lambda s: f"G{s[1]//s[2]}_bs{s[3]}")
def test_e4m3_forced_generic_matches_oracle(pkv, shape):
    cached, hq, hkv, bs = shape
    w = workloads.e4m3(workloads.custom(80 + bs, cached, hq, hkv, 128, 128, bs))
    out, lse, *_ = gpu_e4m3_step(pkv, w, 3, flags=pkv.DECODE_GENERIC)
    ro, rl, *_ = oracle_e4m3_step(w)
    assert_attention_close(out, lse, ro, rl, f"e4m3 forced generic {shape}")
    assert pkv.device_status() == 0


def test_e4m3_append_saturates_and_flags(pkv):
    """Large new values saturate to +-448 codes; skipped and out-of-range
    slots behave as in the bf16 append."""
    g = torch.Generator().manual_seed(4)
    nb, hkv, bs = 6, 2, 16
    k = torch.zeros(nb, hkv, bs, 128, dtype=torch.uint8)
    v = torch.zeros(nb, hkv, bs, 128, dtype=torch.uint8)
    kn = (torch.randn(5, hkv, 128, generator=g) * 20).to(torch.bfloat16)
    vn = (torch.randn(5, hkv, 128, generator=g) * 3).to(torch.bfloat16)
    ks = torch.tensor([0.01, 0.2])
    vs = torch.tensor([0.05, 0.5])
    slots = torch.tensor([0, 17, -1, 95, 96], dtype=torch.int64)        # 96 is past the pool
    dev = "cuda"
    kd, vd = k.to(dev), v.to(dev)
    pkv.kv_append_e4m3(kd, vd, kn.to(dev), vn.to(dev), slots.to(dev), ks.to(dev), vs.to(dev))
    assert pkv.device_status() == pkv.DEV_SLOT
    kh, vh = k.numpy().copy(), v.numpy().copy()
    assert oracle.kv_append_e4m3(kh, vh, bits(kn), bits(vn), ks.numpy(), vs.numpy(),
                                 slots.numpy(), bs) == 1
    assert np.array_equal(kd.cpu().numpy(), kh) and np.array_equal(vd.cpu().numpy(), vh)
    assert (kh == 0x7E).any() and (kh == 0xFE).any()      # some values saturated


def test_e4m3_copy_blocks(pkv):
    g = torch.Generator().manual_seed(5)
    k = torch.randint(0, 256, (8, 2, 16, 128), generator=g, dtype=torch.uint8)
    v = torch.randint(0, 256, (8, 2, 16, 128), generator=g, dtype=torch.uint8)
    dev = "cuda"
    kd, vd = k.to(dev), v.to(dev)
    src = torch.tensor([1, 3], dtype=torch.int32)
    dst = torch.tensor([6, 0], dtype=torch.int32)
    pkv.copy_blocks_e4m3(kd, vd, src.to(dev), dst.to(dev))
    torch.cuda.synchronize()
    ek, ev = k.clone(), v.clone()
    ek[dst.long()] = k[src.long()]
    ev[dst.long()] = v[src.long()]
    assert torch.equal(kd.cpu(), ek) and torch.equal(vd.cpu(), ev)
    assert pkv.device_status() == 0


@pytest.mark.parametrize("hq", [8, 16, 32], ids=["G4", "G8", "G16"])
def test_e4m3_single_token_is_exact(pkv, hq):
    """One token: out is its stored value times the value scale, rounded
    once to fp32; lse is its score."""
    w = workloads.e4m3(workloads.custom(9, [0, 0], hq, 2, 128, 128, 16))
    out, lse, *_ = gpu_e4m3_step(pkv, w, 1)
    ro, rl, _, rv = oracle_e4m3_step(w)
    assert np.array_equal(out, ro.astype(np.float32))
    assert np.abs(lse - rl).max() <= 1e-4


def test_e4m3_nan_codes_in_unused_slots_do_not_leak(pkv):
    w = workloads.e4m3(workloads.custom(13, [20, 50], 32, 2, 128, 128, 16, extra_blocks=0))
    for b in range(2):
        L = int(w.seq_lens[b])
        last = int(w.block_tables[b, (L - 1) // 16])
        w.k_codes[last, :, L % 16 or 16:] = 0x7F
        w.v_codes[last, :, L % 16 or 16:] = 0xFF
    out, lse, *_ = gpu_e4m3_step(pkv, w, 1)
    assert np.isfinite(out).all() and np.isfinite(lse).all()
    ro, rl, *_ = oracle_e4m3_step(w)
    assert_attention_close(out, lse, ro, rl, "nan tail")


@pytest.mark.parametrize("splits", [1, 3])
def test_e4m3_rising_scores(pkv, splits):
    """Keys grow along the sequence: the running max keeps rising past the
    slack and the accumulators are rescaled in TMEM."""
    w = workloads.custom(92, [1500, 700], 32, 2, 128, 128, 16)
    k = w.k_pool.float()
    for b in range(2):
        L = int(w.seq_lens[b])
        for j in range(L):
            blk = int(w.block_tables[b, j // 16])
            k[blk, :, j % 16] *= 1.0 + 6.0 * j / L
    w.k_pool = k.to(torch.bfloat16)
    w = workloads.e4m3(w)
    w.k_scale *= 7.0                                      # keep the grown keys in range
    w.k_codes = (w.k_pool.float() / w.k_scale.view(1, -1, 1, 1)).clamp(-448, 448).to(
        torch.float8_e4m3fn).view(torch.uint8)
    out, lse, *_ = gpu_e4m3_step(pkv, w, splits)
    ro, rl, *_ = oracle_e4m3_step(w)
    assert_attention_close(out, lse, ro, rl, f"rising/{splits}")
    assert pkv.device_status() == 0


def test_e4m3_bad_seq_len_and_block_id_are_flagged(pkv):
    w = workloads.e4m3(workloads.custom(12, [100, 100], 32, 2, 128, 128, 16))
    dev = "cuda"
    k, v = w.k_codes.to(dev), w.v_codes.to(dev)
    ks, vs = w.k_scale.to(dev), w.v_scale.to(dev)
    q = w.q.to(dev)
    lens = w.seq_lens.clone()
    lens[1] = 10_000
    out, lse = pkv.paged_decode_attn_e4m3(q, k, v, ks, vs, w.block_tables.to(dev), lens.to(dev),
                                          w.scale, num_splits=2)
    assert pkv.device_status() == pkv.DEV_SEQ_LEN
    assert torch.isneginf(lse[1]).all() and (out[1] == 0).all()
    bt = w.block_tables.clone()
    bt[0, 3] = 1 << 20
    out, lse = pkv.paged_decode_attn_e4m3(q, k, v, ks, vs, bt.to(dev), w.seq_lens.to(dev),
                                          w.scale, num_splits=2)
    assert pkv.device_status() == pkv.DEV_BLOCK_ID
    assert torch.isfinite(out).all() and torch.isfinite(lse).all()


def test_e4m3_full_size_sampled_rows(pkv):
    """8 x 32K GQA step (32/8 heads, block 16) over an E4M3 cache at the
    benchmark's split count: three whole sequences against the oracle."""
    from bench import DEFAULT_SPLITS
    w = workloads.make("long32k_e4m3")
    out, lse, *_ = gpu_e4m3_step(pkv, w, DEFAULT_SPLITS["long32k_e4m3"])
    assert pkv.device_status() == 0
    k, v = oracle_e4m3_cache(w)
    for b in (0, 3, 7):
        ro, rl = oracle.paged_decode_attn_e4m3(w.q.numpy()[b:b + 1], k, v, w.k_scale.numpy(),
                                               w.v_scale.numpy(), w.block_tables.numpy()[b:b + 1],
                                               w.seq_lens.numpy()[b:b + 1], w.scale)
        assert_attention_close(out[b:b + 1], lse[b:b + 1], ro, rl, f"sequence {b}")


def test_e4m3_quantisation_error_is_reported(pkv):
    """Not parity (the stored values differ from the bf16 ones): the FP8
    cache's output against the bf16 cache's, on the same data, stays small.
    The pages ask for the accuracy effect of quantisation to be checked."""
    w = workloads.custom(21, [2000, 517], 32, 8, 128, 128, 16)
    dev = "cuda"
    ob, _ = pkv.paged_decode_attn(w.q.to(dev), w.k_pool.to(dev), w.v_pool.to(dev),
                                  w.block_tables.to(dev), w.seq_lens.to(dev), w.scale)
    w = workloads.e4m3(w)
    k, v = w.k_codes.to(dev), w.v_codes.to(dev)
    o8, _ = pkv.paged_decode_attn_e4m3(w.q.to(dev), k, v, w.k_scale.to(dev), w.v_scale.to(dev),
                                       w.block_tables.to(dev), w.seq_lens.to(dev), w.scale)
    torch.cuda.synchronize()
    rel = ((o8 - ob).norm(dim=-1) / ob.norm(dim=-1)).max().item()
    print(f"E4M3 vs bf16 cache: max row rel-L2 {rel:.4f}")
    assert rel < 0.1


# ---------------------------------------------------------------- multi-token

def multi_e4m3_case(seed, cached, T, hq, hkv, dk, dv, bs):
    from tests.test_gpu_multi import multi_case
    return workloads.e4m3(multi_case(seed, cached, T, hq, hkv, dk, dv, bs))


def gpu_multi_e4m3(pkv, w, splits, flags=0, dev="cuda"):
    k, v = w.k_codes.to(dev), w.v_codes.to(dev)
    ks, vs = w.k_scale.to(dev), w.v_scale.to(dev)
    bt = w.block_tables.to(dev)
    slots = pkv.slot_mapping(k, v, bt, w.new_seq.to(dev), w.new_pos.to(dev))
    pkv.kv_append_e4m3(k, v, w.k_new.to(dev), w.v_new.to(dev), slots, ks, vs)
    out, lse = pkv.paged_decode_attn_multi_e4m3(w.q.to(dev), k, v, ks, vs, bt,
                                                w.seq_lens.to(dev), w.scale, num_splits=splits,
                                                flags=flags)
    torch.cuda.synchronize()
    return out.cpu().numpy(), lse.cpu().numpy()


def oracle_multi_e4m3(w):
    """Each (sequence, token) as its own row over the sequence's table, token t
    of T seeing the first seq_lens[b] - T + 1 + t tokens (none if that is not
    positive)."""
    k, v = oracle_e4m3_cache(w)
    B, T = w.q.shape[0], w.q.shape[1]
    L = w.seq_lens.numpy().astype(np.int64)
    q = w.q.numpy().reshape(B * T, *w.q.shape[2:])
    tables = np.repeat(w.block_tables.numpy(), T, axis=0)
    lens = np.array([max(0, L[b] - T + 1 + t) for b in range(B) for t in range(T)],
                    dtype=np.int32)
    out, lse = oracle.paged_decode_attn_e4m3(q, k, v, w.k_scale.numpy(), w.v_scale.numpy(),
                                             tables, lens, w.scale)
    return out.reshape(B, T, *out.shape[1:]), lse.reshape(B, T, -1)


# (cached, T, Hq, Hkv, Dk, Dv, block size): G x T = 16, 8 and 4 rows folded
# into one tensor-core work item (G 4, 8, 4, 2, 1), and shapes run as one
# row per (sequence, token) (G x T = 48, head dim 64, MLA dims)
MULTI_SHAPES = [
    ([300, 7, 64], 4, 32, 8, 128, 128, 16),
    ([129, 40], 2, 16, 2, 128, 128, 32),
    ([90, 12, 200], 2, 16, 4, 128, 128, 32),
    ([150, 33], 2, 8, 4, 128, 128, 16),
    ([70, 4], 4, 4, 4, 128, 128, 64),
    ([150, 40], 4, 16, 2, 128, 128, 16),      # 8 heads x 4 tokens: two head groups
    ([80, 300], 2, 32, 2, 128, 128, 32),      # 16 heads x 2 tokens: two head groups
    ([200, 3], 3, 16, 1, 128, 128, 64),
    ([77, 5], 2, 8, 4, 64, 64, 8),
    ([60, 9], 2, 16, 1, 576, 512, 64),
]


@pytest.mark.parametrize("shape", MULTI_SHAPES,
                         ids=lambda s: f"T{s[1]}_G{s[2]//s[3]}_Dk{s[4]}_bs{s[6]}")
@pytest.mark.parametrize("splits", [1, 3, 0])
def test_e4m3_multi_token_matches_oracle(pkv, shape, splits):
    cached, T, hq, hkv, dk, dv, bs = shape
    w = multi_e4m3_case(700 + T + dk + hq, cached, T, hq, hkv, dk, dv, bs)
    out, lse = gpu_multi_e4m3(pkv, w, splits)
    ro, rl = oracle_multi_e4m3(w)
    assert_attention_close(out, lse, ro, rl, f"e4m3 multi {shape}/{splits}")
    assert pkv.device_status() == 0


def test_e4m3_multi_token_forced_generic_and_causality(pkv):
    """The CUDA-core kernel on a tensor-core shape gives the oracle's rows too;
    and token t of a sequence differs from token t+1 only through the one
    more token it may not see."""
    w = multi_e4m3_case(5, [150, 20], 4, 32, 8, 128, 128, 16)
    out_g, lse_g = gpu_multi_e4m3(pkv, w, 2, flags=pkv.DECODE_GENERIC)
    ro, rl = oracle_multi_e4m3(w)
    assert_attention_close(out_g, lse_g, ro, rl, "forced generic")
    # the oracle's own rows differ between tokens (the causal limit matters)
    assert not np.allclose(rl[:, 0], rl[:, 3])
    assert pkv.device_status() == 0


@pytest.mark.parametrize("splits", [1, 2])
@pytest.mark.parametrize("T,hq", [(3, 16), (4, 8)], ids=["rows_per_token", "folded"])
@pytest.mark.parametrize("held", ["one", "T-1"])
def test_e4m3_multi_token_short_sequence_is_flagged(pkv, splits, T, hq, held):
    """A sequence holding fewer tokens than T (one, or T - 1): its rows with
    no token give out 0 and lse -inf, the device flags the length -- through
    one row per (sequence, token) and through the folded tensor-core rows."""
    n = 1 if held == "one" else T - 1
    w = multi_e4m3_case(9, [20, 0], T, hq, 2, 128, 128, 16)
    w.seq_lens = torch.tensor([20 + T, n], dtype=torch.int32)
    pkv.device_status(reset=True)
    out, lse = gpu_multi_e4m3(pkv, w, splits)
    assert np.isneginf(lse[1, :T - n]).all() and (out[1, :T - n] == 0).all()
    assert np.isfinite(lse[1, T - n:]).all() and np.isfinite(lse[0]).all()
    ro, rl = oracle_multi_e4m3(w)
    assert_attention_close(out, lse, ro, rl, "short")
    assert pkv.device_status(reset=True) & pkv.DEV_SEQ_LEN


def test_e4m3_spec4_full_size_sampled_rows(pkv):
    """Speculative verification at 8 x 32K over an FP8 cache (4 new tokens
    per sequence, the benchmark's split count): whole (sequence, token) rows
    against the oracle."""
    from bench import DEFAULT_SPLITS
    w = workloads.make("spec4_32k_e4m3")
    out, lse = gpu_multi_e4m3(pkv, w, DEFAULT_SPLITS["spec4_32k_e4m3"])
    k, v = oracle_e4m3_cache(w)
    T = w.tokens_per_seq
    for b, t in [(0, 0), (3, 2), (7, 3)]:
        end = np.array([int(w.seq_lens[b]) - (T - 1) + t], dtype=np.int32)
        ro, rl = oracle.paged_decode_attn_e4m3(w.q.numpy()[b:b + 1, t], k, v, w.k_scale.numpy(),
                                               w.v_scale.numpy(), w.block_tables.numpy()[b:b + 1],
                                               w.seq_lens.numpy()[b:b + 1], w.scale, tok_end=end)
        assert_attention_close(out[b, t][None], lse[b, t][None], ro, rl, f"row {b}/{t}")
    assert pkv.device_status() == 0


@pytest.mark.parametrize("interleave", [1, 16])
def test_e4m3_dcp200k_full_size(pkv, interleave):
    """The 200,000-token DCP step over an FP8 cache as the benchmark runs it:
    every token quantised into its interleaved partition, the 4 partitions as
    the rows of one E4M3 call at the benchmark's split count, then merged;
    the pools byte for byte, every partition and the merge against the
    oracle."""
    from bench import DEFAULT_SPLITS
    w = workloads.e4m3(workloads.dcp200k(interleave=interleave))
    N, P, bs = int(w.seq_lens[0]), w.num_parts, w.block_size
    dev = "cuda"
    k, v = w.k_codes.to(dev), w.v_codes.to(dev)
    ks, vs = w.k_scale.to(dev), w.v_scale.to(dev)
    ptab = w.part_tables.to(dev)
    kt, vt = w.k_tokens.to(dev), w.v_tokens.to(dev)
    pkv.kv_append_e4m3(k, v, kt[:N - 1], vt[:N - 1],
                       pkv.interleave_slot_mapping(k, v, 0, N - 1, P, interleave, ptab), ks, vs)
    pkv.kv_append_e4m3(k, v, w.k_new.to(dev), w.v_new.to(dev),
                       pkv.interleave_slot_mapping(k, v, N - 1, 1, P, interleave, ptab), ks, vs)
    plen = torch.tensor([pkv.interleave_partition_len(N, P, interleave, r) for r in range(P)],
                        dtype=torch.int32)
    pq = w.q.to(dev).expand(P, w.num_q_heads, w.head_dim_k).contiguous()
    po, pl = pkv.paged_decode_attn_e4m3(pq, k, v, ks, vs, ptab, plen.to(dev), w.scale,
                                        num_splits=DEFAULT_SPLITS["dcp200k_e4m3"])
    mo, ml = pkv.lse_merge(po.unsqueeze(1), pl.unsqueeze(1))
    torch.cuda.synchronize()
    assert pkv.device_status() == 0
    kc, vc = w.k_codes.numpy().copy(), w.v_codes.numpy().copy()
    part, local = oracle.interleave(N, P, interleave)
    pslots = oracle.slot_mapping(w.part_tables.numpy(), part, local, bs)
    assert oracle.kv_append_e4m3(kc, vc, bits(w.k_tokens), bits(w.v_tokens), w.k_scale.numpy(),
                                 w.v_scale.numpy(), pslots, bs) == 0
    assert np.array_equal(k.cpu().numpy(), kc) and np.array_equal(v.cpu().numpy(), vc)
    counts = np.bincount(part, minlength=P).astype(np.int32)
    assert counts.tolist() == plen.tolist()
    ro, rl = [], []
    for r in range(P):
        o, l = oracle.paged_decode_attn_e4m3(w.q.numpy(), kc, vc, w.k_scale.numpy(),
                                             w.v_scale.numpy(), w.part_tables.numpy()[r:r + 1],
                                             counts[r:r + 1], w.scale)
        ro.append(o)
        rl.append(l)
        assert_attention_close(po[r:r + 1].cpu().numpy(), pl[r:r + 1].cpu().numpy(), o, l,
                               f"partition {r}")
    oo, ol = oracle.lse_merge(np.stack(ro), np.stack(rl))
    assert_attention_close(mo.cpu().numpy(), ml.cpu().numpy(), oo, ol, "merged")
