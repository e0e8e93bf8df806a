"""GPU parity of decode attention and the LSE merge against the oracle, on
small cases that span several tiles and ragged tails, every kernel variant
and the degenerate cases."""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests._steps import assert_attention_close, gpu_step, oracle_step
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
@pytest.mark.parametrize("splits", [1, 2, 3, 16, 0])
@pytest.mark.parametrize("flags", [0, 1])
def test_workload_step_matches_oracle(pkv, name, splits, flags):
    w = workloads.make(name)
    out, lse, k, v, slots = gpu_step(pkv, w, num_splits=splits, flags=flags)
    ro, rl, ok_, ov_, oslots = oracle_step(w)
    assert np.array_equal(slots.cpu().numpy(), oslots)
    assert np.array_equal(bits(k.cpu()), ok_) and np.array_equal(bits(v.cpu()), ov_)
    assert_attention_close(out.cpu().numpy(), lse.cpu().numpy(), ro, rl, f"{name}/{splits}/{flags}")
    assert pkv.device_status() == 0


# (cached lengths, Hq, Hkv, D, block size): every tensor-core variant (G = 1,
# 2, 4, 8; D = 64, 128; block sizes 8..256) plus generic-only shapes.
SHAPES = [
    ([0, 1, 15, 16, 63, 64, 65, 200], 8, 8, 128, 16),     # G=1
    ([5, 130, 77], 16, 8, 128, 32),                       # G=2
    ([300, 1, 64], 8, 2, 64, 8),                          # G=4, D=64
    ([1000, 513, 7], 16, 2, 128, 64),                     # G=8
    ([700, 129], 8, 1, 64, 128),                          # G=8, D=64, bs 128
    ([520, 3], 4, 1, 128, 256),                           # G=4, bs 256
    ([0, 300, 1, 77], 128, 8, 128, 16),                   # G=16 (128 heads over 8)
    ([450, 31], 32, 2, 64, 32),                           # G=16, D=64
    ([90, 45], 12, 4, 128, 16),                           # G=3: generic kernel
    ([33, 17], 4, 2, 96, 16),                             # D=96: generic kernel
    ([40, 21], 8, 2, 128, 4),                             # bs 4: generic kernel
    ([60], 16, 1, 256, 16),                               # D=256: generic kernel
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"G{s[1]//s[2]}_D{s[3]}_bs{s[4]}")
@pytest.mark.parametrize("splits", [1, 4, 0])
def test_shape_sweep(pkv, shape, splits):
    cached, hq, hkv, d, bs = shape
    w = workloads.custom(100 + d + bs, cached, hq, hkv, d, d, bs)
    out, lse, *_ = gpu_step(pkv, w, num_splits=splits)
    ro, rl, *_ = oracle_step(w)
    assert_attention_close(out.cpu().numpy(), lse.cpu().numpy(), ro, rl, f"{shape}/{splits}")
    assert pkv.device_status() == 0


@pytest.mark.parametrize("cached,hq,hkv,bs", [([0, 300, 1, 77], 128, 8, 16),
                                              ([600, 65], 64, 4, 64), ([200], 16, 1, 256),
                                              ([129, 40, 255], 32, 2, 32), ([700, 5], 16, 1, 128)],
                         ids=["128q_8kv_bs16", "64q_4kv_bs64", "16q_1kv_bs256", "32q_2kv_bs32",
                              "16q_1kv_bs128"])
@pytest.mark.parametrize("splits", [1, 4])
@pytest.mark.parametrize("flags", ["auto", "no_tcgen05"])
def test_group_of_16(pkv, cached, hq, hkv, bs, splits, flags):
    """16 query heads per KV head (head dim 128): the tcgen05 GQA kernel, and
    with no_tcgen05 the warp-level-MMA G = 16 instance."""
    w = workloads.custom(71 + bs, cached, hq, hkv, 128, 128, bs)
    f = pkv.DECODE_NO_TCGEN05 if flags == "no_tcgen05" else 0
    out, lse, *_ = gpu_step(pkv, w, num_splits=splits, flags=f)
    ro, rl, *_ = oracle_step(w)
    assert_attention_close(out.cpu().numpy(), lse.cpu().numpy(), ro, rl, f"G16/{splits}/{flags}")
    assert pkv.device_status() == 0


@pytest.mark.parametrize("splits", [1, 3])
def test_group_of_16_rising_scores(pkv, splits):
    """Keys grow along the sequence, so each row's running max keeps rising
    past the slack: the tcgen05 GQA kernel rescales its accumulator in TMEM."""
    w = workloads.custom(92, [1500, 700], 32, 2, 128, 128, 16)
    k = w.k_pool.float()
    L = w.seq_lens.tolist()
    for b in range(2):
        for j in range(L[b]):
            blk = int(w.block_tables[b, j // 16])
            k[blk, :, j % 16] *= 1.0 + 6.0 * j / L[b]
    w.k_pool = k.to(torch.bfloat16)
    out, lse, *_ = gpu_step(pkv, w, num_splits=splits)
    ro, rl, *_ = oracle_step(w)
    assert_attention_close(out.cpu().numpy(), lse.cpu().numpy(), ro, rl, f"rising/{splits}")
    assert pkv.device_status() == 0


def test_distinct_k_and_v_dims(pkv):
    w = workloads.custom(7, [70, 3], 16, 1, 576, 512, 64)
    out, lse, *_ = gpu_step(pkv, w, num_splits=2)
    ro, rl, *_ = oracle_step(w)
    assert_attention_close(out.cpu().numpy(), lse.cpu().numpy(), ro, rl, "576/512")


@pytest.mark.parametrize("flags", [0, 1, 2])
@pytest.mark.parametrize("hq", [16, 64], ids=["G4", "G16"])
def test_partials_match_oracle_token_ranges(pkv, flags, hq):
    """Split s of row b covers [s*C, min(L, (s+1)*C)), C = 64*ceil(L/(64*S));
    a row of length 0 is an empty row, not a flagged one."""
    w = workloads.custom(31, [400, 70, 1, 0], hq, 4, 128, 128, 16)
    S = 5
    dev = "cuda"
    k, v, bt = w.k_pool.to(dev), w.v_pool.to(dev), w.block_tables.to(dev)
    lens = w.seq_lens.clone()
    lens[3] = 0
    op, lp = pkv.paged_decode_attn_partial(w.q.to(dev), k, v, bt, lens.to(dev), w.scale, S,
                                           flags=flags)
    assert pkv.device_status() == 0
    kb, vb = bits(w.k_pool), bits(w.v_pool)
    L = lens.numpy().astype(np.int64)
    C = 64 * (-(-L // (64 * S)))
    for s in range(S):
        begin = np.minimum(s * C, L).astype(np.int32)
        end = np.minimum((s + 1) * C, L).astype(np.int32)
        ro, rl = oracle.paged_decode_attn(w.q.numpy(), kb, vb, w.block_tables.numpy(), L,
                                          w.scale, tok_begin=begin, tok_end=end)
        assert_attention_close(op[s].cpu().numpy(), lp[s].cpu().numpy(), ro, rl, f"split {s}")
    # merging the partials on the GPU gives the unsplit oracle result
    mo, ml = pkv.lse_merge(op, lp)
    ro, rl = oracle.paged_decode_attn(w.q.numpy(), kb, vb, w.block_tables.numpy(), L, w.scale)
    assert_attention_close(mo.cpu().numpy(), ml.cpu().numpy(), ro, rl, "merged partials")


@pytest.mark.parametrize("P,empty", [(1, 0.0), (4, 0.0), (16, 0.3), (40, 0.5), (3, 1.0)])
def test_lse_merge_matches_oracle(pkv, P, empty):
    out_p, lse_p = workloads.random_partials(50 + P, P, 3, 8, 128, empty_fraction=empty)
    mo, ml = pkv.lse_merge(out_p.cuda(), lse_p.cuda())
    ro, rl = oracle.lse_merge(out_p.numpy(), lse_p.numpy())
    assert_attention_close(mo.cpu().numpy(), ml.cpu().numpy(), ro, rl, f"merge P={P}")


def test_merge_of_far_apart_partials(pkv):
    out_p = torch.tensor([[[1.0] * 8], [[3.0] * 8], [[0.0] * 8]])
    lse_p = torch.tensor([[-500.0], [400.0], [float("-inf")]])
    mo, ml = pkv.lse_merge(out_p.cuda(), lse_p.cuda())
    assert mo.cpu().tolist() == [[3.0] * 8] and ml.cpu().tolist() == [400.0]


@pytest.mark.parametrize("hq", [8, 32], ids=["G4", "G16"])
def test_single_token_is_exact_value(pkv, hq):
    w = workloads.custom(9, [0, 0], hq, 2, 128, 128, 16)
    out, lse, k, v, _ = gpu_step(pkv, w, num_splits=1)
    ro, rl, *_ = oracle_step(w)
    # one token: out is exactly its V row (in fp32)
    vv = w.v_new.float().numpy()
    for b in range(2):
        for h in range(hq):
            assert np.array_equal(out[b, h].cpu().numpy(), vv[b, h // (hq // 2)])
    assert np.abs(lse.cpu().numpy() - rl).max() <= 1e-4


@pytest.mark.parametrize("hq", [8, 32], ids=["G4", "G16"])
def test_bad_seq_len_and_block_id_are_flagged_not_faulted(pkv, hq):
    w = workloads.custom(12, [100, 100], hq, 2, 128, 128, 16)
    dev = "cuda"
    k, v = w.k_pool.to(dev), w.v_pool.to(dev)
    q = w.q.to(dev)
    lens = w.seq_lens.clone()
    lens[1] = 10_000                       # longer than its table
    for flags in (0, 1, 2):
        out, lse = pkv.paged_decode_attn(q, k, v, w.block_tables.to(dev), lens.to(dev), w.scale,
                                         num_splits=2, flags=flags)
        assert pkv.device_status() == pkv.DEV_SEQ_LEN
        assert torch.isneginf(lse[1]).all() and (out[1] == 0).all()
        assert torch.isfinite(lse[0]).all()
        bt = w.block_tables.clone()
        bt[0, 3] = 1 << 20                 # block id outside the pool
        out, lse = pkv.paged_decode_attn(q, k, v, bt.to(dev), w.seq_lens.to(dev), w.scale,
                                         num_splits=2, flags=flags)
        assert pkv.device_status() == pkv.DEV_BLOCK_ID
        assert torch.isfinite(out).all() and torch.isfinite(lse).all()


@pytest.mark.parametrize("hq", [16, 32], ids=["G8", "G16"])
def test_unused_slots_holding_nan_do_not_leak(pkv, hq):
    """Slots past the end of a sequence's last block may hold any bits."""
    w = workloads.custom(13, [20, 50], hq, 2, 128, 128, 16, extra_blocks=0)
    k, v = w.k_pool.clone(), w.v_pool.clone()
    for b in range(2):
        L = int(w.seq_lens[b])
        last = int(w.block_tables[b, (L - 1) // 16])
        k[last, :, L % 16 or 16:] = float("nan")
        v[last, :, L % 16 or 16:] = float("nan")
    w.k_pool, w.v_pool = k, v
    for flags in (0, 1):
        out, lse, *_ = gpu_step(pkv, w, num_splits=1, flags=flags)
        assert torch.isfinite(out).all() and torch.isfinite(lse).all()
        ro, rl, *_ = oracle_step(w)
        assert_attention_close(out.cpu().numpy(), lse.cpu().numpy(), ro, rl, "nan tail")


def test_batch_zero_and_empty_work(pkv):
    q = torch.empty(0, 8, 128, device="cuda")
    k = torch.zeros(4, 2, 16, 128, dtype=torch.bfloat16, device="cuda")
    out, lse = pkv.paged_decode_attn(q, k, k, torch.zeros(0, 1, dtype=torch.int32, device="cuda"),
                                     torch.zeros(0, dtype=torch.int32, device="cuda"), 0.1,
                                     num_splits=1)
    assert out.shape == (0, 8, 128) and lse.shape == (0, 8)
    pkv.kv_append(k, k, torch.empty(0, 2, 128, dtype=torch.bfloat16, device="cuda"),
                  torch.empty(0, 2, 128, dtype=torch.bfloat16, device="cuda"),
                  torch.empty(0, dtype=torch.int64, device="cuda"))
    assert pkv.device_status() == 0


def test_scale_is_applied(pkv):
    w = workloads.custom(14, [90], 8, 2, 64, 64, 16)
    w.scale = 0.37 / math.sqrt(64)
    out, lse, *_ = gpu_step(pkv, w, num_splits=2)
    ro, rl, *_ = oracle_step(w)
    assert_attention_close(out.cpu().numpy(), lse.cpu().numpy(), ro, rl, "scale")


def test_workspace_reused_across_calls(pkv):
    """One workspace, filled with garbage first, serves many calls, shapes and
    split counts in a row: each call clears the completion counters it uses."""
    big = workloads.custom(41, [300, 90, 1000, 0, 17, 64], 32, 8, 128, 128, 16)
    small = workloads.custom(42, [40, 700], 16, 2, 128, 128, 32)
    need = max(pkv.decode_workspace_size(6, 32, 128, 7), pkv.decode_workspace_size(2, 16, 128, 5))
    ws = torch.randint(0, 255, (need,), dtype=torch.uint8, device="cuda")
    for w, splits in [(big, 7), (small, 5), (big, 3), (small, 5), (big, 7)]:
        ro, rl, *_ = oracle_step(w)
        k, v = w.k_pool.cuda(), w.v_pool.cuda()
        slots = pkv.slot_mapping(k, v, w.block_tables.cuda(), w.new_seq.cuda(), w.new_pos.cuda())
        pkv.kv_append(k, v, w.k_new.cuda(), w.v_new.cuda(), slots)
        out, lse = pkv.paged_decode_attn(w.q.cuda(), k, v, w.block_tables.cuda(),
                                         w.seq_lens.cuda(), w.scale, num_splits=splits,
                                         workspace=ws)
        torch.cuda.synchronize()
        assert_attention_close(out.cpu().numpy(), lse.cpu().numpy(), ro, rl, f"reuse {splits}")
    assert pkv.device_status() == 0


# Large query groups (multiples of 32) run on the MLA-shaped tensor-core
# kernel: (cached lengths, Hq, Hkv, Dk, Dv, block size).
MLA_SHAPES = [
    ([70, 3, 200], 32, 1, 576, 512, 64),
    ([130, 1], 128, 1, 576, 512, 64),
    ([300, 45], 64, 2, 128, 128, 32),      # G 32, D 128: tcgen05 GQA, two head groups
    ([513, 0, 31], 64, 1, 192, 256, 128),
    ([1000], 32, 1, 64, 64, 256),
    # multiples of 64 heads: the tcgen05 kernel (ragged tiles, two KV heads,
    # block sizes 64 and 256, head dims up to 576 / 512)
    ([127, 128, 255, 1, 700], 128, 2, 576, 512, 64),
    ([2000, 63], 64, 1, 512, 512, 256),
    ([383], 192, 1, 128, 384, 128),
]


@pytest.mark.parametrize("shape", MLA_SHAPES,
                         ids=lambda s: f"G{s[1]//s[2]}_Dk{s[3]}_Dv{s[4]}_bs{s[5]}")
@pytest.mark.parametrize("splits", [1, 3, 0])
@pytest.mark.parametrize("flags", [0, "no_tcgen05"])
def test_large_group_kernel(pkv, shape, splits, flags):
    """Large query groups; with no_tcgen05 the warp-level-MMA kernel takes the
    shapes the tcgen05 kernel would have run."""
    cached, hq, hkv, dk, dv, bs = shape
    f = pkv.DECODE_NO_TCGEN05 if flags == "no_tcgen05" else 0
    w = workloads.custom(200 + dk + bs, cached, hq, hkv, dk, dv, bs)
    out, lse, *_ = gpu_step(pkv, w, num_splits=splits, flags=f)
    ro, rl, *_ = oracle_step(w)
    assert_attention_close(out.cpu().numpy(), lse.cpu().numpy(), ro, rl,
                           f"{shape}/{splits}/{flags}")
    assert pkv.device_status() == 0


@pytest.mark.parametrize("flags", [0, "no_tcgen05"])
@pytest.mark.parametrize("splits", [1, 2])
def test_large_group_rising_scores(pkv, flags, splits):
    """Keys grow along the sequence, so a head's running max keeps rising
    (by more than 2^8 in probability between tiles): the kernels must rescale
    what they have accumulated, in TMEM for the tcgen05 kernel."""
    w = workloads.custom(91, [1500, 700], 128, 1, 576, 512, 64)
    k = w.k_pool.float()
    L = w.seq_lens.tolist()
    for b in range(2):
        for j in range(L[b]):
            blk = int(w.block_tables[b, j // 64])
            k[blk, :, j % 64] *= 1.0 + 5.0 * j / L[b]
    w.k_pool = k.to(torch.bfloat16)
    f = pkv.DECODE_NO_TCGEN05 if flags == "no_tcgen05" else 0
    out, lse, *_ = gpu_step(pkv, w, num_splits=splits, flags=f)
    ro, rl, *_ = oracle_step(w)
    assert_attention_close(out.cpu().numpy(), lse.cpu().numpy(), ro, rl, f"rising/{splits}")
    assert pkv.device_status() == 0


def test_large_group_partials_and_nan_tail(pkv):
    """Per-split partials of the large-group kernel against the oracle's token
    ranges, with NaN bits in the unused slots of each last block."""
    w = workloads.custom(77, [150, 9], 64, 1, 576, 512, 64, extra_blocks=0)
    k, v = w.k_pool.clone(), w.v_pool.clone()
    for b in range(2):
        L = int(w.seq_lens[b])
        last = int(w.block_tables[b, (L - 1) // 64])
        k[last, :, L % 64 or 64:] = float("nan")
        v[last, :, L % 64 or 64:] = float("nan")
    w.k_pool, w.v_pool = k, v
    S = 3
    dev = "cuda"
    op, lp = pkv.paged_decode_attn_partial(w.q.to(dev), w.k_pool.to(dev), w.v_pool.to(dev),
                                           w.block_tables.to(dev), w.seq_lens.to(dev), w.scale, S)
    torch.cuda.synchronize()
    assert torch.isfinite(op).all()
    kb, vb = bits(w.k_pool), bits(w.v_pool)
    L = w.seq_lens.numpy().astype(np.int64)
    C = 64 * (-(-L // (64 * S)))
    for s in range(S):
        begin = np.minimum(s * C, L).astype(np.int32)
        end = np.minimum((s + 1) * C, L).astype(np.int32)
        ro, rl = oracle.paged_decode_attn(w.q.numpy(), kb, vb, w.block_tables.numpy(), L,
                                          w.scale, tok_begin=begin, tok_end=end)
        assert_attention_close(op[s].cpu().numpy(), lp[s].cpu().numpy(), ro, rl, f"split {s}")
    assert pkv.device_status() == 0
