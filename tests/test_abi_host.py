"""CPU tests of the C ABI library: it loads, exports every function
include/pkv.h declares, and its host-only logic (argument checks that fail
before any CUDA call, workspace sizing, the partition-length rule and the
block manager) is right.  No compute call reaches a GPU here."""
from __future__ import annotations

import ctypes
import os
import re

import numpy as np
import pytest

import oracle
from tests._util import golden

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pkv.h")


@pytest.fixture(scope="module")
def pkv():
    import __graft_entry__
    __graft_entry__.build()
    import paged_kv_cache_93_gb300 as m
    return m


def declared_functions():
    text = open(HEADER, encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b(pkv_[a-z0-9_]+)\s*\(", text)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ["pkv_kv_append", "pkv_paged_decode_attn", "pkv_paged_decode_attn_partial",
              "pkv_lse_merge", "pkv_copy_blocks", "pkv_slot_mapping",
              "pkv_interleave_slot_mapping", "pkv_decode_workspace_size", "pkv_status_string",
              "pkv_device_status", "pkv_bm_create", "pkv_bm_append"]:
        assert n in names


def test_library_exports_every_declared_symbol(pkv):
    lib = ctypes.CDLL(pkv.library_path)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing
    from paged_kv_cache_93_gb300 import _lib
    assert set(_lib.SIGNATURES) == set(declared_functions())


def test_withhold_control_is_refused_unless_enabled(pkv):
    """The test control of the failure path is an unknown flag until a test
    enables it, and the entry points that never take it refuse it always
    (host checks: nothing reaches a GPU)."""
    lib = pkv.lib
    desc = pkv.CacheDesc(16, 16, 8, 128, 128)
    p = ctypes.c_void_p(0x1000)
    f = pkv.DECODE_TEST_WITHHOLD
    assert lib.pkv_test_enable_withhold(0) == 0
    assert lib.pkv_paged_decode_attn(ctypes.byref(desc), p, 1, 32, p, p, p, 4, p, 1.0, 1, None, 0,
                                     p, p, f, None) == -1
    assert lib.pkv_paged_decode_attn_partial(ctypes.byref(desc), p, 1, 32, p, p, p, 4, p, 1.0, 1,
                                             p, p, f, None) == -1
    try:
        assert lib.pkv_test_enable_withhold(1) == 0
        assert lib.pkv_paged_decode_attn_e4m3(ctypes.byref(desc), p, 1, 32, p, p, p, p, p, 4, p,
                                              1.0, 1, None, 0, p, p, f, None) == -1
        assert lib.pkv_paged_decode_attn_multi(ctypes.byref(desc), p, 1, 2, 32, p, p, p, 4, p,
                                               1.0, 1, p, 1 << 20, p, p, f, None) == -1
    finally:
        lib.pkv_test_enable_withhold(0)


def test_status_strings(pkv):
    for code in range(0, -9, -1):
        s = pkv.lib.pkv_status_string(code).decode()
        assert s and s != "unknown status"
    assert pkv.lib.pkv_status_string(-99).decode() == "unknown status"


def test_host_validation_rejects_before_any_launch(pkv):
    lib = pkv.lib
    desc = pkv.CacheDesc(16, 16, 8, 128, 128)
    # null pools / inputs: rejected by the host checks
    assert lib.pkv_kv_append(ctypes.byref(desc), None, None, None, None, None, 4, None) == -1
    assert lib.pkv_copy_blocks(ctypes.byref(desc), None, None, None, None, 2, None) == -1
    assert lib.pkv_slot_mapping(ctypes.byref(desc), None, 1, 1, None, None, 3, None, None) == -1
    # zero-sized work is a no-op success
    assert lib.pkv_kv_append(ctypes.byref(desc), None, None, None, None, None, 0, None) == 0
    # misaligned pointers
    bad = ctypes.c_void_p(0x1008)
    assert lib.pkv_kv_append(ctypes.byref(desc), bad, bad, bad, bad, bad, 1, None) == -3
    # Hq not a multiple of Hkv -> shape error; bad flag -> invalid arg
    p = ctypes.c_void_p(0x1000)
    assert lib.pkv_paged_decode_attn(ctypes.byref(desc), p, 1, 12, p, p, p, 4, p, 1.0, 1, None, 0,
                                     p, p, 0, None) == -2
    assert lib.pkv_paged_decode_attn(ctypes.byref(desc), p, 1, 16, p, p, p, 4, p, 1.0, 1, None, 0,
                                     p, p, 4, None) == -1
    assert lib.pkv_paged_decode_attn(ctypes.byref(desc), p, 1, 16, p, p, p, 4, p, 1.0, 300, None,
                                     0, p, p, 0, None) == -1
    # splits > 1 without workspace
    assert lib.pkv_paged_decode_attn(ctypes.byref(desc), p, 1, 16, p, p, p, 4, p, 1.0, 4, None, 0,
                                     p, p, 0, None) == -4
    # head dim not a multiple of 8
    d2 = pkv.CacheDesc(16, 16, 8, 100, 128)
    assert lib.pkv_paged_decode_attn(ctypes.byref(d2), p, 1, 16, p, p, p, 4, p, 1.0, 1, None, 0,
                                     p, p, 0, None) in (-1, -2)
    assert lib.pkv_lse_merge(0, p, p, 4, 128, p, p, None) == -1


def test_multi_token_host_rules(pkv):
    lib = pkv.lib
    p = ctypes.c_void_p(0x1000)
    desc = pkv.CacheDesc(16, 16, 8, 128, 128)
    args = lambda T, S, ws, nbytes: (ctypes.byref(desc), p, 2, T, 32, p, p, p, 4, p, 1.0, S, ws,
                                     nbytes, p, p, 0, None)
    assert lib.pkv_paged_decode_attn_multi(*args(0, 2, p, 1 << 30)) == -1     # no query token
    assert lib.pkv_paged_decode_attn_multi(*args(65, 2, p, 1 << 30)) == -1    # more than 64
    need = lib.pkv_decode_multi_workspace_size(2, 4, 32, 128, 4, 2)
    # the per-token views of the tables + the split partials of 8 rows
    assert need >= 2 * 4 * 4 * 4 + 2 * 4 * 4 + pkv.decode_workspace_size(8, 32, 128, 2)
    assert lib.pkv_paged_decode_attn_multi(*args(4, 2, None, 0)) == -4
    assert lib.pkv_paged_decode_attn_multi(*args(4, 2, p, need - 1)) == -4
    assert lib.pkv_decode_multi_workspace_size(2, 0, 32, 128, 4, 2) == 0


def test_values_inside_keys_host_rules(pkv):
    """v_pool NULL = the values are the first head_dim_v dims of each key row:
    append needs v_new NULL as well, and head_dim_v may not exceed head_dim_k."""
    lib = pkv.lib
    p = ctypes.c_void_p(0x1000)
    latent = pkv.CacheDesc(16, 64, 1, 576, 512)
    wide = pkv.CacheDesc(16, 64, 1, 128, 256)
    # one of v_pool / v_new NULL, the other not
    assert lib.pkv_kv_append(ctypes.byref(latent), p, None, p, p, p, 1, None) == -1
    assert lib.pkv_kv_append(ctypes.byref(latent), p, p, p, None, p, 1, None) == -1
    # values wider than the keys cannot live inside them
    assert lib.pkv_kv_append(ctypes.byref(wide), p, None, p, None, p, 1, None) == -2
    assert lib.pkv_copy_blocks(ctypes.byref(wide), p, None, p, p, 1, None) == -2
    assert lib.pkv_paged_decode_attn(ctypes.byref(wide), p, 1, 16, p, None, p, 4, p, 1.0, 1,
                                     None, 0, p, p, 0, None) == -2
    assert lib.pkv_paged_decode_attn_partial(ctypes.byref(wide), p, 1, 16, p, None, p, 4, p,
                                             1.0, 2, p, p, 0, None) == -2


def test_workspace_size(pkv):
    assert pkv.decode_workspace_size(8, 32, 128, 1) == 0
    n = pkv.decode_workspace_size(8, 32, 128, 16)
    rows = 16 * 8 * 32
    assert n >= rows * 128 * 4 + rows * 4
    assert n % 256 == 0


@pytest.mark.parametrize("N,P,I", [(200_000, 4, 1), (200_000, 4, 16), (1000, 3, 7), (5, 4, 2),
                                   (0, 2, 3), (17, 1, 4)])
def test_partition_len_matches_oracle_count(pkv, N, P, I):
    part, _ = oracle.interleave(N, P, I)
    counts = np.bincount(part, minlength=P)
    assert [pkv.interleave_partition_len(N, P, I, r) for r in range(P)] == counts.tolist()


def test_partition_len_dcp_example(pkv):
    gd = golden("dcp_interleave.txt")
    for I in (1, 16):
        assert [pkv.interleave_partition_len(gd["num_tokens"], gd["dcp_size"], I, r)
                for r in range(gd["dcp_size"])] == [gd["tokens_per_partition"]] * gd["dcp_size"]


# ------------------------------------------------------------- block manager

def test_block_manager_accounting_example(pkv):
    """The worked example: block size 4; A holds 6 tokens, B 9; A ends and its
    blocks serve a new request; B grows to 12 (no new block) then 13 (one)."""
    gd = golden("block_accounting.txt")
    bs = gd["block_size"]
    bm = pkv.BlockManager(8, bs)
    a, b = bm.add_sequence(), bm.add_sequence()
    slots_a, _ = bm.append(a, gd["tokens_A"])
    slots_b, _ = bm.append(b, gd["tokens_B"])
    ta, tb = bm.block_table(a), bm.block_table(b)
    assert (len(ta), len(tb)) == (gd["blocks_A"], gd["blocks_B"])
    assert (len(ta) + len(tb)) * bs - gd["total_tokens"] == gd["slack_slots"]
    assert bm.num_free == 8 - gd["blocks_A"] - gd["blocks_B"]
    # slots follow each table
    assert slots_b == [oracle.slot_of(np.array(tb, np.int32), j, bs) for j in range(len(slots_b))]
    bm.free(a)
    assert bm.num_free == 8 - gd["blocks_B"]
    assert all(bm.ref_count(x) == 0 for x in ta)
    c = bm.add_sequence()
    bm.append(c, 3)
    assert bm.block_table(c)[0] in ta        # a returned block is reused
    bm.append(b, gd["B_grown_tokens"] - gd["tokens_B"])
    assert len(bm.block_table(b)) == gd["B_grown_blocks"]
    bm.append(b, gd["B_next_tokens"] - gd["B_grown_tokens"])
    tb2 = bm.block_table(b)
    assert len(tb2) == gd["B_next_blocks"] and tb2[:3] == tb   # no compaction
    assert tb2[3] in ta                                        # A's other block


def test_block_manager_shared_blocks_and_copy_on_write(pkv):
    bm = pkv.BlockManager(10, 4, initial_order=[9, 8, 7, 6, 5, 4, 3, 2, 1, 0])
    p = bm.add_sequence()
    bm.append(p, 10)                     # blocks 9, 8, 7 (tail holds 2)
    tp = bm.block_table(p)
    assert tp == [9, 8, 7]
    c1, c2 = bm.fork(p), bm.fork(p)
    assert all(bm.ref_count(x) == 3 for x in tp)
    slots, cow = bm.append(c1, 1)        # writes into shared tail -> copy-on-write
    assert len(cow) == 1 and cow[0][0] == 7
    new_tail = cow[0][1]
    assert bm.block_table(c1) == [9, 8, new_tail] and slots == [new_tail * 4 + 2]
    assert bm.ref_count(7) == 2 and bm.ref_count(new_tail) == 1
    assert bm.block_table(p) == tp and bm.block_table(c2) == tp   # others unchanged
    # a full shared block is never copied: fill c2's tail privately, then grow
    _, cow2 = bm.append(c2, 2)
    assert len(cow2) == 1
    _, cow3 = bm.append(c2, 1)
    assert cow3 == []
    # freeing keeps blocks that others still use
    bm.free(p)
    assert bm.ref_count(9) == 2 and bm.ref_count(7) == 0
    bm.free(c1)
    bm.free(c2)
    assert bm.num_free == 10


def test_block_manager_no_space_is_all_or_nothing(pkv):
    bm = pkv.BlockManager(3, 4)
    s = bm.add_sequence()
    bm.append(s, 10)
    with pytest.raises(pkv.PkvError) as e:
        bm.append(s, 5)                  # needs 2 more blocks, only 0 free
    assert e.value.status == -7
    assert bm.seq_len(s) == 10 and bm.num_free == 0
    with pytest.raises(pkv.PkvError):
        bm.free(12345)


def test_block_manager_rejects_bad_order(pkv):
    with pytest.raises(ValueError):
        pkv.BlockManager(3, 4, initial_order=[0, 0, 1])


def test_e4m3_host_rules(pkv):
    """The E4M3 entry points refuse, before any device work: undefined flags,
    missing scales or value pool, bad shapes, misaligned code pools, block
    copies whose rows are not whole 16-byte vectors."""
    lib = pkv.lib
    p = ctypes.c_void_p(0x1000)
    odd = ctypes.c_void_p(0x1004)
    ok = pkv.CacheDesc(16, 16, 2, 128, 128)
    d12 = pkv.CacheDesc(16, 16, 2, 12, 12)

    def attn(desc, hq, k_scale=p, v_scale=p, v_pool=p, flags=0):
        return lib.pkv_paged_decode_attn_e4m3(ctypes.byref(desc), p, 1, hq, p, v_pool, k_scale,
                                              v_scale, p, 4, p, 1.0, 1, None, 0, p, p, flags,
                                              None)
    assert attn(ok, 8, flags=8) == -1                  # undefined flag bit
    assert attn(ok, 8, k_scale=None) == -1
    assert attn(ok, 8, v_scale=None) == -1
    assert attn(ok, 8, v_pool=None) == -1
    assert attn(ok, 3) == -2                           # heads not a multiple of KV heads
    assert attn(d12, 8) == -2                          # head dims multiples of 8
    assert lib.pkv_kv_append_e4m3(ctypes.byref(ok), p, p, p, p, None, p, p, 1, None) == -1
    assert lib.pkv_kv_append_e4m3(ctypes.byref(ok), odd, p, p, p, p, p, p, 1, None) == -3
    assert lib.pkv_copy_blocks_e4m3(ctypes.byref(ok), p, None, p, p, 1, None) == -1
    one = pkv.CacheDesc(16, 1, 1, 8, 8)                # 8-byte block rows
    assert lib.pkv_copy_blocks_e4m3(ctypes.byref(one), p, p, p, p, 1, None) == -2
    # the split choice: enough items for the resident CTAs
    assert 1 <= lib.pkv_decode_auto_splits_e4m3(ctypes.byref(ok), 8, 8, 32768) <= 256

    def partial(S=1, out_part=p, lse_part=p, k_scale=p, flags=0):
        return lib.pkv_paged_decode_attn_partial_e4m3(ctypes.byref(ok), p, 1, 8, p, p, k_scale,
                                                      p, p, 4, p, 1.0, S, out_part, lse_part,
                                                      flags, None)
    assert partial(S=0) == -1                          # the partials need S >= 1
    assert partial(out_part=None) == -1
    assert partial(lse_part=None) == -1
    assert partial(k_scale=None) == -1
    assert partial(out_part=odd) == -3                 # out_part 16-byte aligned
    assert partial(flags=pkv.DECODE_TEST_WITHHOLD) == -1


def test_binding_keeps_code_pools_out_of_bf16_calls(pkv):
    """The bf16 calls size rows at two bytes an element; the binding refuses
    one-byte code pools for them (they have E4M3 forms) before any C call."""
    import torch
    k = torch.zeros(4, 1, 16, 64, dtype=torch.uint8)
    v = torch.zeros(4, 1, 16, 64, dtype=torch.uint8)
    i32 = torch.zeros(1, dtype=torch.int32)
    q = torch.zeros(1, 2, 64)
    bt = torch.zeros(1, 4, dtype=torch.int32)
    with pytest.raises(TypeError, match="k_pool must be torch.bfloat16"):
        pkv.copy_blocks(k, v, i32, i32)
    with pytest.raises(TypeError, match="k_pool must be torch.bfloat16"):
        pkv.kv_append(k, v, torch.zeros(1, 1, 64, dtype=torch.bfloat16),
                      torch.zeros(1, 1, 64, dtype=torch.bfloat16), torch.zeros(1, dtype=torch.int64))
    with pytest.raises(TypeError, match="k_pool must be torch.bfloat16"):
        pkv.paged_decode_attn(q, k, v, bt, i32, 0.125)
    with pytest.raises(TypeError, match="k_pool must be torch.bfloat16"):
        pkv.paged_decode_attn_partial(q, k, v, bt, i32, 0.125, 2)
