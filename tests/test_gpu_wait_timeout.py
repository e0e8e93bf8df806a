"""The failure path of the pipelined decode kernels, made to run on purpose
and without any fault.

Every wait of a kernel's copy/compute pipeline is bounded; when one runs out
the kernel raises PKV_DEV_TIMEOUT in the device status word, every role of
the CTA leaves its loop with nothing in flight, and the rows of every work
item the CTA gave up on come back NaN (output and LSE; the merge passes a NaN
partial on).  The test control PKV_DECODE_TEST_WITHHOLD (enabled only through
pkv_test_enable_withhold) makes the copy producer issue no copy at all and
limits each wait to 1 ms, so the first wait for a copy runs out while
nothing is in flight.  Checked for the warp-level GQA kernel and the tcgen05
large-group kernel: the call returns promptly, the status word holds
PKV_DEV_TIMEOUT, every row is reported NaN, and the next ordinary call on
the same device is right (against the oracle) with a clean status word;
also for the large-group kernel's E4M3 mode, whose converter warps wait for
codes that never land.
"""
from __future__ import annotations

import time

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests._steps import assert_attention_close
from tests._util import bits

pytestmark = pytest.mark.gpu

# (name, workloads.custom arguments: seed, cached lengths, Hq, Hkv, Dk, Dv, block size, splits)
CASES = [
    ("gqa_tma", (21, [700, 300, 64], 32, 8, 128, 128, 16), 3),    # warp-level GQA kernel
    ("gqa_tma_one_split", (23, [257, 90], 32, 8, 128, 128, 16), 1),
    ("mla_tc", (22, [900, 200], 128, 1, 576, 512, 64), 2),        # tcgen05 large-group kernel
]


@pytest.fixture(scope="module")
def pkv():
    import __graft_entry__
    __graft_entry__.build()
    import paged_kv_cache_93_gb300 as m
    m.device_status(reset=True)
    return m


def _inputs(w, dev="cuda"):
    return (w.q.to(dev), w.k_pool.to(dev), w.v_pool.to(dev), w.block_tables.to(dev),
            w.seq_lens.to(dev))


@pytest.mark.parametrize("name, shape, splits", CASES, ids=[c[0] for c in CASES])
def test_wait_that_runs_out_is_reported_and_the_device_recovers(pkv, name, shape, splits):
    w = workloads.custom(*shape)
    q, k, v, bt, lens = _inputs(w)
    assert pkv.device_status(reset=True) == 0
    assert pkv.lib.pkv_test_enable_withhold(1) == 0
    try:
        t0 = time.perf_counter()
        out, lse = pkv.paged_decode_attn(q, k, v, bt, lens, w.scale, num_splits=splits,
                                         flags=pkv.DECODE_TEST_WITHHOLD)
        torch.cuda.synchronize()
        elapsed = time.perf_counter() - t0
    finally:
        pkv.lib.pkv_test_enable_withhold(0)
    assert elapsed < 10.0, f"{name}: the call took {elapsed:.1f} s"
    status = pkv.device_status(reset=True)
    assert status & pkv.DEV_TIMEOUT, f"{name}: status word {status:#x}"
    assert status & ~pkv.DEV_TIMEOUT == 0, f"{name}: status word {status:#x}"
    # every row had a chunk that needed a copy: every row is reported NaN
    assert torch.isnan(out).all() and torch.isnan(lse).all(), name

    # the same call without the control, on the same device and data
    out2, lse2 = pkv.paged_decode_attn(q, k, v, bt, lens, w.scale, num_splits=splits)
    torch.cuda.synchronize()
    assert pkv.device_status(reset=True) == 0
    ro, rl = oracle.paged_decode_attn(w.q.numpy(), bits(w.k_pool), bits(w.v_pool),
                                      w.block_tables.numpy(), w.seq_lens.numpy(), w.scale)
    assert_attention_close(out2.cpu().numpy(), lse2.cpu().numpy(), ro, rl, f"{name} after")


def test_e4m3_large_group_wait_that_runs_out(pkv):
    """The same over an FP8 cache on the large-group kernel's E4M3 mode,
    whose converter warps wait for codes that never land: the converters,
    the MMA issuer and the softmax all leave with nothing in flight."""
    w = workloads.e4m3(workloads.custom(26, [900, 200], 128, 1, 576, 512, 64))
    dev = "cuda"
    q, k, v = w.q.to(dev), w.k_codes.to(dev), w.v_codes.to(dev)
    ks, vs = w.k_scale.to(dev), w.v_scale.to(dev)
    bt, lens = w.block_tables.to(dev), w.seq_lens.to(dev)
    assert pkv.device_status(reset=True) == 0
    assert pkv.lib.pkv_test_enable_withhold(1) == 0
    try:
        t0 = time.perf_counter()
        out, lse = pkv.paged_decode_attn_e4m3(q, k, v, ks, vs, bt, lens, w.scale, num_splits=2,
                                              flags=pkv.DECODE_TEST_WITHHOLD)
        torch.cuda.synchronize()
        elapsed = time.perf_counter() - t0
        # a GQA shape over an FP8 cache runs another kernel: refused
        g = workloads.e4m3(workloads.custom(27, [300, 40], 32, 8, 128, 128, 16))
        with pytest.raises(pkv.PkvError):
            pkv.paged_decode_attn_e4m3(g.q.to(dev), g.k_codes.to(dev), g.v_codes.to(dev),
                                       g.k_scale.to(dev), g.v_scale.to(dev),
                                       g.block_tables.to(dev), g.seq_lens.to(dev), g.scale,
                                       num_splits=2, flags=pkv.DECODE_TEST_WITHHOLD)
    finally:
        pkv.lib.pkv_test_enable_withhold(0)
    assert elapsed < 10.0, f"the call took {elapsed:.1f} s"
    status = pkv.device_status(reset=True)
    assert status == pkv.DEV_TIMEOUT, f"status word {status:#x}"
    assert torch.isnan(out).all() and torch.isnan(lse).all()
    out2, lse2 = pkv.paged_decode_attn_e4m3(q, k, v, ks, vs, bt, lens, w.scale, num_splits=2)
    torch.cuda.synchronize()
    assert pkv.device_status(reset=True) == 0
    ro, rl = oracle.paged_decode_attn_e4m3(w.q.numpy(), w.k_codes.numpy(), w.v_codes.numpy(),
                                           w.k_scale.numpy(), w.v_scale.numpy(),
                                           w.block_tables.numpy(), w.seq_lens.numpy(), w.scale)
    assert_attention_close(out2.cpu().numpy(), lse2.cpu().numpy(), ro, rl, "e4m3 after")


def test_partials_of_abandoned_chunks_are_nan(pkv):
    """pkv_paged_decode_attn_partial under the control: every non-empty chunk
    is NaN; a chunk with no token still gives the empty result (it waits on
    nothing)."""
    w = workloads.custom(24, [600, 64], 32, 8, 128, 128, 16)
    q, k, v, bt, lens = _inputs(w)
    S = 4
    op = torch.zeros(S, w.batch, w.num_q_heads, w.head_dim_v, device="cuda")
    lp = torch.zeros(S, w.batch, w.num_q_heads, device="cuda")
    assert pkv.lib.pkv_test_enable_withhold(1) == 0
    try:
        pkv.paged_decode_attn_partial(q, k, v, bt, lens, w.scale, S, out_part=op, lse_part=lp,
                                      flags=pkv.DECODE_TEST_WITHHOLD)
        torch.cuda.synchronize()
    finally:
        pkv.lib.pkv_test_enable_withhold(0)
    assert pkv.device_status(reset=True) & pkv.DEV_TIMEOUT
    lp = lp.cpu().numpy()
    for b, L in enumerate(w.seq_lens.tolist()):
        chunk = 64 * -(-L // (64 * S))
        for s in range(S):
            if s * chunk < L:
                assert np.isnan(lp[s, b]).all(), (b, s)
            else:
                assert np.isneginf(lp[s, b]).all(), (b, s)


def test_control_refused_for_kernels_that_do_not_read_it(pkv):
    """A shape that runs on another kernel (here the tcgen05 GQA kernel, 16
    rows per KV head) is refused before anything is launched."""
    w = workloads.custom(25, [300, 40], 64, 4, 128, 128, 16)
    q, k, v, bt, lens = _inputs(w)
    assert pkv.lib.pkv_test_enable_withhold(1) == 0
    try:
        with pytest.raises(pkv.PkvError):
            pkv.paged_decode_attn(q, k, v, bt, lens, w.scale, num_splits=2,
                                  flags=pkv.DECODE_TEST_WITHHOLD)
    finally:
        pkv.lib.pkv_test_enable_withhold(0)
    assert pkv.device_status(reset=True) == 0
