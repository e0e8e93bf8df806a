"""The scratch-free decode entry point, pkv_paged_decode_attn_noalloc.

Some embedders hand the library their inputs and outputs but cannot give it
a workspace: their host framework owns all device memory and lets no other
component call cudaMalloc, or their decode loop must never allocate.  For
them the library keeps the split partials in a fixed scratch array compiled
into it.  This file checks, through the C ABI, that two calls in a row give
the same results as the regular entry point (with a caller workspace), and
that a request larger than the scratch is refused.  It is collected last so
that a run stopping at the first failure has run every other test first, and
it is self-contained so it also passes alone in a fresh process.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

import workloads
from tests._steps import assert_attention_close, auto_splits
from tests._util import bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    import __graft_entry__
    __graft_entry__.build()
    import paged_kv_cache_93_gb300 as m
    m.device_status(reset=True)
    return m


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _call(pkv, name, w, dev, splits, workspace=None):
    """One decode-attention call through the C ABI; returns (out, lse)."""
    k, v = w.k_pool.to(dev), w.v_pool.to(dev)
    bt, lens, q = w.block_tables.to(dev), w.seq_lens.to(dev), w.q.to(dev)
    desc = pkv.cache_desc(k, v)
    B, Hq = w.batch, w.num_q_heads
    out = torch.full((B, Hq, w.head_dim_v), float("nan"), device=dev)
    lse = torch.full((B, Hq), float("nan"), device=dev)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    common = (ctypes.byref(desc), _ptr(q), B, Hq, _ptr(k), _ptr(v), _ptr(bt), bt.shape[1],
              _ptr(lens), ctypes.c_float(w.scale), splits)
    if name == "noalloc":
        rc = pkv.lib.pkv_paged_decode_attn_noalloc(*common, _ptr(out), _ptr(lse), 0, stream)
    else:
        nbytes = 0 if workspace is None else workspace.numel()
        rc = pkv.lib.pkv_paged_decode_attn(*common, _ptr(workspace), nbytes, _ptr(out),
                                           _ptr(lse), 0, stream)
    torch.cuda.synchronize()
    assert rc == 0, f"{name}: status {rc}"
    return out.cpu().numpy(), lse.cpu().numpy()


def _workspace_for(pkv, w, splits):
    if splits == 0:
        splits = auto_splits(pkv, w)
    need = pkv.decode_workspace_size(w.batch, w.num_q_heads, w.head_dim_v, splits)
    return torch.empty(max(need, 16), dtype=torch.uint8, device="cuda")


def test_noalloc_matches_workspace_entry_point_twice(pkv):
    """The same kernels run on the same inputs, so the scratch-free call must
    give the regular call's bits exactly; the partials only live elsewhere."""
    import oracle
    dev = "cuda"
    cases = [(workloads.long32k(batch=2, context=8192), 16),
             (workloads.mix(), 3),                   # a different shape on the second call
             (workloads.long32k(batch=2, context=8192), 0)]   # the split count chosen inside
    for w, splits in cases:
        ref_o, ref_l = _call(pkv, "workspace", w, dev, splits, _workspace_for(pkv, w, splits))
        got_o, got_l = _call(pkv, "noalloc", w, dev, splits)
        assert np.isfinite(got_o).all()
        assert np.array_equal(got_o, ref_o) and np.array_equal(got_l, ref_l), w.name
    # the num_splits = 0 call against the oracle as well
    ro, rl = oracle.paged_decode_attn(w.q.numpy(), bits(w.k_pool), bits(w.v_pool),
                                      w.block_tables.numpy(), w.seq_lens.numpy(), w.scale)
    assert_attention_close(got_o, got_l, ro, rl, "noalloc, num_splits = 0")
    assert pkv.device_status() == 0


def test_noalloc_refuses_partials_beyond_the_scratch(pkv):
    w = workloads.custom(3, [40] * 64, 64, 8, 128, 128, 16)
    # 64 sequences x 64 heads x 129 floats x 256 splits is far beyond 8 MiB
    k, v = w.k_pool.cuda(), w.v_pool.cuda()
    desc = pkv.cache_desc(k, v)
    out = torch.empty(64, 64, 128, device="cuda")
    lse = torch.empty(64, 64, device="cuda")
    rc = pkv.lib.pkv_paged_decode_attn_noalloc(
        ctypes.byref(desc), _ptr(w.q.cuda()), 64, 64, _ptr(k), _ptr(v),
        _ptr(w.block_tables.cuda()), w.block_tables.shape[1], _ptr(w.seq_lens.cuda()),
        ctypes.c_float(w.scale), 256, _ptr(out), _ptr(lse), 0,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == -4        # PKV_ERR_WORKSPACE_TOO_SMALL


def test_noalloc_e4m3_matches_workspace_call_and_oracle(pkv):
    """The FP8 form: the same bits as pkv_paged_decode_attn_e4m3 with a caller
    workspace, and the oracle's attention over the stored codes."""
    import oracle
    dev = "cuda"
    w = workloads.e4m3(workloads.custom(12, [3000, 700, 45], 32, 8, 128, 128, 16))
    kc, vc = w.k_codes.to(dev), w.v_codes.to(dev)
    ks, vs = w.k_scale.to(dev), w.v_scale.to(dev)
    bt, lens, q = w.block_tables.to(dev), w.seq_lens.to(dev), w.q.to(dev)
    desc = pkv.cache_desc(kc, vc)
    B, Hq = w.batch, w.num_q_heads
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    ro, rl = oracle.paged_decode_attn_e4m3(w.q.numpy(), w.k_codes.numpy(), w.v_codes.numpy(),
                                           w.k_scale.numpy(), w.v_scale.numpy(),
                                           w.block_tables.numpy(), w.seq_lens.numpy(), w.scale)
    # 5 splits twice in a row, then the split count chosen inside (num_splits = 0)
    for splits in (5, 5, 0):
        ref_o, ref_l = pkv.paged_decode_attn_e4m3(q, kc, vc, ks, vs, bt, lens, w.scale,
                                                  num_splits=splits)
        out = torch.full((B, Hq, w.head_dim_v), float("nan"), device=dev)
        lse = torch.full((B, Hq), float("nan"), device=dev)
        rc = pkv.lib.pkv_paged_decode_attn_noalloc_e4m3(
            ctypes.byref(desc), _ptr(q), B, Hq, _ptr(kc), _ptr(vc), _ptr(ks), _ptr(vs), _ptr(bt),
            bt.shape[1], _ptr(lens), ctypes.c_float(w.scale), splits, _ptr(out), _ptr(lse), 0,
            stream)
        torch.cuda.synchronize()
        assert rc == 0
        assert torch.equal(out, ref_o) and torch.equal(lse, ref_l), f"splits {splits}"
        assert_attention_close(out.cpu().numpy(), lse.cpu().numpy(), ro, rl,
                               f"noalloc e4m3, num_splits = {splits}")
    assert pkv.device_status() == 0


def test_noalloc_checks_arguments_before_the_scratch_limit(pkv):
    """A request the regular entry point rejects gets the same status from
    the scratch-free one, even when it would also exceed the scratch."""
    w = workloads.custom(3, [40] * 64, 64, 8, 128, 128, 16)
    k, v = w.k_pool.cuda(), w.v_pool.cuda()
    desc = pkv.cache_desc(k, v)
    out = torch.empty(64, 64, 128, device="cuda")
    lse = torch.empty(64, 64, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    args = (ctypes.byref(desc), _ptr(w.q.cuda()), 64, 64, _ptr(k), _ptr(v),
            _ptr(w.block_tables.cuda()), w.block_tables.shape[1], _ptr(w.seq_lens.cuda()),
            ctypes.c_float(w.scale))
    for splits, flags in ((300, 0), (256, 0x40)):     # too many splits; an unknown flag
        rc_reg = pkv.lib.pkv_paged_decode_attn(*args, splits, None, 0, _ptr(out), _ptr(lse),
                                               flags, stream)
        rc_na = pkv.lib.pkv_paged_decode_attn_noalloc(*args, splits, _ptr(out), _ptr(lse), flags,
                                                      stream)
        assert rc_reg == rc_na == -1                    # PKV_ERR_INVALID_ARG
