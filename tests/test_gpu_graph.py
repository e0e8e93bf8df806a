"""A whole decode step -- slot mapping, append, split attention and merge --
captured once in a CUDA graph and replayed: the library's calls allocate
nothing, never synchronise with the host and launch with programmatic
dependencies, so they capture as they are.  Replays on fresh inputs must give
the same bits as the same calls made eagerly."""
from __future__ import annotations

import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    import __graft_entry__
    __graft_entry__.build()
    import paged_kv_cache_93_gb300 as m
    m.device_status(reset=True)
    return m


class StepBuffers:
    """Static device buffers of one step (a graph replays fixed addresses)."""

    def __init__(self, pkv, w, splits):
        dev = "cuda"
        self.pkv, self.w, self.splits = pkv, w, splits
        self.k, self.v = w.k_pool.to(dev), w.v_pool.to(dev)
        self.bt, self.lens = w.block_tables.to(dev), w.seq_lens.to(dev)
        self.q = w.q.to(dev)
        self.seq, self.pos = w.new_seq.to(dev), w.new_pos.to(dev)
        self.k_new, self.v_new = w.k_new.to(dev), w.v_new.to(dev)
        B, Hq, Dv = w.batch, w.num_q_heads, w.head_dim_v
        self.slots = torch.empty(self.pos.numel(), dtype=torch.int64, device=dev)
        self.out = torch.empty(B, Hq, Dv, device=dev)
        self.lse = torch.empty(B, Hq, device=dev)
        self.ws = torch.empty(max(1, pkv.decode_workspace_size(B, Hq, Dv, splits)),
                              dtype=torch.uint8, device=dev)

    def step(self):
        p = self.pkv
        p.slot_mapping(self.k, self.v, self.bt, self.seq, self.pos, out=self.slots)
        p.kv_append(self.k, self.v, self.k_new, self.v_new, self.slots)
        p.paged_decode_attn(self.q, self.k, self.v, self.bt, self.lens, self.w.scale,
                            num_splits=self.splits, workspace=self.ws, out=self.out,
                            lse=self.lse)


@pytest.mark.parametrize("name,splits", [("mix", 1), ("mix", 3), ("tiny", 2),
                                         ("long32k_small", 16)])
def test_step_replays_in_a_cuda_graph(pkv, name, splits):
    mk = (lambda: workloads.long32k(batch=2, context=4096)) \
        if name == "long32k_small" else (lambda: workloads.make(name))
    w0, w1 = mk(), mk()
    # the same tables and lengths (a replay reuses them), fresh values
    g = torch.Generator().manual_seed(12)
    for f in ("k_pool", "v_pool", "q", "k_new", "v_new"):
        t = getattr(w1, f)
        setattr(w1, f, torch.randn(t.shape, generator=g).to(t.dtype))
    g_buf = StepBuffers(pkv, w0, splits)
    g_buf.step()                        # warm-up: one-time per-device setup happens here
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        g_buf.step()
    # new inputs into the captured buffers, then replay
    for dst, src in [(g_buf.k, w1.k_pool), (g_buf.v, w1.v_pool), (g_buf.q, w1.q),
                     (g_buf.k_new, w1.k_new), (g_buf.v_new, w1.v_new)]:
        dst.copy_(src)
    graph.replay()
    torch.cuda.synchronize()
    # the same calls made eagerly on the same inputs
    e_buf = StepBuffers(pkv, w1, splits)
    e_buf.step()
    torch.cuda.synchronize()
    assert torch.equal(g_buf.out, e_buf.out) and torch.equal(g_buf.lse, e_buf.lse)
    assert torch.equal(g_buf.k, e_buf.k) and torch.equal(g_buf.v, e_buf.v)
    # a second replay after the append is idempotent for the same inputs
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(g_buf.out, e_buf.out)
    assert pkv.device_status() == 0
