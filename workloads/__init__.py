"""Seeded synthetic inputs shared by the GPU library's tests and benchmark and
by the CPU oracle.

This module only draws random numbers and lays out which physical block holds
which logical block; it holds none of the attention, merge, append, slot or
partition arithmetic.  Values are fp32 N(0, 1) from a seeded CPU
``torch.Generator``; K/V values are rounded to bf16 (round-to-nearest-even by
``Tensor.to``) so both sides consume identical bits.

The five workloads are synthetic stand-ins for those the pages discuss:

1. ``tiny``      -- the block-accounting example of "PagedAttentionとは？" ("要求の終了で
                    空いたブロックを再利用する具体例": block size 4, requests of 6 and 9
                    tokens) with 4 query / 2 KV heads, head_dim 64, 8 shuffled blocks.
2. ``mix``       -- continuous batching mix of "1,000 人が同時に AI に質問したら…"
                    ("ラボで測ったこと": prompts 8-32, answers 16-96): 16 sequences with
                    context U{24..128}, GQA 32/8, head_dim 128, block size 16, 256 blocks.
3. ``long32k``   -- long-context GQA decode: batch 8 x 32,768 tokens, 32/8 heads,
                    head_dim 128, block size 16, a random permutation of 16,384 blocks.
4. ``dcp200k``   -- the DCP example of "なぜ長文LLMは遅くなるのか" (200,000 tokens over
                    DCP size 4): batch 1, 64/8 heads, head_dim 128, block size 16.
5. ``agent_mla`` -- agent traffic of "vLLM AgentX リリース" ("エージェントワークロードの
                    特性": long shared prefixes): 32 sequences sharing a 136,040-token
                    prefix, suffixes U{2000..10000}, 128 query heads over 1 latent KV
                    head, K dim 576, V dim 512, block size 64.

Every workload describes one decode step: the cache before the step
(``k_pool``/``v_pool`` + ``block_tables``), the copy-on-write pairs the step
performs first (``cow_src``/``cow_dst``, possibly empty), the tokens it
appends (``new_seq``/``new_pos``/``k_new``/``v_new``; the last appended token
of each sequence is its decode token), and the query of the new token.
``seq_lens`` is the context each sequence attends over after the appends.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

__all__ = ["Workload", "make", "NAMES", "tiny", "mix", "long32k", "dcp200k", "agent_mla",
           "custom", "random_partials", "e4m3"]

NAMES = ("tiny", "mix", "long32k", "dcp200k", "agent_mla")


@dataclass
class Workload:
    name: str
    num_q_heads: int
    num_kv_heads: int
    head_dim_k: int
    head_dim_v: int
    block_size: int
    q: torch.Tensor                 # [B, Hq, Dk] fp32
    k_pool: torch.Tensor            # [num_blocks, Hkv, bs, Dk] bf16, cache before the step
    v_pool: torch.Tensor | None     # [num_blocks, Hkv, bs, Dv] bf16; None: values inside K
    block_tables: torch.Tensor      # [B, max_blocks] int32, -1 past the last used block
    seq_lens: torch.Tensor          # [B] int32, tokens attended after the appends
    scale: float
    new_seq: torch.Tensor           # [T] int32, sequence of each appended token
    new_pos: torch.Tensor           # [T] int64, logical position of each appended token
    k_new: torch.Tensor             # [T, Hkv, Dk] bf16
    v_new: torch.Tensor | None      # [T, Hkv, Dv] bf16; None: values inside K
    cow_src: torch.Tensor = field(default_factory=lambda: torch.empty(0, dtype=torch.int32))
    cow_dst: torch.Tensor = field(default_factory=lambda: torch.empty(0, dtype=torch.int32))
    # DCP-style interleaved partitions (dcp200k only): the partition count and
    # interleave size, the table each partition's local KV uses, and the
    # logical K/V of every token of the (single) sequence in token order.
    num_parts: int = 0
    interleave: int = 0
    part_tables: torch.Tensor | None = None      # [P, max_part_blocks] int32
    k_tokens: torch.Tensor | None = None         # [N, Hkv, Dk] bf16
    v_tokens: torch.Tensor | None = None         # [N, Hkv, Dv] bf16
    info: dict = field(default_factory=dict)
    # Multi-token steps: q is [B, tokens_per_seq, Hq, Dk] and the last
    # tokens_per_seq tokens of each sequence are the step's new ones.
    tokens_per_seq: int = 1
    # FP8 cache (see e4m3()): uint8 code pools before the step and fp32
    # dequantisation scales per KV head.
    k_codes: torch.Tensor | None = None
    v_codes: torch.Tensor | None = None
    k_scale: torch.Tensor | None = None
    v_scale: torch.Tensor | None = None

    @property
    def batch(self) -> int:
        return int(self.q.shape[0])

    @property
    def num_blocks(self) -> int:
        return int(self.k_pool.shape[0])

    @property
    def max_blocks(self) -> int:
        return int(self.block_tables.shape[1])


def _normal(g: torch.Generator, shape, dtype=torch.float32) -> torch.Tensor:
    return torch.randn(*shape, generator=g, dtype=torch.float32).to(dtype)


def _tables(perm: torch.Tensor, counts: list[int], width: int) -> torch.Tensor:
    """Hand out physical blocks from `perm` in order: sequence b receives the
    next counts[b] entries as its logical blocks 0..counts[b]-1."""
    t = torch.full((len(counts), width), -1, dtype=torch.int32)
    at = 0
    for b, c in enumerate(counts):
        t[b, :c] = perm[at:at + c].to(torch.int32)
        at += c
    return t


def _ceil_div(a: int, b: int) -> int:
    return -(-a // b)


def _decode_tokens(g, cached: list[int], hkv: int, dk: int, dv: int):
    """One appended decode token per sequence, at position cached[b]."""
    B = len(cached)
    new_seq = torch.arange(B, dtype=torch.int32)
    new_pos = torch.tensor(cached, dtype=torch.int64)
    k_new = _normal(g, (B, hkv, dk), torch.bfloat16)
    v_new = _normal(g, (B, hkv, dv), torch.bfloat16)
    return new_seq, new_pos, k_new, v_new


def _gqa(name, seed, cached, hq, hkv, d, bs, num_blocks, table_width=None):
    g = torch.Generator().manual_seed(seed)
    B = len(cached)
    lens = [c + 1 for c in cached]
    counts = [_ceil_div(n, bs) for n in lens]
    width = table_width or max(counts)
    assert sum(counts) <= num_blocks
    perm = torch.randperm(num_blocks, generator=g)
    tables = _tables(perm, counts, width)
    k_pool = _normal(g, (num_blocks, hkv, bs, d), torch.bfloat16)
    v_pool = _normal(g, (num_blocks, hkv, bs, d), torch.bfloat16)
    q = _normal(g, (B, hq, d))
    new_seq, new_pos, k_new, v_new = _decode_tokens(g, cached, hkv, d, d)
    return Workload(name, hq, hkv, d, d, bs, q, k_pool, v_pool, tables,
                    torch.tensor(lens, dtype=torch.int32), 1.0 / math.sqrt(d),
                    new_seq, new_pos, k_new, v_new)


def tiny(seed: int = 1) -> Workload:
    """Two sequences holding 6 and 9 tokens, block size 4, 8 shuffled blocks."""
    return _gqa("tiny", seed, [6, 9], hq=4, hkv=2, d=64, bs=4, num_blocks=8)


def mix(seed: int = 2) -> Workload:
    """16 sequences, cached context U{24..128}, one decode token each."""
    g = torch.Generator().manual_seed(seed)
    cached = torch.randint(24, 129, (16,), generator=g).tolist()
    return _gqa("mix", seed + 1000, cached, hq=32, hkv=8, d=128, bs=16, num_blocks=256)


def long32k(seed: int = 3, batch: int = 8, context: int = 32768) -> Workload:
    """batch x `context` tokens (the decode token included), every block used."""
    bs = 16
    num_blocks = batch * context // bs
    return _gqa("long32k", seed, [context - 1] * batch, hq=32, hkv=8, d=128, bs=bs,
                num_blocks=num_blocks)


def spec_verify(seed: int = 6, batch: int = 8, context: int = 32768, tokens: int = 4,
                hq: int = 32, hkv: int = 8, d: int = 128, bs: int = 16,
                name: str = "spec4_32k") -> Workload:
    """Speculative verification: batch x `context` tokens, the last `tokens`
    of each sequence appended in the step; each new token queries the cache
    causally (query t sees the context up to and including new token t).
    Every block of the pool is used when context is a multiple of bs."""
    g = torch.Generator().manual_seed(seed)
    counts = [_ceil_div(context, bs)] * batch
    num_blocks = sum(counts)
    perm = torch.randperm(num_blocks, generator=g)
    tables = _tables(perm, counts, max(counts))
    k_pool = _normal(g, (num_blocks, hkv, bs, d), torch.bfloat16)
    v_pool = _normal(g, (num_blocks, hkv, bs, d), torch.bfloat16)
    q = _normal(g, (batch, tokens, hq, d))
    new_seq = torch.arange(batch, dtype=torch.int32).repeat_interleave(tokens)
    new_pos = (context - tokens + torch.arange(tokens, dtype=torch.int64)).repeat(batch)
    k_new = _normal(g, (batch * tokens, hkv, d), torch.bfloat16)
    v_new = _normal(g, (batch * tokens, hkv, d), torch.bfloat16)
    w = Workload(name, hq, hkv, d, d, bs, q, k_pool, v_pool, tables,
                 torch.full((batch,), context, dtype=torch.int32), 1.0 / math.sqrt(d),
                 new_seq, new_pos, k_new, v_new)
    w.tokens_per_seq = tokens
    return w


def dcp200k(seed: int = 4, context: int = 200_000, num_parts: int = 4,
            interleave: int = 1) -> Workload:
    """One 200,000-token sequence (the decode token is the last) with the
    logical K/V of every token, an unsplit table and one table per partition
    over disjoint blocks of one shared, permuted pool."""
    g = torch.Generator().manual_seed(seed)
    hq, hkv, d, bs = 64, 8, 128, 16
    unsplit_blocks = _ceil_div(context, bs)
    # Capacity only: no partition can hold more than context / P + interleave
    # tokens, so every partition gets a table of that many tokens' blocks.
    part_capacity = _ceil_div(_ceil_div(context, num_parts) + interleave, bs)
    num_blocks = unsplit_blocks + num_parts * part_capacity
    perm = torch.randperm(num_blocks, generator=g)
    table = _tables(perm[:unsplit_blocks], [unsplit_blocks], unsplit_blocks)
    part_tables = _tables(perm[unsplit_blocks:], [part_capacity] * num_parts, part_capacity)
    k_tokens = _normal(g, (context, hkv, d), torch.bfloat16)
    v_tokens = _normal(g, (context, hkv, d), torch.bfloat16)
    k_pool = _normal(g, (num_blocks, hkv, bs, d), torch.bfloat16)
    v_pool = _normal(g, (num_blocks, hkv, bs, d), torch.bfloat16)
    q = _normal(g, (1, hq, d))
    # The decode token is appended by the step; the others are cached before it.
    new_seq = torch.zeros(1, dtype=torch.int32)
    new_pos = torch.tensor([context - 1], dtype=torch.int64)
    w = Workload("dcp200k", hq, hkv, d, d, bs, q, k_pool, v_pool, table,
                 torch.tensor([context], dtype=torch.int32), 1.0 / math.sqrt(d),
                 new_seq, new_pos, k_tokens[context - 1:].clone(), v_tokens[context - 1:].clone())
    w.num_parts, w.interleave = num_parts, interleave
    w.part_tables, w.k_tokens, w.v_tokens = part_tables, k_tokens, v_tokens
    return w


def agent_mla(seed: int = 5, num_seqs: int = 32, prefix: int = 136_040,
              suffix_range=(2000, 10000), latent: bool = False) -> Workload:
    """Shared-prefix MLA-shaped decode.  The prefix fills 2,125 blocks of 64
    tokens plus a shared tail block holding prefix % 64 tokens; every sequence
    first copies the tail into a private block (copy-on-write), then appends its
    suffix and its decode token, and attends over prefix + suffix + 1 tokens.
    latent: the cache keeps no value pool (v_pool and v_new are None); a
    token's value is the first 512 dims of its 576-dim key row."""
    g = torch.Generator().manual_seed(seed)
    hq, hkv, dk, dv, bs = 128, 1, 576, 512, 64
    suffix = torch.randint(suffix_range[0], suffix_range[1] + 1, (num_seqs,), generator=g).tolist()
    full, tail_fill = divmod(prefix, bs)
    lens = [prefix + s + 1 for s in suffix]
    counts = [_ceil_div(n, bs) for n in lens]
    shared = full + (1 if tail_fill else 0)
    private = [c - full for c in counts]          # private tail copy + suffix blocks
    num_blocks = shared + sum(private)
    perm = torch.randperm(num_blocks, generator=g)
    width = max(counts)
    tables = torch.full((num_seqs, width), -1, dtype=torch.int32)
    tables[:, :full] = perm[:full].to(torch.int32)
    shared_tail = int(perm[full]) if tail_fill else -1
    at = shared
    for b in range(num_seqs):
        tables[b, full:counts[b]] = perm[at:at + private[b]].to(torch.int32)
        at += private[b]
    if tail_fill:
        cow_src = torch.full((num_seqs,), shared_tail, dtype=torch.int32)
        cow_dst = tables[:, full].clone()
    else:
        cow_src = torch.empty(0, dtype=torch.int32)
        cow_dst = torch.empty(0, dtype=torch.int32)
    k_pool = _normal(g, (num_blocks, hkv, bs, dk), torch.bfloat16)
    v_pool = None if latent else _normal(g, (num_blocks, hkv, bs, dv), torch.bfloat16)
    q = _normal(g, (num_seqs, hq, dk))
    seq_ids, positions = [], []
    for b in range(num_seqs):
        n = suffix[b] + 1
        seq_ids.append(torch.full((n,), b, dtype=torch.int32))
        positions.append(torch.arange(prefix, prefix + n, dtype=torch.int64))
    new_seq = torch.cat(seq_ids)
    new_pos = torch.cat(positions)
    T = int(new_seq.numel())
    k_new = _normal(g, (T, hkv, dk), torch.bfloat16)
    v_new = None if latent else _normal(g, (T, hkv, dv), torch.bfloat16)
    w = Workload("agent_mla_latent" if latent else "agent_mla", hq, hkv, dk, dv, bs, q, k_pool,
                 v_pool, tables,
                 torch.tensor(lens, dtype=torch.int32), 1.0 / math.sqrt(dk),
                 new_seq, new_pos, k_new, v_new, cow_src, cow_dst)
    w.info = {"prefix": prefix, "suffix": suffix, "shared_blocks": shared,
              "shared_tail": shared_tail}
    return w


def custom(seed: int, cached: list[int], hq: int, hkv: int, dk: int, dv: int, bs: int,
           extra_blocks: int = 3, name: str = "custom") -> Workload:
    """Any GQA/MLA shape: sequences holding `cached` tokens, one decode token
    each, blocks drawn from a shuffled pool with `extra_blocks` spare."""
    g = torch.Generator().manual_seed(seed)
    B = len(cached)
    lens = [c + 1 for c in cached]
    counts = [_ceil_div(n, bs) for n in lens]
    num_blocks = sum(counts) + extra_blocks
    perm = torch.randperm(num_blocks, generator=g)
    tables = _tables(perm, counts, max(counts))
    k_pool = _normal(g, (num_blocks, hkv, bs, dk), torch.bfloat16)
    v_pool = _normal(g, (num_blocks, hkv, bs, dv), torch.bfloat16)
    q = _normal(g, (B, hq, dk))
    new_seq, new_pos, k_new, v_new = _decode_tokens(g, cached, hkv, dk, dv)
    return Workload(name, hq, hkv, dk, dv, bs, q, k_pool, v_pool, tables,
                    torch.tensor(lens, dtype=torch.int32), 1.0 / math.sqrt(dk),
                    new_seq, new_pos, k_new, v_new)


def shared_prefix(seed: int, prefix_blocks: int, suffix_cached: list[int], hq: int, hkv: int,
                  dk: int, dv: int, bs: int, latent: bool = False) -> Workload:
    """Sequences whose first `prefix_blocks` table entries are the same
    physical blocks, each followed by its own blocks: sequence b holds
    prefix_blocks * bs + suffix_cached[b] tokens, then one decode token.
    info["prefix_table"] holds the shared blocks.  latent: no value pool."""
    g = torch.Generator().manual_seed(seed)
    B = len(suffix_cached)
    P = prefix_blocks * bs
    lens = [P + c + 1 for c in suffix_cached]
    own = [_ceil_div(n, bs) - prefix_blocks for n in lens]
    num_blocks = prefix_blocks + sum(own) + 2
    perm = torch.randperm(num_blocks, generator=g)
    width = prefix_blocks + max(own)
    tables = torch.full((B, width), -1, dtype=torch.int32)
    tables[:, :prefix_blocks] = perm[:prefix_blocks].to(torch.int32)
    at = prefix_blocks
    for b in range(B):
        tables[b, prefix_blocks:prefix_blocks + own[b]] = perm[at:at + own[b]].to(torch.int32)
        at += own[b]
    k_pool = _normal(g, (num_blocks, hkv, bs, dk), torch.bfloat16)
    v_pool = None if latent else _normal(g, (num_blocks, hkv, bs, dv), torch.bfloat16)
    q = _normal(g, (B, hq, dk))
    new_seq, new_pos, k_new, v_new = _decode_tokens(g, [P + c for c in suffix_cached], hkv,
                                                    dk, dv)
    if latent:
        v_new = None
    w = Workload("shared_prefix", hq, hkv, dk, dv, bs, q, k_pool, v_pool, tables,
                 torch.tensor(lens, dtype=torch.int32), 1.0 / math.sqrt(dk),
                 new_seq, new_pos, k_new, v_new)
    w.info = {"prefix_table": tables[0, :prefix_blocks].clone()}
    return w


def e4m3(w: Workload, seed: int = 11) -> Workload:
    """The same step over an FP8 (E4M3) cache.  Each KV head gets scales near
    8/448 (so an 8-sigma value is the largest code); the cache before the
    step holds torch's float8_e4m3fn cast of the bf16 pools divided by their
    head's scale, clipped to +-448 -- a stand-in for a cache filled by
    earlier appends.  The step's new tokens stay bf16 (the append quantises
    them).  Needs a separate value pool.  A step with copy-on-write pairs
    copies the blocks' codes."""
    assert w.v_pool is not None
    g = torch.Generator().manual_seed(seed)
    hkv = w.num_kv_heads
    ks = (8.0 / 448.0) * (1.0 + 0.5 * torch.rand(hkv, generator=g))
    vs = (8.0 / 448.0) * (1.0 + 0.5 * torch.rand(hkv, generator=g))

    def codes(pool, s):
        x = pool.float().div_(s.view(1, -1, 1, 1)).clamp_(-448.0, 448.0)
        return x.to(torch.float8_e4m3fn).view(torch.uint8)

    w.k_codes, w.v_codes = codes(w.k_pool, ks), codes(w.v_pool, vs)
    w.k_scale, w.v_scale = ks.float(), vs.float()
    w.name = w.name + "_e4m3"
    return w


def make(name: str, **kw) -> Workload:
    if name == "long32k_e4m3":
        return e4m3(long32k(**kw))
    if name == "spec4_32k_e4m3":
        return e4m3(spec_verify(**kw))
    if name == "dcp200k_e4m3":
        return e4m3(dcp200k(**kw))
    if name == "agent_mla_e4m3":
        return e4m3(agent_mla(**kw))
    if name == "agent_mla_latent":
        return agent_mla(latent=True, **kw)
    if name == "agent_mla_cascade":
        return agent_mla(**kw)
    if name == "spec4_32k":
        return spec_verify(**kw)
    return {"tiny": tiny, "mix": mix, "long32k": long32k, "dcp200k": dcp200k,
            "agent_mla": agent_mla}[name](**kw)


def random_partials(seed: int, num_parts: int, batch: int, heads: int, dv: int,
                    empty_fraction: float = 0.0):
    """Seeded partial outputs [P, B, H, Dv] and LSEs [P, B, H] (fp32) for the
    merge; a fraction of the partials is marked empty (lse = -inf, out = 0)."""
    g = torch.Generator().manual_seed(seed)
    out = _normal(g, (num_parts, batch, heads, dv))
    lse = _normal(g, (num_parts, batch, heads)) * 4.0 + 10.0
    if empty_fraction > 0:
        empty = torch.rand(num_parts, batch, heads, generator=g) < empty_fraction
        lse[empty] = float("-inf")
        out[empty] = 0.0
    return out, lse
