"""paged_kv_cache_93_gb300 -- paged KV-cache decode attention on GB300.

A thin binding over libpkv.so (include/pkv.h).  Every function here only
marshals torch tensors (device pointers, shapes, the current CUDA stream)
into one C call; all arithmetic runs in the library's CUDA kernels.  Outputs
that the caller does not pass are allocated with torch.

Layouts (one layer): k_pool [num_blocks, Hkv, block_size, Dk] bf16,
v_pool [num_blocks, Hkv, block_size, Dv] bf16, block_tables [B, max_blocks]
int32, seq_lens [B] int32, q [B, Hq, Dk] fp32, out [B, Hq, Dv] fp32,
lse [B, Hq] fp32 (natural log).  An FP8 cache holds E4M3 codes in uint8
pools of the same shapes, with fp32 dequantisation scales per KV head
(the *_e4m3 functions).
"""
from __future__ import annotations

import ctypes

import torch

from . import _lib
from ._lib import (DECODE_GENERIC, DECODE_NO_TCGEN05, DECODE_TEST_WITHHOLD, DEV_BLOCK_ID,
                   DEV_COPY_CONFLICT, DEV_PREFIX, DEV_SEQ_LEN, DEV_SLOT, DEV_TABLE_RANGE,
                   DEV_TIMEOUT, CacheDesc, PkvError)

__all__ = [
    "CacheDesc", "PkvError", "ValuesInKeys", "cache_desc", "kv_append", "slot_mapping", "copy_blocks",
    "interleave_slot_mapping", "interleave_partition_len", "decode_workspace_size",
    "decode_auto_splits", "paged_decode_attn", "paged_decode_attn_partial",
    "paged_decode_attn_multi", "lse_merge", "kv_append_e4m3", "copy_blocks_e4m3",
    "paged_decode_attn_e4m3", "paged_decode_attn_partial_e4m3", "paged_decode_attn_multi_e4m3",
    "paged_decode_attn_cascade",
    "decode_cascade_splits", "DEV_PREFIX",
    "device_status", "BlockManager", "library_path", "DECODE_GENERIC", "DECODE_NO_TCGEN05",
    "DECODE_TEST_WITHHOLD", "DEV_BLOCK_ID",
    "DEV_SLOT", "DEV_SEQ_LEN", "DEV_COPY_CONFLICT", "DEV_TIMEOUT", "DEV_TABLE_RANGE",
]

lib = _lib.load()
library_path = _lib.LIB_PATH


def _check(where: str, status: int) -> None:
    if status != _lib.PKV_OK:
        raise PkvError(where, status, lib.pkv_status_string(status).decode())


def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _need(t: torch.Tensor, name: str, dtype: torch.dtype, dim: int | None = None):
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dim is not None and t.dim() != dim:
        raise ValueError(f"{name} must have {dim} dims, got {t.dim()}")


class ValuesInKeys:
    """Pass as `v_pool` when the cache keeps no separate value pool: the value
    of a token is the first `head_dim_v` dims of its key row (the latent
    layout of multi-head latent attention).  Marshalled as a NULL v_pool."""

    def __init__(self, head_dim_v: int):
        self.head_dim_v = int(head_dim_v)


def _v_ptr(v_pool):
    return None if isinstance(v_pool, ValuesInKeys) else _ptr(v_pool)


def cache_desc(k_pool: torch.Tensor, v_pool) -> CacheDesc:
    """Shape of a bf16 cache, or of an E4M3 one (uint8 code pools)."""
    dtype = torch.uint8 if k_pool.dtype == torch.uint8 else torch.bfloat16
    _need(k_pool, "k_pool", dtype, 4)
    nb, hkv, bs, dk = k_pool.shape
    if isinstance(v_pool, ValuesInKeys):
        if dtype != torch.bfloat16:
            raise ValueError("values inside the keys need a bf16 cache")
        if not 0 < v_pool.head_dim_v <= dk:
            raise ValueError("values inside the keys need 0 < head_dim_v <= head_dim_k")
        return CacheDesc(nb, bs, hkv, dk, v_pool.head_dim_v)
    _need(v_pool, "v_pool", dtype, 4)
    if tuple(v_pool.shape[:3]) != (nb, hkv, bs):
        raise ValueError("k_pool and v_pool disagree on [num_blocks, Hkv, block_size]")
    return CacheDesc(nb, bs, hkv, dk, v_pool.shape[3])


def _bf16_desc(k_pool: torch.Tensor, v_pool) -> CacheDesc:
    """cache_desc for the calls that take bf16 pools only (the C calls size
    every row from the element count at two bytes an element, so a code pool
    given to them would be read and written past its end)."""
    _need(k_pool, "k_pool", torch.bfloat16, 4)
    return cache_desc(k_pool, v_pool)


def device_status(reset: bool = True, stream=None) -> int:
    """Synchronize `stream` and return the device status word (PKV_DEV_* bits)."""
    flags = ctypes.c_uint32(0)
    _check("pkv_device_status", lib.pkv_device_status(ctypes.byref(flags), int(reset),
                                                      _stream(stream)))
    return int(flags.value)


def slot_mapping(k_pool, v_pool, block_tables, seq_ids, positions, out=None, stream=None):
    """Slots of (sequence, position) pairs through the block tables (int64 [T])."""
    desc = cache_desc(k_pool, v_pool)
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(seq_ids, "seq_ids", torch.int32, 1)
    _need(positions, "positions", torch.int64, 1)
    T = positions.numel()
    if out is None:
        out = torch.empty(T, dtype=torch.int64, device=positions.device)
    _check("pkv_slot_mapping", lib.pkv_slot_mapping(
        ctypes.byref(desc), _ptr(block_tables), block_tables.shape[0], block_tables.shape[1],
        _ptr(seq_ids), _ptr(positions), T, _ptr(out), _stream(stream)))
    return out


def kv_append(k_pool, v_pool, k_new, v_new, slots, stream=None) -> None:
    """Write k_new [T, Hkv, Dk] / v_new [T, Hkv, Dv] (bf16) at slots [T] (int64).
    With v_pool = ValuesInKeys(Dv), v_new must be None (only K is written)."""
    desc = _bf16_desc(k_pool, v_pool)
    _need(k_new, "k_new", torch.bfloat16, 3)
    if isinstance(v_pool, ValuesInKeys):
        if v_new is not None:
            raise ValueError("v_new must be None when the values are inside the keys")
    else:
        _need(v_new, "v_new", torch.bfloat16, 3)
    _need(slots, "slot_mapping", torch.int64, 1)
    _check("pkv_kv_append", lib.pkv_kv_append(
        ctypes.byref(desc), _ptr(k_pool), _v_ptr(v_pool), _ptr(k_new), _ptr(v_new),
        _ptr(slots), slots.numel(), _stream(stream)))


def copy_blocks(k_pool, v_pool, src, dst, stream=None) -> None:
    """Copy-on-write duplication: block src[i] -> block dst[i] (int32 device
    arrays), bf16 pools (copy_blocks_e4m3 for code pools)."""
    desc = _bf16_desc(k_pool, v_pool)
    _need(src, "src", torch.int32, 1)
    _need(dst, "dst", torch.int32, 1)
    if src.numel() != dst.numel():
        raise ValueError("src and dst lengths differ")
    _check("pkv_copy_blocks", lib.pkv_copy_blocks(
        ctypes.byref(desc), _ptr(k_pool), _v_ptr(v_pool), _ptr(src), _ptr(dst), src.numel(),
        _stream(stream)))


def _e4m3_desc(k_pool, v_pool, k_scale, v_scale) -> CacheDesc:
    _need(k_pool, "k_pool", torch.uint8, 4)
    desc = cache_desc(k_pool, v_pool)
    _need(k_scale, "k_scale", torch.float32, 1)
    _need(v_scale, "v_scale", torch.float32, 1)
    if k_scale.numel() != desc.num_kv_heads or v_scale.numel() != desc.num_kv_heads:
        raise ValueError("k_scale and v_scale hold one scale per KV head")
    return desc


def kv_append_e4m3(k_pool, v_pool, k_new, v_new, slots, k_scale, v_scale, stream=None) -> None:
    """Quantise k_new / v_new (bf16 [T, Hkv, D]) into the E4M3 pools at slots
    [T]: element x of KV head g becomes the code nearest to x / scale[g]."""
    desc = _e4m3_desc(k_pool, v_pool, k_scale, v_scale)
    _need(k_new, "k_new", torch.bfloat16, 3)
    _need(v_new, "v_new", torch.bfloat16, 3)
    _need(slots, "slot_mapping", torch.int64, 1)
    _check("pkv_kv_append_e4m3", lib.pkv_kv_append_e4m3(
        ctypes.byref(desc), _ptr(k_pool), _ptr(v_pool), _ptr(k_new), _ptr(v_new),
        _ptr(k_scale), _ptr(v_scale), _ptr(slots), slots.numel(), _stream(stream)))


def copy_blocks_e4m3(k_pool, v_pool, src, dst, stream=None) -> None:
    """copy_blocks for E4M3 pools."""
    _need(k_pool, "k_pool", torch.uint8, 4)
    desc = cache_desc(k_pool, v_pool)
    _need(src, "src", torch.int32, 1)
    _need(dst, "dst", torch.int32, 1)
    if src.numel() != dst.numel():
        raise ValueError("src and dst lengths differ")
    _check("pkv_copy_blocks_e4m3", lib.pkv_copy_blocks_e4m3(
        ctypes.byref(desc), _ptr(k_pool), _ptr(v_pool), _ptr(src), _ptr(dst), src.numel(),
        _stream(stream)))


def interleave_slot_mapping(k_pool, v_pool, first_token: int, num_tokens: int, num_parts: int,
                            interleave: int, part_block_tables, out=None, part_out=None,
                            stream=None):
    """Slots of tokens first_token.. in their DCP partition's table (int64 [T])."""
    desc = cache_desc(k_pool, v_pool)
    _need(part_block_tables, "part_block_tables", torch.int32, 2)
    if out is None:
        out = torch.empty(num_tokens, dtype=torch.int64, device=part_block_tables.device)
    _check("pkv_interleave_slot_mapping", lib.pkv_interleave_slot_mapping(
        ctypes.byref(desc), int(first_token), int(num_tokens), int(num_parts), int(interleave),
        _ptr(part_block_tables), part_block_tables.shape[1], _ptr(out), _ptr(part_out),
        _stream(stream)))
    return out


def interleave_partition_len(num_tokens: int, num_parts: int, interleave: int, part: int) -> int:
    n = lib.pkv_interleave_partition_len(int(num_tokens), int(num_parts), int(interleave),
                                         int(part))
    if n < 0:
        raise ValueError("invalid interleave arguments")
    return int(n)


def decode_workspace_size(batch: int, num_q_heads: int, head_dim_v: int, num_splits: int) -> int:
    return int(lib.pkv_decode_workspace_size(batch, num_q_heads, head_dim_v, num_splits))


def decode_auto_splits(k_pool, v_pool, batch: int, num_q_heads: int, max_seq_len: int) -> int:
    desc = _bf16_desc(k_pool, v_pool)
    return int(lib.pkv_decode_auto_splits(ctypes.byref(desc), batch, num_q_heads, max_seq_len))


def _decode_common(q, k_pool, v_pool, block_tables, seq_lens):
    desc = _bf16_desc(k_pool, v_pool)
    _need(q, "q", torch.float32, 3)
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    return desc


def paged_decode_attn(q, k_pool, v_pool, block_tables, seq_lens, scale: float,
                      num_splits: int = 0, workspace=None, out=None, lse=None, flags: int = 0,
                      stream=None):
    """Decode attention of q [B, Hq, Dk] over the paged cache -> (out, lse)."""
    desc = _decode_common(q, k_pool, v_pool, block_tables, seq_lens)
    B, Hq, _ = q.shape
    if out is None:
        out = torch.empty(B, Hq, desc.head_dim_v, dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty(B, Hq, dtype=torch.float32, device=q.device)
    S = num_splits
    if S == 0:
        S = int(lib.pkv_decode_auto_splits(ctypes.byref(desc), B, Hq,
                                           block_tables.shape[1] * desc.block_size))
    need = decode_workspace_size(B, Hq, desc.head_dim_v, S)
    if need and (workspace is None or workspace.numel() * workspace.element_size() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("pkv_paged_decode_attn", lib.pkv_paged_decode_attn(
        ctypes.byref(desc), _ptr(q), B, Hq, _ptr(k_pool), _v_ptr(v_pool), _ptr(block_tables),
        block_tables.shape[1], _ptr(seq_lens), float(scale), S, _ptr(workspace), ws_bytes,
        _ptr(out), _ptr(lse), int(flags), _stream(stream)))
    return out, lse


def decode_cascade_splits(k_pool, v_pool, batch: int, num_q_heads: int, max_blocks: int,
                          prefix_blocks: int, prefix_splits: int = 0,
                          suffix_splits: int = 0) -> tuple[int, int]:
    """The (prefix, suffix) split counts a cascade call uses (0 = chosen)."""
    desc = _bf16_desc(k_pool, v_pool)
    s1, s2 = ctypes.c_int32(prefix_splits), ctypes.c_int32(suffix_splits)
    _check("pkv_decode_cascade_splits", lib.pkv_decode_cascade_splits(
        ctypes.byref(desc), batch, num_q_heads, max_blocks, prefix_blocks, ctypes.byref(s1),
        ctypes.byref(s2)))
    return int(s1.value), int(s2.value)


def paged_decode_attn_cascade(q, k_pool, v_pool, prefix_table, block_tables, seq_lens,
                              scale: float, prefix_splits: int = 0, suffix_splits: int = 0,
                              workspace=None, out=None, lse=None, flags: int = 0, stream=None):
    """Decode attention of q [B, Hq, Dk] for sequences whose tables begin with
    the shared blocks `prefix_table` [prefix_blocks] int32 -> (out, lse), as a
    cascade: all rows over the shared prefix, each sequence over its rest,
    merged.  Same result as paged_decode_attn on those tables."""
    desc = _decode_common(q, k_pool, v_pool, block_tables, seq_lens)
    _need(prefix_table, "prefix_table", torch.int32, 1)
    B, Hq, _ = q.shape
    if out is None:
        out = torch.empty(B, Hq, desc.head_dim_v, dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty(B, Hq, dtype=torch.float32, device=q.device)
    P, mb = prefix_table.shape[0], block_tables.shape[1]
    need = int(lib.pkv_decode_cascade_workspace_size(ctypes.byref(desc), B, Hq, mb, P,
                                                     int(prefix_splits), int(suffix_splits)))
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    _check("pkv_paged_decode_attn_cascade", lib.pkv_paged_decode_attn_cascade(
        ctypes.byref(desc), _ptr(q), B, Hq, _ptr(k_pool), _v_ptr(v_pool), _ptr(prefix_table), P,
        _ptr(block_tables), mb, _ptr(seq_lens), float(scale), int(prefix_splits),
        int(suffix_splits), _ptr(workspace), ws_bytes, _ptr(out), _ptr(lse), int(flags),
        _stream(stream)))
    return out, lse


def paged_decode_attn_e4m3(q, k_pool, v_pool, k_scale, v_scale, block_tables, seq_lens,
                           scale: float, num_splits: int = 0, workspace=None, out=None,
                           lse=None, flags: int = 0, stream=None):
    """Decode attention over an E4M3 cache (uint8 code pools, fp32 scales per
    KV head) -> (out, lse); num_splits 0 lets the library choose."""
    desc = _e4m3_desc(k_pool, v_pool, k_scale, v_scale)
    _need(q, "q", torch.float32, 3)
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    B, Hq, _ = q.shape
    if out is None:
        out = torch.empty(B, Hq, desc.head_dim_v, dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty(B, Hq, dtype=torch.float32, device=q.device)
    S = num_splits or int(lib.pkv_decode_auto_splits_e4m3(
        ctypes.byref(desc), B, Hq, block_tables.shape[1] * desc.block_size))
    need = decode_workspace_size(B, Hq, desc.head_dim_v, S)
    if need and (workspace is None or workspace.numel() * workspace.element_size() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("pkv_paged_decode_attn_e4m3", lib.pkv_paged_decode_attn_e4m3(
        ctypes.byref(desc), _ptr(q), B, Hq, _ptr(k_pool), _ptr(v_pool), _ptr(k_scale),
        _ptr(v_scale), _ptr(block_tables), block_tables.shape[1], _ptr(seq_lens), float(scale),
        S, _ptr(workspace), ws_bytes, _ptr(out), _ptr(lse), int(flags), _stream(stream)))
    return out, lse


def paged_decode_attn_partial_e4m3(q, k_pool, v_pool, k_scale, v_scale, block_tables,
                                   seq_lens, scale: float, num_splits: int, out_part=None,
                                   lse_part=None, flags: int = 0, stream=None):
    """Per-split partials over an E4M3 cache -> (out_part [S, B, Hq, Dv],
    lse_part [S, B, Hq])."""
    desc = _e4m3_desc(k_pool, v_pool, k_scale, v_scale)
    _need(q, "q", torch.float32, 3)
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    B, Hq, _ = q.shape
    S = int(num_splits)
    if out_part is None:
        out_part = torch.empty(S, B, Hq, desc.head_dim_v, dtype=torch.float32, device=q.device)
    if lse_part is None:
        lse_part = torch.empty(S, B, Hq, dtype=torch.float32, device=q.device)
    _check("pkv_paged_decode_attn_partial_e4m3", lib.pkv_paged_decode_attn_partial_e4m3(
        ctypes.byref(desc), _ptr(q), B, Hq, _ptr(k_pool), _ptr(v_pool), _ptr(k_scale),
        _ptr(v_scale), _ptr(block_tables), block_tables.shape[1], _ptr(seq_lens), float(scale),
        S, _ptr(out_part), _ptr(lse_part), int(flags), _stream(stream)))
    return out_part, lse_part


def paged_decode_attn_multi_e4m3(q, k_pool, v_pool, k_scale, v_scale, block_tables, seq_lens,
                                 scale: float, num_splits: int = 0, workspace=None, out=None,
                                 lse=None, flags: int = 0, stream=None):
    """The multi-token step (q [B, T, Hq, Dk], causal over the last T tokens) over
    an E4M3 cache -> (out [B, T, Hq, Dv], lse [B, T, Hq])."""
    desc = _e4m3_desc(k_pool, v_pool, k_scale, v_scale)
    _need(q, "q", torch.float32, 4)
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    B, T, Hq, _ = q.shape
    if out is None:
        out = torch.empty(B, T, Hq, desc.head_dim_v, dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty(B, T, Hq, dtype=torch.float32, device=q.device)
    S = num_splits or int(lib.pkv_decode_multi_auto_splits_e4m3(
        ctypes.byref(desc), B, T, Hq, block_tables.shape[1] * desc.block_size))
    need = int(lib.pkv_decode_multi_workspace_size(B, T, Hq, desc.head_dim_v,
                                                   block_tables.shape[1], S))
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    _check("pkv_paged_decode_attn_multi_e4m3", lib.pkv_paged_decode_attn_multi_e4m3(
        ctypes.byref(desc), _ptr(q), B, T, Hq, _ptr(k_pool), _ptr(v_pool), _ptr(k_scale),
        _ptr(v_scale), _ptr(block_tables), block_tables.shape[1], _ptr(seq_lens), float(scale),
        S, _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(out), _ptr(lse),
        int(flags), _stream(stream)))
    return out, lse


def paged_decode_attn_partial(q, k_pool, v_pool, block_tables, seq_lens, scale: float,
                              num_splits: int, out_part=None, lse_part=None, flags: int = 0,
                              stream=None):
    """Per-split partials -> (out_part [S, B, Hq, Dv], lse_part [S, B, Hq])."""
    desc = _decode_common(q, k_pool, v_pool, block_tables, seq_lens)
    B, Hq, _ = q.shape
    S = int(num_splits)
    if out_part is None:
        out_part = torch.empty(S, B, Hq, desc.head_dim_v, dtype=torch.float32, device=q.device)
    if lse_part is None:
        lse_part = torch.empty(S, B, Hq, dtype=torch.float32, device=q.device)
    _check("pkv_paged_decode_attn_partial", lib.pkv_paged_decode_attn_partial(
        ctypes.byref(desc), _ptr(q), B, Hq, _ptr(k_pool), _v_ptr(v_pool), _ptr(block_tables),
        block_tables.shape[1], _ptr(seq_lens), float(scale), S, _ptr(out_part), _ptr(lse_part),
        int(flags), _stream(stream)))
    return out_part, lse_part


def paged_decode_attn_multi(q, k_pool, v_pool, block_tables, seq_lens, scale: float,
                            num_splits: int = 0, workspace=None, out=None, lse=None,
                            flags: int = 0, stream=None):
    """Several new tokens per sequence (q [B, T, Hq, Dk]); query t attends to
    the first seq_lens[b] - T + 1 + t tokens -> (out [B, T, Hq, Dv], lse [B, T, Hq])."""
    desc = _bf16_desc(k_pool, v_pool)
    _need(q, "q", torch.float32, 4)
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    B, T, Hq, _ = q.shape
    if out is None:
        out = torch.empty(B, T, Hq, desc.head_dim_v, dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty(B, T, Hq, dtype=torch.float32, device=q.device)
    S = num_splits
    if S == 0:
        S = int(lib.pkv_decode_multi_auto_splits(ctypes.byref(desc), B, T, Hq,
                                                 block_tables.shape[1] * desc.block_size,
                                                 int(flags)))
    need = int(lib.pkv_decode_multi_workspace_size(B, T, Hq, desc.head_dim_v,
                                                   block_tables.shape[1], S))
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    _check("pkv_paged_decode_attn_multi", lib.pkv_paged_decode_attn_multi(
        ctypes.byref(desc), _ptr(q), B, T, Hq, _ptr(k_pool), _v_ptr(v_pool),
        _ptr(block_tables), block_tables.shape[1], _ptr(seq_lens), float(scale), S,
        _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(out), _ptr(lse),
        int(flags), _stream(stream)))
    return out, lse


def lse_merge(out_part, lse_part, out=None, lse=None, stream=None):
    """Merge P partials: out_part [P, ..., Dv], lse_part [P, ...] -> (out, lse)."""
    _need(out_part, "out_part", torch.float32)
    _need(lse_part, "lse_part", torch.float32)
    P, dv = out_part.shape[0], out_part.shape[-1]
    rows = out_part[0].numel() // dv
    if lse_part.numel() != P * rows:
        raise ValueError("lse_part does not match out_part")
    if out is None:
        out = torch.empty(out_part.shape[1:], dtype=torch.float32, device=out_part.device)
    if lse is None:
        lse = torch.empty(lse_part.shape[1:], dtype=torch.float32, device=lse_part.device)
    _check("pkv_lse_merge", lib.pkv_lse_merge(P, _ptr(out_part), _ptr(lse_part), rows, dv,
                                              _ptr(out), _ptr(lse), _stream(stream)))
    return out, lse


class BlockManager:
    """Host block manager (C++): allocation, reuse, ref-counted sharing, copy-on-write."""

    def __init__(self, num_blocks: int, block_size: int, initial_order=None):
        self.block_size = int(block_size)
        arr = None
        if initial_order is not None:
            order = [int(x) for x in initial_order]
            arr = (ctypes.c_int32 * len(order))(*order)
        self._h = lib.pkv_bm_create(int(num_blocks), int(block_size), arr)
        if not self._h:
            raise ValueError("pkv_bm_create: invalid arguments")

    def __del__(self):
        h = getattr(self, "_h", None)
        if h:
            lib.pkv_bm_destroy(h)
            self._h = None

    def add_sequence(self) -> int:
        sid = ctypes.c_int64(0)
        _check("pkv_bm_add_sequence", lib.pkv_bm_add_sequence(self._h, ctypes.byref(sid)))
        return int(sid.value)

    def fork(self, parent: int) -> int:
        sid = ctypes.c_int64(0)
        _check("pkv_bm_fork", lib.pkv_bm_fork(self._h, int(parent), ctypes.byref(sid)))
        return int(sid.value)

    def append(self, seq: int, num_tokens: int):
        """-> (slots list, copy-on-write pairs [(src, dst)])."""
        slots = (ctypes.c_int64 * max(1, num_tokens))()
        src = (ctypes.c_int32 * 1)()
        dst = (ctypes.c_int32 * 1)()
        n = ctypes.c_int32(0)
        _check("pkv_bm_append", lib.pkv_bm_append(self._h, int(seq), int(num_tokens), slots, src,
                                                  dst, 1, ctypes.byref(n)))
        return list(slots[:num_tokens]), [(src[i], dst[i]) for i in range(n.value)]

    def free(self, seq: int) -> None:
        _check("pkv_bm_free", lib.pkv_bm_free(self._h, int(seq)))

    def block_table(self, seq: int):
        nb = ctypes.c_int32(0)
        ln = ctypes.c_int64(0)
        rc = lib.pkv_bm_block_table(self._h, int(seq), None, 0, ctypes.byref(nb), ctypes.byref(ln))
        if rc not in (0, -2):          # -2: capacity 0 too small, sizes still reported
            _check("pkv_bm_block_table", rc)
        buf = (ctypes.c_int32 * max(1, nb.value))()
        _check("pkv_bm_block_table", lib.pkv_bm_block_table(self._h, int(seq), buf, nb.value,
                                                            ctypes.byref(nb), ctypes.byref(ln)))
        return list(buf[:nb.value])

    def seq_len(self, seq: int) -> int:
        nb = ctypes.c_int32(0)
        ln = ctypes.c_int64(0)
        rc = lib.pkv_bm_block_table(self._h, int(seq), None, 0, ctypes.byref(nb), ctypes.byref(ln))
        if rc not in (0, -2):
            _check("pkv_bm_block_table", rc)
        return int(ln.value)

    @property
    def num_free(self) -> int:
        return int(lib.pkv_bm_num_free(self._h))

    def ref_count(self, block: int) -> int:
        return int(lib.pkv_bm_ref_count(self._h, int(block)))
