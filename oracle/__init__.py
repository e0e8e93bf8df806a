"""CPU oracle for paged decode attention (test infrastructure).

This package is the plain, slow statement of what the GPU library computes.
Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU
baseline leg may import it; the GPU library never does, and the two share no
code.  The arithmetic lives in ``oracle.c`` (plain loops, fp64); this module
only builds that file with gcc, marshals numpy arrays into it, and adds the
two closed-form counting rules the pages state in prose.

Pages cited (title, section):

* "PagedAttentionとは？KVキャッシュを分割してLLMのメモリの無駄を減らす仕組み" --
  "PagedAttentionはブロック表で論理順序と物理配置を分ける" (block table),
  "要求の終了で空いたブロックを再利用する具体例" (block accounting example),
  "共通ブロックの共有とコピーオンライト" (ref counts, copy-on-write).
* "1,000 人が同時に AI に質問したら、誰が最初に答えをもらうのか? KV キャッシュと continuous
  batching" -- "KV キャッシュは何を保持するのか?" (append, then attend) and
  "KV キャッシュのメモリが同時実行数を制限する仕組み" (bytes per token).
* "なぜ長文LLMは遅くなるのか｜Decode Context ParallelismでKVキャッシュを分散する" --
  interleaved token assignment and the three-stage DCP decode step (LSE
  correction and sum of the partial outputs); bytes per cached number by
  data type (FP8: one byte) and KV-cache quantisation to FP8 (E4M3 storage
  below).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``_oracle.so`` with gcc (host code only)."""
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-std=c11", "-pthread",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def load_library(path: str) -> ctypes.CDLL:
    """Load an oracle shared object and declare its signatures."""
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    i32, i64, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
    lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_to_double.restype = f64
    lib.oracle_slot_of.argtypes = [P, i64, i32]
    lib.oracle_slot_of.restype = i64
    lib.oracle_kv_append.argtypes = [i32, i32, i32, i32, i32, P, P, P, P, P, i64]
    lib.oracle_kv_append.restype = i64
    lib.oracle_copy_blocks.argtypes = [i32, i32, i32, i32, i32, P, P, P, P, i32]
    lib.oracle_copy_blocks.restype = i32
    lib.oracle_interleave.argtypes = [i64, i32, i32, P, P]
    lib.oracle_interleave.restype = None
    lib.oracle_lse_merge.argtypes = [i32, i64, i32, P, P, P, P]
    lib.oracle_lse_merge.restype = None
    lib.oracle_paged_decode_attn.argtypes = [i32, i32, i32, i32, i32, i32, i32, P, P, P,
                                             P, P, P, P, f64, P, P, i32]
    lib.oracle_paged_decode_attn.restype = i32
    lib.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
    lib.oracle_e4m3_to_double.restype = f64
    lib.oracle_e4m3_from_double.argtypes = [f64]
    lib.oracle_e4m3_from_double.restype = ctypes.c_uint8
    lib.oracle_kv_append_e4m3.argtypes = [i32, i32, i32, i32, i32, P, P, P, P, P, P, P, i64]
    lib.oracle_kv_append_e4m3.restype = i64
    lib.oracle_paged_decode_attn_e4m3.argtypes = [i32, i32, i32, i32, i32, i32, i32, P, P, P,
                                                  P, P, P, P, P, P, f64, P, P, i32]
    lib.oracle_paged_decode_attn_e4m3.restype = i32
    return lib


def _get():
    global _lib
    with _lock:
        if _lib is None:
            _lib = load_library(build())
    return _lib


def _ptr(a: np.ndarray | None):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    """A C-contiguous array of exactly `dtype` (no value conversion for bit types)."""
    a = np.asarray(a)
    if a.dtype != np.dtype(dtype):
        if np.dtype(dtype) == np.uint16 and a.dtype == np.int16:
            a = a.view(np.uint16)
        else:
            a = a.astype(dtype)
    return np.ascontiguousarray(a)


# --------------------------------------------------------------------------
# closed-form counting rules stated in prose on the pages
# --------------------------------------------------------------------------

def kv_bytes_per_token(layers: int, kv_heads: int, head_dim: int, bytes_per_number: int) -> int:
    """Bytes of raw K and V per token: 2 (key and value) x layers x KV heads x
    head size x bytes per number ("KV キャッシュのメモリが同時実行数を制限する仕組み").
    It assumes one K and one V vector per KV head (MHA/GQA)."""
    return 2 * layers * kv_heads * head_dim * bytes_per_number


def blocks_needed(num_tokens: int, block_size: int) -> int:
    """Blocks a sequence holds: the current block is used until it is full, then
    one more is taken ("PagedAttentionはブロック表で論理順序と物理配置を分ける"), so a
    sequence of n tokens holds the smallest number of blocks that fits n."""
    blocks = 0
    while blocks * block_size < num_tokens:
        blocks += 1
    return blocks


# --------------------------------------------------------------------------
# wrappers over oracle.c
# --------------------------------------------------------------------------

def bf16_to_double(bits: int) -> float:
    return _get().oracle_bf16_to_double(int(bits) & 0xFFFF)


def slot_of(table_row, pos: int, block_size: int) -> int:
    row = _c(table_row, np.int32)
    return int(_get().oracle_slot_of(_ptr(row), int(pos), int(block_size)))


def slot_mapping(block_tables, seq_ids, positions, block_size: int) -> np.ndarray:
    """Slot of each (sequence, position) pair through that sequence's table row."""
    tables = _c(block_tables, np.int32)
    out = np.empty(len(positions), dtype=np.int64)
    lib = _get()
    for i, (b, pos) in enumerate(zip(seq_ids, positions)):
        row = tables[int(b)]
        out[i] = lib.oracle_slot_of(_ptr(row), int(pos), int(block_size))
    return out


def kv_append(k_pool, v_pool, k_new, v_new, slots, block_size: int) -> int:
    """In-place scatter of new tokens into the pools (uint16 bf16 bit arrays of
    shape [num_blocks, Hkv, bs, D]).  Returns the count of out-of-range slots."""
    assert k_pool.dtype == np.uint16 and k_pool.flags.c_contiguous
    assert v_pool.dtype == np.uint16 and v_pool.flags.c_contiguous
    nb, hkv, bs, dk = k_pool.shape
    dv = v_pool.shape[3]
    assert bs == block_size
    kn = _c(k_new, np.uint16)
    vn = _c(v_new, np.uint16)
    sl = _c(slots, np.int64)
    return int(_get().oracle_kv_append(nb, bs, hkv, dk, dv, _ptr(k_pool), _ptr(v_pool),
                                       _ptr(kn), _ptr(vn), _ptr(sl), len(sl)))


def copy_blocks(k_pool, v_pool, src, dst) -> int:
    assert k_pool.dtype == np.uint16 and k_pool.flags.c_contiguous
    assert v_pool.dtype == np.uint16 and v_pool.flags.c_contiguous
    nb, hkv, bs, dk = k_pool.shape
    dv = v_pool.shape[3]
    s = _c(src, np.int32)
    d = _c(dst, np.int32)
    assert len(s) == len(d)
    return int(_get().oracle_copy_blocks(nb, bs, hkv, dk, dv, _ptr(k_pool), _ptr(v_pool),
                                         _ptr(s), _ptr(d), len(s)))


def interleave(num_tokens: int, num_parts: int, interleave_size: int):
    """(partition of each token, position inside its partition)."""
    part = np.empty(num_tokens, dtype=np.int32)
    local = np.empty(num_tokens, dtype=np.int64)
    _get().oracle_interleave(int(num_tokens), int(num_parts), int(interleave_size),
                             _ptr(part), _ptr(local))
    return part, local


def lse_merge(out_part, lse_part):
    """out_part [P, ..., Dv], lse_part [P, ...] -> (out [..., Dv], lse [...]) in fp64."""
    op = _c(out_part, np.float64)
    lp = _c(lse_part, np.float64)
    P = op.shape[0]
    dv = op.shape[-1]
    rows = int(np.prod(op.shape[1:-1], dtype=np.int64))
    assert lp.shape[0] == P and int(np.prod(lp.shape[1:], dtype=np.int64)) == rows
    out = np.empty(op.shape[1:], dtype=np.float64)
    lse = np.empty(lp.shape[1:], dtype=np.float64)
    _get().oracle_lse_merge(P, rows, dv, _ptr(op), _ptr(lp), _ptr(out), _ptr(lse))
    return out, lse


def paged_decode_attn(q, k_pool, v_pool, block_tables, seq_lens, scale: float,
                      tok_begin=None, tok_end=None, num_threads: int = 0):
    """Exact softmax attention of q [B, Hq, Dk] (fp32) over each sequence's
    tokens, gathered through its block table.  Returns (out [B, Hq, Dv],
    lse [B, Hq]) in fp64.  Optional per-sequence token ranges [begin, end)."""
    q = _c(q, np.float32)
    kp = _c(k_pool, np.uint16)
    vp = _c(v_pool, np.uint16)
    bt = _c(block_tables, np.int32)
    sl = _c(seq_lens, np.int32)
    B, Hq, Dk = q.shape
    nb, hkv, bs, dk = kp.shape
    dv = vp.shape[3]
    assert dk == Dk and bt.shape[0] == B and sl.shape[0] == B
    tb = None if tok_begin is None else _c(tok_begin, np.int32)
    te = None if tok_end is None else _c(tok_end, np.int32)
    out = np.empty((B, Hq, dv), dtype=np.float64)
    lse = np.empty((B, Hq), dtype=np.float64)
    rc = _get().oracle_paged_decode_attn(B, Hq, hkv, Dk, dv, bs, bt.shape[1], _ptr(q),
                                         _ptr(kp), _ptr(vp), _ptr(bt), _ptr(sl), _ptr(tb),
                                         _ptr(te), float(scale), _ptr(out), _ptr(lse),
                                         int(num_threads))
    if rc != 0:
        raise ValueError("oracle_paged_decode_attn: inconsistent arguments")
    return out, lse


def e4m3_to_double(code: int) -> float:
    """Value of one E4M3 code (NaN for the two NaN codes)."""
    return _get().oracle_e4m3_to_double(int(code) & 0xFF)


def e4m3_from_double(x: float) -> int:
    """The E4M3 code nearest to x (ties to even, saturating at +-448)."""
    return int(_get().oracle_e4m3_from_double(float(x)))


def e4m3_table() -> np.ndarray:
    """fp64 value of each of the 256 codes."""
    lib = _get()
    return np.array([lib.oracle_e4m3_to_double(c) for c in range(256)], dtype=np.float64)


def kv_append_e4m3(k_pool, v_pool, k_new, v_new, k_scale, v_scale, slots,
                   block_size: int) -> int:
    """In-place scatter of new bf16 tokens (uint16 bits) into E4M3 pools
    (uint8 [num_blocks, Hkv, bs, D]), each element stored as the code nearest
    to x / scale of its KV head.  Returns the count of out-of-range slots."""
    assert k_pool.dtype == np.uint8 and k_pool.flags.c_contiguous
    assert v_pool.dtype == np.uint8 and v_pool.flags.c_contiguous
    nb, hkv, bs, dk = k_pool.shape
    dv = v_pool.shape[3]
    assert bs == block_size
    kn = _c(k_new, np.uint16)
    vn = _c(v_new, np.uint16)
    ks = _c(k_scale, np.float32)
    vs = _c(v_scale, np.float32)
    assert ks.shape == (hkv,) and vs.shape == (hkv,)
    sl = _c(slots, np.int64)
    return int(_get().oracle_kv_append_e4m3(nb, bs, hkv, dk, dv, _ptr(k_pool), _ptr(v_pool),
                                            _ptr(kn), _ptr(vn), _ptr(ks), _ptr(vs), _ptr(sl),
                                            len(sl)))


def paged_decode_attn_e4m3(q, k_pool, v_pool, k_scale, v_scale, block_tables, seq_lens,
                           scale: float, tok_begin=None, tok_end=None, num_threads: int = 0):
    """paged_decode_attn over E4M3 pools (uint8 codes): K_j and V_j are the
    decoded codes times their KV head's scale.  Returns (out, lse) in fp64."""
    q = _c(q, np.float32)
    kp = _c(k_pool, np.uint8)
    vp = _c(v_pool, np.uint8)
    ks = _c(k_scale, np.float32)
    vs = _c(v_scale, np.float32)
    bt = _c(block_tables, np.int32)
    sl = _c(seq_lens, np.int32)
    B, Hq, Dk = q.shape
    nb, hkv, bs, dk = kp.shape
    dv = vp.shape[3]
    assert dk == Dk and bt.shape[0] == B and sl.shape[0] == B
    assert ks.shape == (hkv,) and vs.shape == (hkv,)
    tb = None if tok_begin is None else _c(tok_begin, np.int32)
    te = None if tok_end is None else _c(tok_end, np.int32)
    out = np.empty((B, Hq, dv), dtype=np.float64)
    lse = np.empty((B, Hq), dtype=np.float64)
    rc = _get().oracle_paged_decode_attn_e4m3(B, Hq, hkv, Dk, dv, bs, bt.shape[1], _ptr(q),
                                              _ptr(kp), _ptr(vp), _ptr(ks), _ptr(vs), _ptr(bt),
                                              _ptr(sl), _ptr(tb), _ptr(te), float(scale),
                                              _ptr(out), _ptr(lse), int(num_threads))
    if rc != 0:
        raise ValueError("oracle_paged_decode_attn_e4m3: inconsistent arguments")
    return out, lse


def paged_decode_attn_multi(q, k_pool, v_pool, block_tables, seq_lens, scale: float,
                            num_threads: int = 0):
    """Several new tokens per sequence: q [B, T, Hq, Dk].  The last T of the
    seq_lens[b] stored tokens are the new ones, and query t attends to the
    tokens j < seq_lens[b] - T + 1 + t (causal among the new tokens): each
    (sequence, query token) is an ordinary decode over that token range.
    Returns (out [B, T, Hq, Dv], lse [B, T, Hq]) in fp64."""
    q = np.ascontiguousarray(q, dtype=np.float32)
    B, T, Hq, Dk = q.shape
    tables = np.repeat(np.asarray(block_tables, dtype=np.int32), T, axis=0)
    lens = np.repeat(np.asarray(seq_lens, dtype=np.int32), T)
    t = np.tile(np.arange(T, dtype=np.int32), B)
    end = np.maximum(lens - (T - 1) + t, 0).astype(np.int32)
    out, lse = paged_decode_attn(q.reshape(B * T, Hq, Dk), k_pool, v_pool, tables, lens, scale,
                                 tok_end=end, num_threads=num_threads)
    return out.reshape(B, T, Hq, -1), lse.reshape(B, T, Hq)
