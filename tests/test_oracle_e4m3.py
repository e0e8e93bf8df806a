"""Pins of the oracle's FP8 (E4M3) cache storage: the code table, the encoder,
the quantising append and attention over E4M3 pools, each checked against
something other than the oracle itself -- torch's own float8_e4m3fn
conversion, literal values of the format, and the bf16 oracle path."""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle


def torch_table() -> np.ndarray:
    codes = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn)
    return codes.to(torch.float64).numpy()


def test_code_table_matches_torch_and_literals():
    t = oracle.e4m3_table()
    ref = torch_table()
    finite = ~np.isnan(ref)
    assert np.array_equal(np.isnan(t), ~finite)
    assert np.array_equal(t[finite], ref[finite])
    # literal values of the format: smallest subnormal, largest subnormal,
    # smallest normal, one, the largest finite magnitude, a value with a
    # full mantissa, signed zero
    assert t[0x01] == 2.0 ** -9 and t[0x07] == 7 * 2.0 ** -9 and t[0x08] == 2.0 ** -6
    assert t[0x38] == 1.0 and t[0x40] == 2.0 and t[0x7E] == 448.0 and t[0x77] == 240.0
    assert t[0xFE] == -448.0 and t[0x80] == 0.0 and math.copysign(1.0, t[0x80]) == -1.0
    assert np.isnan(t[0x7F]) and np.isnan(t[0xFF])
    # 127 non-negative finite codes, strictly increasing
    assert np.all(np.diff(t[:0x7F]) > 0)


def test_encoder_matches_torch_rounding():
    rng = np.random.default_rng(5)
    x = np.concatenate([
        rng.normal(0, 1, 4000), rng.normal(0, 60, 4000), rng.uniform(-463, 463, 2000),
        rng.normal(0, 2.0 ** -7, 2000),                       # subnormal range
    ]).astype(np.float32)
    t = oracle.e4m3_table()
    finite = t[~np.isnan(t)]
    mids = ((finite[1:] + finite[:-1]) / 2)[np.abs(finite[1:]) < 449]   # exact ties
    x = np.concatenate([x, mids.astype(np.float32)]).astype(np.float32)
    got = np.array([oracle.e4m3_from_double(float(v)) for v in x], dtype=np.uint8)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got, ref)


def test_encoder_saturates_and_keeps_nan():
    for v in (448.0, 463.9, 464.0, 1e6, math.inf):
        assert oracle.e4m3_from_double(v) == 0x7E
        assert oracle.e4m3_from_double(-v) == 0xFE
    assert oracle.e4m3_from_double(math.nan) == 0x7F
    assert oracle.e4m3_from_double(-0.0) == 0x80


def _bf16_bits(x: torch.Tensor) -> np.ndarray:
    return x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_append_quantises_like_torch():
    g = torch.Generator().manual_seed(3)
    nb, hkv, bs, dk, dv = 6, 2, 4, 16, 8
    k_new = torch.randn(5, hkv, dk, generator=g) * 3
    v_new = torch.randn(5, hkv, dv, generator=g) * 40
    ks = np.array([0.05, 0.3], dtype=np.float32)
    vs = np.array([0.5, 1.0], dtype=np.float32)
    kp = np.zeros((nb, hkv, bs, dk), dtype=np.uint8)
    vp = np.zeros((nb, hkv, bs, dv), dtype=np.uint8)
    slots = np.array([0, 5, -1, 13, 99], dtype=np.int64)       # one skipped, one out of range
    bad = oracle.kv_append_e4m3(kp, vp, _bf16_bits(k_new), _bf16_bits(v_new), ks, vs, slots, bs)
    assert bad == 1

    def quant(x, s):   # binary32 quotient, then torch's nearest-even cast
        y = x.to(torch.bfloat16).to(torch.float32) / torch.from_numpy(s)[None, :, None]
        assert y.abs().max() < 464
        return y.to(torch.float8_e4m3fn).view(torch.uint8).numpy()

    qk, qv = quant(k_new, ks), quant(v_new, vs)
    ek = np.zeros_like(kp)
    ev = np.zeros_like(vp)
    for t, slot in enumerate(slots):
        if 0 <= slot < nb * bs:
            ek[slot // bs, :, slot % bs] = qk[t]
            ev[slot // bs, :, slot % bs] = qv[t]
    assert np.array_equal(kp, ek) and np.array_equal(vp, ev)


def _e4m3_case(seed, lens, hq, hkv, d, bs):
    rng = np.random.default_rng(seed)
    counts = [-(-n // bs) for n in lens]
    nb = sum(counts) + 2
    perm = rng.permutation(nb).astype(np.int32)
    tables = np.full((len(lens), max(counts)), -1, dtype=np.int32)
    at = 0
    for b, c in enumerate(counts):
        tables[b, :c] = perm[at:at + c]
        at += c
    # finite codes only (not the two NaN codes)
    codes = rng.integers(0, 256, size=(2, nb, hkv, bs, d)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x38
    q = rng.normal(0, 1, (len(lens), hq, d)).astype(np.float32)
    return q, codes[0], codes[1], tables, np.array(lens, dtype=np.int32)


def test_attention_equals_bf16_path_on_exact_values():
    """Power-of-two scales: every dequantised value is exact in bf16, so the
    E4M3 path must give the bf16 oracle's bits on those values."""
    q, kc, vc, tables, lens = _e4m3_case(8, [37, 5, 64], 8, 2, 16, 8)
    ks = np.array([2.0 ** -3, 2.0 ** -5], dtype=np.float32)
    vs = np.array([2.0 ** -1, 4.0], dtype=np.float32)
    t = oracle.e4m3_table()
    kv = t[kc] * ks[None, :, None, None]
    vv = t[vc] * vs[None, :, None, None]
    kb = _bf16_bits(torch.from_numpy(kv))
    vb = _bf16_bits(torch.from_numpy(vv))
    assert np.array_equal(np.array([oracle.bf16_to_double(b) for b in kb.ravel()[:500]]),
                          kv.ravel()[:500])
    o8, l8 = oracle.paged_decode_attn_e4m3(q, kc, vc, ks, vs, tables, lens, 0.25)
    ob, lb = oracle.paged_decode_attn(q, kb, vb, tables, lens, 0.25)
    assert np.array_equal(o8, ob) and np.array_equal(l8, lb)


def test_value_scale_is_linear_and_matches_brute_force():
    q, kc, vc, tables, lens = _e4m3_case(9, [23, 1], 4, 1, 8, 4)
    ks = np.array([0.037], dtype=np.float32)
    o1, l1 = oracle.paged_decode_attn_e4m3(q, kc, vc, ks, np.array([1.0], np.float32),
                                           tables, lens, 0.3)
    o3, l3 = oracle.paged_decode_attn_e4m3(q, kc, vc, ks, np.array([0.3], np.float32),
                                           tables, lens, 0.3)
    assert np.allclose(o3, o1 * np.float64(np.float32(0.3)), rtol=1e-13, atol=0)
    assert np.array_equal(l1, l3)
    # brute force in numpy on the logical token order
    t = oracle.e4m3_table()
    for b, L in enumerate(lens):
        rows = [tables[b, j // 4] for j in range(L)]
        K = np.stack([t[kc[rows[j], 0, j % 4]] for j in range(L)]) * np.float64(ks[0])
        V = np.stack([t[vc[rows[j], 0, j % 4]] for j in range(L)])
        s = 0.3 * (q[b].astype(np.float64) @ K.T)
        m = s.max(axis=1, keepdims=True)
        p = np.exp(s - m)
        ref = (p @ V) / p.sum(axis=1, keepdims=True)
        assert np.allclose(o1[b], ref, rtol=1e-12, atol=1e-12)
        assert np.allclose(l1[b], (m[:, 0] + np.log(p.sum(axis=1))), rtol=0, atol=1e-12)


@pytest.mark.parametrize("mutant", ["round_half_up", "no_subnormals"])
def test_pins_catch_encoder_mistakes(mutant):
    """A plausible mistake in the encoder fails the torch comparison."""
    t = oracle.e4m3_table()
    finite = t[:0x7F]

    def enc(x):
        a = abs(x)
        i = int(np.searchsorted(finite, a))
        lo, hi = finite[max(i - 1, 0)], finite[min(i, 0x7E)]
        if mutant == "round_half_up":
            c = i if a - lo >= hi - a else i - 1
        else:   # flush the subnormal range to zero
            c = 0 if a < 2.0 ** -6 else int(np.argmin(np.abs(finite - a)))
        return max(c, 0) | (0x80 if x < 0 else 0)

    x = np.array([1.0625, 3 * 2.0 ** -10, 2.0 ** -8, 0.75, -1.1875], dtype=np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([enc(float(v)) for v in x], dtype=np.uint8)
    assert not np.array_equal(got, ref)
    assert np.array_equal(np.array([oracle.e4m3_from_double(float(v)) for v in x]), ref)
