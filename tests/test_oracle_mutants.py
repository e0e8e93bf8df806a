"""The pins must be strong enough to catch plausible mistakes in the oracle.

Each mutant below is one such mistake (a dropped term, a wrong sign, index or
operand) planted in a temporary copy of ``oracle/oracle.c``, compiled with
gcc on the CPU.  The whole pin suite of ``test_oracle_pins.py`` then runs
against the mutant, and at least one pin must fail.  The real oracle is never
modified.
"""
from __future__ import annotations

import inspect
import itertools
import os
import subprocess

import pytest

import oracle
from tests import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

MUTANTS = {
    "offset_uses_block_index": ("int64_t off = j % J->bs;", "int64_t off = j / J->bs;"),
    "scale_dropped": ("scores[j - begin] = J->scale * dot;", "scores[j - begin] = dot;"),
    "group_mapping_modulo": ("int32_t g = h / (J->Hq / J->Hkv);", "int32_t g = h % J->Hkv;"),
    "lse_without_max": ("J->lse[row] = m + log(z);", "J->lse[row] = log(z);"),
    "output_not_normalised": ("o[d] /= z;", "o[d] /= 1.0;"),
    "exp_without_shift": ("double p = exp(scores[j - begin] - m);",
                          "double p = exp(scores[j - begin]);"),
    "value_row_uses_k_dim": ("* J->bs + off) * J->Dv;", "* J->bs + off) * J->Dk;"),
    "merge_weight_sign": ("acc += w * out_part", "acc -= w * out_part"),
    "merge_lse_no_log": ("lse[r] = m + log(wsum);", "lse[r] = m + wsum;"),
    "merge_max_is_first": ("if (lse_part[p * rows + r] > m)", "if (p == 0)"),
    "interleave_ignores_size": ("(i / interleave) % num_parts", "i % num_parts"),
    "interleave_local_global": ("local[i] = count[r];", "local[i] = i;"),
    "slot_operands_swapped": ("return (int64_t)table_row[logical_block] * block_size + offset;",
                              "return (int64_t)table_row[offset] * block_size + logical_block;"),
    "append_head_stride": ("k_new[(t * num_kv_heads + g) * head_dim_k + d];",
                           "k_new[(g * num_kv_heads + t) * head_dim_k + d];"),
    "copy_skips_values": ("memcpy(v_pool + (size_t)dst[i] * v_block",
                          "if (0) memcpy(v_pool + (size_t)dst[i] * v_block"),
    "bf16_wrong_shift": ("((uint32_t)bits) << 16;", "((uint32_t)bits) << 15;"),
    "range_end_ignored": ("if (end > J->seq_lens[b])\n        end = J->seq_lens[b];",
                          "end = J->seq_lens[b];"),
}


def _pin_calls():
    """Every pin test of test_oracle_pins as a zero-argument callable."""
    calls = []
    for name, fn in inspect.getmembers(pins, inspect.isfunction):
        if not name.startswith("test_"):
            continue
        marks = [m for m in getattr(fn, "pytestmark", []) if m.name == "parametrize"]
        if not marks:
            calls.append((name, fn, {}))
            continue
        grids = []
        for m in marks:
            names = [s.strip() for s in m.args[0].split(",")]
            grids.append([dict(zip(names, v if len(names) > 1 else (v,))) for v in m.args[1]])
        for combo in itertools.product(*grids):
            kw = {}
            for d in combo:
                kw.update(d)
            calls.append((name, fn, kw))
    return calls


def _build_mutant(tmp_path, name, old, new):
    src = open(SRC, encoding="utf-8").read()
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    mutated = src.replace(old, new)
    c_path = tmp_path / f"{name}.c"
    so_path = tmp_path / f"{name}.so"
    c_path.write_text(mutated, encoding="utf-8")
    subprocess.check_call(["gcc", "-O1", "-fPIC", "-shared", "-std=c11", "-pthread",
                           "-o", str(so_path), str(c_path), "-lm"])
    return oracle.load_library(str(so_path))


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path, monkeypatch):
    old, new = MUTANTS[name]
    lib = _build_mutant(tmp_path, name, old, new)
    monkeypatch.setattr(oracle, "_lib", lib)
    caught = []
    for test_name, fn, kw in _pin_calls():
        try:
            fn(**kw)
        except (AssertionError, ValueError, IndexError) as e:   # a pin failed
            caught.append((test_name, type(e).__name__))
    assert caught, f"mutant {name} survived every pin"


def test_unmutated_oracle_passes_every_pin():
    for _, fn, kw in _pin_calls():
        fn(**kw)
