"""Benchmark of the paged decode-attention step on GB300.

Default workload (`long32k`): batch 8, every context 32,768 tokens, GQA 32
query / 8 KV heads, head_dim 128, bf16 K/V, block size 16, physical blocks a
random permutation of a 16,384-block pool, split-KV over 16 chunks merged
with lse_merge.  One step = slot mapping + kv_append of the 8 decode tokens
+ the split attention kernel + the LSE merge (the exact launches that
pkv_paged_decode_attn makes), with the KV cache resident in HBM.  Steps run
back to back: the 1.07 GB of KV a step reads is 8x the 129 MB L2, so no
flush is needed between them (a flush would add its own write-back traffic).
The same step at the split count the library chooses itself (num_splits = 0)
is timed as well and reported as `library_auto_splits`.

Besides the mean over the timed steps, the line carries per-step CUDA-event
times (median, min, mean; `ms_per_step_events`), the same step with L2
evicted before every repetition (`cold_l2`), and the oracle on one host core
(`cpu_baseline.single_thread`) for the four GQA workloads.

Other workloads (--workload): `dcp200k` (one 200,000-token sequence split
into 4 interleaved partitions, each attended separately and merged) and
`agent_mla` (32 sequences sharing a 136K-token prefix, MLA-shaped 128 heads
over one 576/512 latent head, copy-on-write of the shared tail + append +
attention).

Metric: HBM GB/s over the step's algorithmic bytes (every cached K/V byte
once, plus q, block tables, appended tokens, out and lse), its fraction of the
measured peak, and sequence-tokens/s.  Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "paged decode-attn HBM GB/s (% of GB300 peak), seq-tokens/s at 32K ctx GQA"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS_SUSTAINED = 1700.0
# Per workload: the committed ncu summary of its dominant kernel and the
# sources that kernel is built from (the summary's traffic counts only while
# their hash matches).
PROFILES = {
    "long32k": ("decode_tma_long32k.txt", ("decode_tma.cu", "pkv_device.cuh", "pkv_math.cuh")),
    "dcp200k": ("decode_tma_dcp200k.txt", ("decode_tma.cu", "pkv_device.cuh", "pkv_math.cuh")),
    "dcp200k_e4m3": ("decode_gqa_tc_e4m3_dcp200k.txt",
                     ("decode_gqa_tc_e4m3.cu", "pkv_device.cuh", "pkv_tcgen05.cuh",
                      "pkv_pipeline.cuh", "pkv_math.cuh")),
    "spec4_32k": ("decode_gqa_tc_spec4_32k.txt",
                  ("decode_gqa_tc.cu", "pkv_device.cuh", "pkv_tcgen05.cuh", "pkv_pipeline.cuh",
                   "pkv_math.cuh")),
    "spec4_32k_e4m3": ("decode_gqa_tc_e4m3_spec4_32k.txt",
                       ("decode_gqa_tc_e4m3.cu", "pkv_device.cuh", "pkv_tcgen05.cuh",
                        "pkv_pipeline.cuh", "pkv_math.cuh")),
    "long32k_e4m3": ("decode_gqa_tc_e4m3_long32k.txt",
                     ("decode_gqa_tc_e4m3.cu", "pkv_device.cuh", "pkv_tcgen05.cuh",
                      "pkv_pipeline.cuh", "pkv_math.cuh")),
    "agent_mla": ("decode_mla_tc_agent_mla.txt",
                  ("decode_mla_tc.cu", "pkv_device.cuh", "pkv_tcgen05.cuh", "pkv_pipeline.cuh",
                   "pkv_math.cuh")),
    "agent_mla_e4m3": ("decode_mla_tc_e4m3_agent_mla.txt",
                       ("decode_mla_tc.cu", "pkv_device.cuh", "pkv_tcgen05.cuh",
                        "pkv_pipeline.cuh", "pkv_math.cuh")),
}


# ----------------------------------------------------------------- helpers

def elem_bytes(w) -> int:
    """Bytes of one cached number: 1 for an E4M3 cache, 2 for bf16."""
    return 1 if w.k_codes is not None else 2


def kv_bytes_per_token(w) -> int:
    """K and V bytes one token occupies in one layer: (Dk + Dv) x Hkv x the
    element size, or Dk x Hkv x it when the values live inside the key rows."""
    if w.v_pool is None:
        return w.head_dim_k * w.num_kv_heads * elem_bytes(w)
    return (w.head_dim_k + w.head_dim_v) * w.num_kv_heads * elem_bytes(w)


def unique_kv_tokens(w) -> int:
    """Tokens of K/V the step must read, a physical block shared by several
    sequences counted once (the most tokens any of them uses in it)."""
    used = {}
    tables = w.block_tables.tolist()
    for b, L in enumerate(w.seq_lens.tolist()):
        for i in range(-(-L // w.block_size)):
            n = min(w.block_size, L - i * w.block_size)
            phys = tables[b][i]
            used[phys] = max(used.get(phys, 0), n)
    return sum(used.values())


def step_bytes(w, splits: int):
    """Algorithmic bytes of one step, and of one launch of the split kernel."""
    lens = w.seq_lens.to(torch.int64)
    kv = unique_kv_tokens(w) * kv_bytes_per_token(w)
    B, Hq = w.batch, w.num_q_heads
    rows = w.q.numel() // w.head_dim_k          # (sequence, query token, head) rows
    q = rows * w.head_dim_k * 4
    tables = int(((lens + w.block_size - 1) // w.block_size).sum()) * 4 + B * 4
    out = rows * (w.head_dim_v + 1) * 4
    T = int(w.new_pos.numel())
    # the append reads bf16 new tokens and writes cache elements
    append = T * (kv_bytes_per_token(w) // elem_bytes(w)) * (2 + elem_bytes(w)) + T * (8 + 4 + 8)
    kernel = kv + q + tables
    return kv + q + tables + out + append, kernel


def load_peak(key="hbm_gbs", fallback=None):
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)[key]), "measured"
    except Exception:
        return (FALLBACK_HBM_GBS if fallback is None else fallback), "fallback"


def kernel_flops(w):
    """Algorithmic flops of one split-kernel launch: every (token, query head)
    pair costs a Dk-long and a Dv-long multiply-add chain."""
    return int(w.seq_lens.to(torch.int64).sum()) * w.num_q_heads * \
        (w.head_dim_k + w.head_dim_v) * 2


def code_only(text: str) -> str:
    """C++ source without its comments and blank space: the profile summaries
    are tied to the code they measured, not to its comments."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def stored_traffic(workload):
    """Per-launch DRAM bytes from the workload's committed ncu summary, if it
    was taken on the current kernel sources (else None)."""
    if workload not in PROFILES:
        return None
    name, sources = PROFILES[workload]
    try:
        h = hashlib.sha256()
        for src in sources:
            with open(os.path.join(ROOT, "paged_kv_cache_93_gb300", "csrc", src),
                      encoding="utf-8") as f:
                h.update(code_only(f.read()).encode())
        vals = {}
        with open(os.path.join(ROOT, "profiles", name), encoding="utf-8") as f:
            for line in f:
                if "=" in line and not line.lstrip().startswith("#"):
                    k, v = line.split("=", 1)
                    vals[k.strip()] = v.strip()
        if vals.get("source_sha256") != h.hexdigest():
            return None
        return int(vals["traffic_bytes_per_launch"])
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed region runs."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.samples = []
        self.proc = None
        self.window = None
        ident = str(device_index)
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            ident = uuid if uuid.startswith("GPU-") else f"GPU-{uuid}"
        except Exception:
            pass
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", ident, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [x.strip() for x in line.split(",")]))

    def wait_ready(self, timeout=5.0):
        t = time.time()
        while self.proc and not self.samples and time.time() - t < timeout:
            time.sleep(0.02)

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0, t1):
        rows = [s for ts, s in self.samples if t0 <= ts <= t1 and len(s) >= 8]
        if not rows:
            rows = [s for _, s in self.samples if len(s) >= 8][-3:]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[0]) for r in rows if num(r[0]) is not None]
        mx = [num(r[1]) for r in rows if num(r[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[4:8]) if v.strip() == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


def bits_view(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


# ------------------------------------------------------------ device state

class Step:
    """Device-resident state of one GQA workload and its decode step."""
    kernel_name = "decode_tma_kernel (split attention)"

    def __init__(self, pkv, w, dev, splits):
        self.pkv, self.w, self.splits = pkv, w, splits
        self.k = w.k_pool.to(dev)
        self.v = pkv.ValuesInKeys(w.head_dim_v) if w.v_pool is None else w.v_pool.to(dev)
        self.bt = w.block_tables.to(dev)
        self.lens = w.seq_lens.to(dev)
        self.q = w.q.to(dev)
        self.new_seq = w.new_seq.to(dev)
        self.new_pos = w.new_pos.to(dev)
        self.k_new = w.k_new.to(dev)
        self.v_new = None if w.v_new is None else w.v_new.to(dev)
        B, Hq = w.batch, w.num_q_heads
        self.slots = torch.empty(w.new_pos.numel(), dtype=torch.int64, device=dev)
        self.out = torch.empty(B, Hq, w.head_dim_v, device=dev)
        self.lse = torch.empty(B, Hq, device=dev)
        self.ws = torch.zeros(max(1, pkv.decode_workspace_size(B, Hq, w.head_dim_v, splits)),
                              dtype=torch.uint8, device=dev)
        self.out_part = torch.empty(splits, B, Hq, w.head_dim_v, device=dev)
        self.lse_part = torch.empty(splits, B, Hq, device=dev)
        self.launches = 4   # slot, append, split, merge
        self.desc = (f"slot_mapping + kv_append ({w.new_pos.numel()} decode tokens) + "
                     f"paged_decode_attn ({splits} splits) = split kernel + lse_merge")

    def kernel(self):
        """The split attention kernel alone (the roofline's kernel)."""
        self.pkv.paged_decode_attn_partial(self.q, self.k, self.v, self.bt, self.lens,
                                           self.w.scale, self.splits, out_part=self.out_part,
                                           lse_part=self.lse_part)

    def attend(self, ev_a=None, ev_b=None):
        """What pkv_paged_decode_attn launches: the split kernel, then the merge
        (events, if given, bracket the split kernel)."""
        if self.splits == 1 or ev_a is None:
            if ev_a is not None:
                ev_a.record()
            self.pkv.paged_decode_attn(self.q, self.k, self.v, self.bt, self.lens, self.w.scale,
                                       num_splits=self.splits, workspace=self.ws, out=self.out,
                                       lse=self.lse)
            if ev_b is not None:
                ev_b.record()
            return
        ev_a.record()
        self.kernel()
        ev_b.record()
        self.pkv.lse_merge(self.out_part, self.lse_part, out=self.out, lse=self.lse)

    def run(self, ev_a=None, ev_b=None):
        p = self.pkv
        p.slot_mapping(self.k, self.v, self.bt, self.new_seq, self.new_pos, out=self.slots)
        p.kv_append(self.k, self.v, self.k_new, self.v_new, self.slots)
        self.attend(ev_a, ev_b)


class DcpStep(Step):
    """200K tokens in P interleaved partitions: the decode token goes to its
    partition, each partition is attended separately (its own block table),
    and the P partial results are merged."""

    def __init__(self, pkv, w, dev, splits):
        super().__init__(pkv, w, dev, splits)
        N, P = int(w.seq_lens[0]), w.num_parts
        self.ptab = w.part_tables.to(dev)
        kt, vt = w.k_tokens.to(dev), w.v_tokens.to(dev)
        pkv.kv_append(self.k, self.v, kt[:N - 1], vt[:N - 1],
                      pkv.interleave_slot_mapping(self.k, self.v, 0, N - 1, P, w.interleave,
                                                  self.ptab))
        del kt, vt
        self.N, self.P = N, P
        # The P partitions are attended in ONE launch, as P rows of a batch
        # that share the query and each read their own table -- the
        # single-GPU image of P DCP ranks attending concurrently.
        self.plen = torch.tensor([pkv.interleave_partition_len(N, P, w.interleave, r)
                                  for r in range(P)], dtype=torch.int32, device=dev)
        Hq, Dv = w.num_q_heads, w.head_dim_v
        self.pq = self.q.expand(P, Hq, w.head_dim_k).contiguous()
        self.pout = torch.empty(P, Hq, Dv, device=dev)
        self.plse = torch.empty(P, Hq, device=dev)
        self.ws = torch.zeros(pkv.decode_workspace_size(P, Hq, Dv, splits), dtype=torch.uint8,
                              device=dev)
        self.sp_out = torch.empty(splits, P, Hq, Dv, device=dev)
        self.sp_lse = torch.empty(splits, P, Hq, device=dev)
        self.launches = 2 + 2 + 1
        self.desc = (f"interleave slot + kv_append (decode token) + paged_decode_attn over the "
                     f"{P} partitions in one launch ({splits} splits each) + lse_merge over the "
                     f"{P} partition results")

    def kernel(self):
        self.pkv.paged_decode_attn_partial(self.pq, self.k, self.v, self.ptab, self.plen,
                                           self.w.scale, self.splits, out_part=self.sp_out,
                                           lse_part=self.sp_lse)

    def run(self, ev_a=None, ev_b=None):
        p, w = self.pkv, self.w
        p.interleave_slot_mapping(self.k, self.v, self.N - 1, 1, self.P, w.interleave, self.ptab,
                                  out=self.slots)
        p.kv_append(self.k, self.v, self.k_new, self.v_new, self.slots)
        if ev_a is None:
            p.paged_decode_attn(self.pq, self.k, self.v, self.ptab, self.plen, w.scale,
                                num_splits=self.splits, workspace=self.ws, out=self.pout,
                                lse=self.plse)
        else:
            ev_a.record()
            self.kernel()
            ev_b.record()
            p.lse_merge(self.sp_out, self.sp_lse, out=self.pout, lse=self.plse)
        p.lse_merge(self.pout, self.plse, out=self.out[0], lse=self.lse[0])


class DcpE4m3Step(DcpStep):
    """The DCP step over an FP8 (E4M3) cache: the 200K tokens are quantised
    into their partitions by the E4M3 append, the partitions attended in one
    pkv_paged_decode_attn_e4m3 call and merged."""
    kernel_name = ("decode_gqa_tc_e4m3_kernel over the partitions (split attention, "
                   "pkv_paged_decode_attn_partial_e4m3, groups of 8)")

    def __init__(self, pkv, w, dev, splits):
        self.pkv, self.w, self.splits = pkv, w, splits
        self.k, self.v = w.k_codes.to(dev), w.v_codes.to(dev)
        self.k_scale, self.v_scale = w.k_scale.to(dev), w.v_scale.to(dev)
        self.q = w.q.to(dev)
        self.k_new, self.v_new = w.k_new.to(dev), w.v_new.to(dev)
        N, P = int(w.seq_lens[0]), w.num_parts
        self.ptab = w.part_tables.to(dev)
        kt, vt = w.k_tokens.to(dev), w.v_tokens.to(dev)
        pkv.kv_append_e4m3(self.k, self.v, kt[:N - 1], vt[:N - 1],
                           pkv.interleave_slot_mapping(self.k, self.v, 0, N - 1, P,
                                                       w.interleave, self.ptab),
                           self.k_scale, self.v_scale)
        del kt, vt
        self.N, self.P = N, P
        self.plen = torch.tensor([pkv.interleave_partition_len(N, P, w.interleave, r)
                                  for r in range(P)], dtype=torch.int32, device=dev)
        Hq, Dv = w.num_q_heads, w.head_dim_v
        self.pq = self.q.expand(P, Hq, w.head_dim_k).contiguous()
        self.pout = torch.empty(P, Hq, Dv, device=dev)
        self.plse = torch.empty(P, Hq, device=dev)
        self.out = torch.empty(1, Hq, Dv, device=dev)
        self.lse = torch.empty(1, Hq, device=dev)
        self.slots = torch.empty(1, dtype=torch.int64, device=dev)
        self.ws = torch.zeros(max(1, pkv.decode_workspace_size(P, Hq, Dv, splits)),
                              dtype=torch.uint8, device=dev)
        self.sp_out = torch.empty(splits, P, Hq, Dv, device=dev)
        self.sp_lse = torch.empty(splits, P, Hq, device=dev)
        self.launches = 2 + 2 + 1
        self.desc = (f"interleave slot + kv_append_e4m3 (decode token) + "
                     f"paged_decode_attn_e4m3 over the {P} partitions in one launch "
                     f"({splits} splits each, + its merge) + lse_merge over the {P} "
                     f"partition results")

    def kernel(self):
        self.pkv.paged_decode_attn_partial_e4m3(self.pq, self.k, self.v, self.k_scale,
                                                self.v_scale, self.ptab, self.plen, self.w.scale,
                                                self.splits, out_part=self.sp_out,
                                                lse_part=self.sp_lse)

    def run(self, ev_a=None, ev_b=None):
        p, w = self.pkv, self.w
        p.interleave_slot_mapping(self.k, self.v, self.N - 1, 1, self.P, w.interleave, self.ptab,
                                  out=self.slots)
        p.kv_append_e4m3(self.k, self.v, self.k_new, self.v_new, self.slots, self.k_scale,
                         self.v_scale)
        if ev_a is None:
            p.paged_decode_attn_e4m3(self.pq, self.k, self.v, self.k_scale, self.v_scale,
                                     self.ptab, self.plen, w.scale, num_splits=self.splits,
                                     workspace=self.ws, out=self.pout, lse=self.plse)
        else:
            ev_a.record()
            self.kernel()
            ev_b.record()
            p.lse_merge(self.sp_out, self.sp_lse, out=self.pout, lse=self.plse)
        p.lse_merge(self.pout, self.plse, out=self.out[0], lse=self.lse[0])


class AgentStep(Step):
    """Shared-prefix MLA-shaped step: copy-on-write of each sequence's shared
    tail, append of the decode tokens, attention (the suffixes are appended
    once, before timing)."""
    kernel_name = "decode_mla_tc_kernel (split attention, tcgen05 + TMEM)"
    bound = "tensor"

    def __init__(self, pkv, w, dev, splits):
        super().__init__(pkv, w, dev, splits)
        self.src, self.dst = w.cow_src.to(dev), w.cow_dst.to(dev)
        pkv.copy_blocks(self.k, self.v, self.src, self.dst)
        last = torch.zeros(w.new_seq.numel(), dtype=torch.bool)
        last[torch.cumsum(torch.bincount(w.new_seq.long()), 0) - 1] = True
        setup = ~last
        sl = pkv.slot_mapping(self.k, self.v, self.bt, self.new_seq[setup.to(dev)],
                              self.new_pos[setup.to(dev)])
        vs = None if self.v_new is None else self.v_new[setup.to(dev)]
        pkv.kv_append(self.k, self.v, self.k_new[setup.to(dev)], vs, sl)
        keep = last.to(dev)
        self.new_seq, self.new_pos = self.new_seq[keep], self.new_pos[keep]
        self.k_new = self.k_new[keep].contiguous()
        if self.v_new is not None:
            self.v_new = self.v_new[keep].contiguous()
        self.slots = torch.empty(self.new_pos.numel(), dtype=torch.int64, device=dev)
        self.launches = 5   # copy, slot, append, split, merge
        self.desc = (f"copy_blocks ({self.src.numel()} CoW pairs) + slot_mapping + kv_append "
                     f"({self.new_pos.numel()} decode tokens) + split attention ({splits} "
                     f"splits) + lse_merge")

    def run(self, ev_a=None, ev_b=None):
        self.pkv.copy_blocks(self.k, self.v, self.src, self.dst)
        super().run(ev_a, ev_b)


class AgentCascadeStep(AgentStep):
    """The shared-prefix step with the cascade: every sequence's 128 query
    rows over the 2,125 shared full blocks as one virtual sequence, each
    sequence over the rest of its table (copied tail block + suffix), both
    in one tcgen05 launch, then the merge of the two sets of partials."""
    kernel_name = ("pkv_paged_decode_attn_cascade (prep + decode_mla_tc_kernel over the prefix "
                   "and suffix problems in one launch + cascade merge)")
    bound = "tensor"

    def __init__(self, pkv, w, dev, splits):
        s1, s2 = splits
        super().__init__(pkv, w, dev, 1)
        full = w.info["prefix"] // w.block_size
        self.ptab = w.block_tables[0, :full].clone().to(dev)
        mb = w.block_tables.shape[1]
        self.s1, self.s2 = pkv.decode_cascade_splits(self.k, self.v, w.batch, w.num_q_heads, mb,
                                                     full, s1, s2)
        need = pkv.lib.pkv_decode_cascade_workspace_size(
            ctypes.byref(pkv.cache_desc(self.k, self.v)), w.batch, w.num_q_heads, mb, full,
            self.s1, self.s2)
        self.ws = torch.zeros(need, dtype=torch.uint8, device=dev)
        self.launches = 6   # copy, slot, append, prep, attention (both parts), merge
        self.desc = (f"copy_blocks ({self.src.numel()} CoW pairs) + slot_mapping + kv_append "
                     f"({self.new_pos.numel()} decode tokens) + paged_decode_attn_cascade "
                     f"({full} shared blocks: {self.s1} prefix splits over the "
                     f"{w.batch * w.num_q_heads} rows of all sequences, {self.s2} suffix "
                     f"splits; one attention launch) + merge")

    def kernel(self):
        """The cascade attention call (prep, one attention launch, merge)."""
        self.pkv.paged_decode_attn_cascade(self.q, self.k, self.v, self.ptab, self.bt, self.lens,
                                           self.w.scale, prefix_splits=self.s1,
                                           suffix_splits=self.s2, workspace=self.ws,
                                           out=self.out, lse=self.lse)

    def attend(self, ev_a=None, ev_b=None):
        if ev_a is not None:
            ev_a.record()
        self.kernel()
        if ev_b is not None:
            ev_b.record()


class MultiStep(Step):
    """Speculative verification: T new tokens per sequence appended, each
    attending causally to the cache (one pkv_paged_decode_attn_multi)."""
    kernel_name = ("pkv_paged_decode_attn_multi (decode_gqa_tc_kernel, tcgen05 + TMEM, with "
                   "4 heads x 4 tokens as the 16 rows of each work item, + lse_merge)")

    def __init__(self, pkv, w, dev, splits):
        super().__init__(pkv, w, dev, splits)
        B, T, Hq, Dv = w.batch, w.tokens_per_seq, w.num_q_heads, w.head_dim_v
        self.out = torch.empty(B, T, Hq, Dv, device=dev)
        self.lse = torch.empty(B, T, Hq, device=dev)
        need = pkv.lib.pkv_decode_multi_workspace_size(B, T, Hq, Dv, w.max_blocks, splits)
        self.ws = torch.zeros(need, dtype=torch.uint8, device=dev)
        self.launches = 4   # slot, append, split (T tokens as rows of an item), merge
        self.desc = (f"slot_mapping + kv_append ({w.new_pos.numel()} new tokens, {T} per "
                     f"sequence) + paged_decode_attn_multi ({splits} splits) = split kernel "
                     f"with the {T} tokens as rows of each work item + lse_merge")

    def kernel(self):
        """The multi-token attention call (its split kernel and merge)."""
        self.pkv.paged_decode_attn_multi(self.q, self.k, self.v, self.bt, self.lens,
                                         self.w.scale, num_splits=self.splits,
                                         workspace=self.ws, out=self.out, lse=self.lse)

    def attend(self, ev_a=None, ev_b=None):
        if ev_a is not None:
            ev_a.record()
        self.kernel()
        if ev_b is not None:
            ev_b.record()


class E4m3Step(Step):
    """The 32K decode step over an FP8 (E4M3) cache: slot mapping, the
    quantising append of the decode tokens, one pkv_paged_decode_attn_e4m3."""
    kernel_name = ("decode_gqa_tc_e4m3_kernel (split attention, "
                   "pkv_paged_decode_attn_partial_e4m3: tcgen05 kind::f8f6f4, E4M3 K/V as "
                   "stored, the query as 4 and the probabilities as 5 E4M3 terms)")

    def __init__(self, pkv, w, dev, splits):
        self.pkv, self.w, self.splits = pkv, w, splits
        self.k, self.v = w.k_codes.to(dev), w.v_codes.to(dev)
        self.k_scale, self.v_scale = w.k_scale.to(dev), w.v_scale.to(dev)
        self.bt, self.lens, self.q = w.block_tables.to(dev), w.seq_lens.to(dev), w.q.to(dev)
        self.new_seq, self.new_pos = w.new_seq.to(dev), w.new_pos.to(dev)
        self.k_new, self.v_new = w.k_new.to(dev), w.v_new.to(dev)
        B, Hq = w.batch, w.num_q_heads
        self.slots = torch.empty(w.new_pos.numel(), dtype=torch.int64, device=dev)
        self.out = torch.empty(B, Hq, w.head_dim_v, device=dev)
        self.lse = torch.empty(B, Hq, device=dev)
        self.ws = torch.zeros(max(1, pkv.decode_workspace_size(B, Hq, w.head_dim_v, splits)),
                              dtype=torch.uint8, device=dev)
        self.out_part = torch.empty(splits, B, Hq, w.head_dim_v, device=dev)
        self.lse_part = torch.empty(splits, B, Hq, device=dev)
        self.launches = 4   # slot, append, split, merge
        self.desc = (f"slot_mapping + kv_append_e4m3 ({w.new_pos.numel()} decode tokens) + "
                     f"paged_decode_attn_e4m3 ({splits} splits) = split kernel + lse_merge")

    def kernel(self):
        """The FP8 split attention kernel alone (the roofline's kernel)."""
        self.pkv.paged_decode_attn_partial_e4m3(self.q, self.k, self.v, self.k_scale,
                                                self.v_scale, self.bt, self.lens, self.w.scale,
                                                self.splits, out_part=self.out_part,
                                                lse_part=self.lse_part)

    def attend(self, ev_a=None, ev_b=None):
        """What pkv_paged_decode_attn_e4m3 launches: the split kernel, then the
        merge (events, if given, bracket the split kernel)."""
        if self.splits == 1 or ev_a is None:
            if ev_a is not None:
                ev_a.record()
            self.pkv.paged_decode_attn_e4m3(self.q, self.k, self.v, self.k_scale, self.v_scale,
                                            self.bt, self.lens, self.w.scale,
                                            num_splits=self.splits, workspace=self.ws,
                                            out=self.out, lse=self.lse)
            if ev_b is not None:
                ev_b.record()
            return
        ev_a.record()
        self.kernel()
        ev_b.record()
        self.pkv.lse_merge(self.out_part, self.lse_part, out=self.out, lse=self.lse)

    def run(self, ev_a=None, ev_b=None):
        p = self.pkv
        p.slot_mapping(self.k, self.v, self.bt, self.new_seq, self.new_pos, out=self.slots)
        p.kv_append_e4m3(self.k, self.v, self.k_new, self.v_new, self.slots, self.k_scale,
                         self.v_scale)
        self.attend(ev_a, ev_b)


class AgentE4m3Step(E4m3Step):
    """The shared-prefix MLA step over an FP8 (E4M3) cache: copy-on-write of
    each sequence's shared tail block (its codes), the quantising append of
    the decode tokens, one pkv_paged_decode_attn_e4m3 (the suffixes are
    appended once, before timing)."""
    kernel_name = ("decode_mla_tc_kernel, E4M3 mode (split attention, "
                   "pkv_paged_decode_attn_partial_e4m3: codes expanded exactly to fp16 in shared "
                   "memory, tcgen05 kind::f16)")
    bound = "tensor"

    def __init__(self, pkv, w, dev, splits):
        super().__init__(pkv, w, dev, splits)
        self.src, self.dst = w.cow_src.to(dev), w.cow_dst.to(dev)
        pkv.copy_blocks_e4m3(self.k, self.v, self.src, self.dst)
        last = torch.zeros(w.new_seq.numel(), dtype=torch.bool)
        last[torch.cumsum(torch.bincount(w.new_seq.long()), 0) - 1] = True
        setup = (~last).to(dev)
        sl = pkv.slot_mapping(self.k, self.v, self.bt, self.new_seq[setup], self.new_pos[setup])
        pkv.kv_append_e4m3(self.k, self.v, self.k_new[setup], self.v_new[setup], sl,
                           self.k_scale, self.v_scale)
        keep = last.to(dev)
        self.new_seq, self.new_pos = self.new_seq[keep], self.new_pos[keep]
        self.k_new = self.k_new[keep].contiguous()
        self.v_new = self.v_new[keep].contiguous()
        self.slots = torch.empty(self.new_pos.numel(), dtype=torch.int64, device=dev)
        self.launches = 5   # copy, slot, append, split, merge
        self.desc = (f"copy_blocks ({self.src.numel()} CoW pairs) + slot_mapping + "
                     f"kv_append_e4m3 ({self.new_pos.numel()} decode tokens) + "
                     f"paged_decode_attn_e4m3 ({splits} splits) = split kernel + lse_merge")

    def run(self, ev_a=None, ev_b=None):
        self.pkv.copy_blocks_e4m3(self.k, self.v, self.src, self.dst)
        super().run(ev_a, ev_b)


class MultiE4m3Step(E4m3Step):
    """Speculative verification over an FP8 (E4M3) cache: T new tokens per
    sequence quantised into the cache, each attending causally (one
    pkv_paged_decode_attn_multi_e4m3)."""
    kernel_name = ("pkv_paged_decode_attn_multi_e4m3 (decode_gqa_tc_e4m3_kernel with 4 heads x "
                   "4 tokens as the 16 rows of each work item, + lse_merge)")

    def __init__(self, pkv, w, dev, splits):
        super().__init__(pkv, w, dev, splits)
        B, T, Hq, Dv = w.batch, w.tokens_per_seq, w.num_q_heads, w.head_dim_v
        self.out = torch.empty(B, T, Hq, Dv, device=dev)
        self.lse = torch.empty(B, T, Hq, device=dev)
        need = pkv.lib.pkv_decode_multi_workspace_size(B, T, Hq, Dv, w.max_blocks, splits)
        self.ws = torch.zeros(need, dtype=torch.uint8, device=dev)
        self.desc = (f"slot_mapping + kv_append_e4m3 ({w.new_pos.numel()} new tokens, {T} per "
                     f"sequence) + paged_decode_attn_multi_e4m3 ({splits} splits) = split "
                     f"kernel with the {T} tokens as rows of each work item + lse_merge")

    def kernel(self):
        """The FP8 multi-token attention call (its split kernel and merge)."""
        self.pkv.paged_decode_attn_multi_e4m3(self.q, self.k, self.v, self.k_scale,
                                              self.v_scale, self.bt, self.lens, self.w.scale,
                                              num_splits=self.splits, workspace=self.ws,
                                              out=self.out, lse=self.lse)

    def attend(self, ev_a=None, ev_b=None):
        if ev_a is not None:
            ev_a.record()
        self.kernel()
        if ev_b is not None:
            ev_b.record()


STEPS = {"long32k": Step, "mix": Step, "tiny": Step, "dcp200k": DcpStep, "agent_mla": AgentStep,
         "agent_mla_latent": AgentStep, "agent_mla_cascade": AgentCascadeStep,
         "spec4_32k": MultiStep, "long32k_e4m3": E4m3Step, "dcp200k_e4m3": DcpE4m3Step,
         "spec4_32k_e4m3": MultiE4m3Step, "agent_mla_e4m3": AgentE4m3Step}
# The 32K workload is timed at 16 splits, the split count its configuration
# names; the split count the library picks by itself (num_splits = 0) is
# timed too and reported beside it (`library_auto_splits`).
DEFAULT_SPLITS = {"long32k": 16, "mix": 1, "tiny": 1, "dcp200k": 19, "agent_mla": 19,
                  "agent_mla_latent": 19, "agent_mla_cascade": (19, 2), "spec4_32k": 9,
                  "long32k_e4m3": 7, "dcp200k_e4m3": 14, "spec4_32k_e4m3": 9,
                  "agent_mla_e4m3": 19}
# Workloads whose line also carries the library's own split choice.
AUTO_SPLITS_ALSO = ("long32k",)
# Workloads of the single-threaded oracle figure (the four GQA configurations)
# and the tokens per sequence of its sample (None = every token).
SINGLE_THREAD_SAMPLE = {"tiny": None, "mix": None, "long32k": 8192, "dcp200k": 32768}


# ------------------------------------------------------------------ arms

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def oracle_gbs(w, tokens: int | None, repeats: int = 1, num_threads: int = 0):
    """Time the CPU oracle over every row of `w`, restricted to the first
    `tokens` tokens of each sequence when given; `num_threads` 0 = all host
    cores."""
    import oracle
    q, bt, lens = w.q.numpy(), w.block_tables.numpy(), w.seq_lens.numpy()
    if w.k_codes is not None:
        kp, vp = w.k_codes.numpy(), w.v_codes.numpy()
    else:
        kp = bits_view(w.k_pool)
        vp = (np.ascontiguousarray(kp[..., :w.head_dim_v]) if w.v_pool is None
              else bits_view(w.v_pool))
    end = None
    if tokens is not None:
        end = np.minimum(lens, tokens).astype(np.int32)
    used = int((end if end is not None else lens).astype(np.int64).sum()) * kv_bytes_per_token(w)
    times = []
    for _ in range(repeats):
        t = time.perf_counter()
        if w.k_codes is not None and w.tokens_per_seq > 1:
            # each (sequence, token) as a row seeing the sample's tokens up to its own
            T, B = w.tokens_per_seq, q.shape[0]
            L = (lens if end is None else end).astype(np.int64)
            rl = np.array([max(0, L[b] - T + 1 + i) for b in range(B) for i in range(T)],
                          dtype=np.int32)
            oracle.paged_decode_attn_e4m3(q.reshape(B * T, *q.shape[2:]), kp, vp,
                                          w.k_scale.numpy(), w.v_scale.numpy(),
                                          np.repeat(bt, T, axis=0), rl, w.scale,
                                          num_threads=num_threads)
        elif w.k_codes is not None:
            oracle.paged_decode_attn_e4m3(q, kp, vp, w.k_scale.numpy(), w.v_scale.numpy(), bt,
                                          lens, w.scale, tok_end=end, num_threads=num_threads)
        elif w.tokens_per_seq > 1:
            # the same step on each sequence's first tokens: query t sees the
            # sample's tokens up to its own
            oracle.paged_decode_attn_multi(q, kp, vp, bt, lens if end is None else end, w.scale,
                                           num_threads=num_threads)
        else:
            oracle.paged_decode_attn(q, kp, vp, bt, lens, w.scale, tok_end=end,
                                     num_threads=num_threads)
        times.append(time.perf_counter() - t)
    return used, times


def workload_splits(args):
    """The split count of the workload (a (prefix, suffix) pair for the
    cascade), --splits / --suffix-splits overriding the defaults."""
    d = DEFAULT_SPLITS[args.workload]
    if isinstance(d, tuple):
        return (args.splits or d[0], args.suffix_splits or d[1])
    return args.splits or d


def workload_desc(w, splits):
    kv = (f"head_dim {w.head_dim_k}, values = first {w.head_dim_v} dims of each key row, bf16"
          if w.v_pool is None else
          f"head_dim {w.head_dim_k}, E4M3 K/V with fp32 scales per KV head"
          if w.k_codes is not None else f"head_dim {w.head_dim_k}, bf16 K/V")
    return (f"{w.name}: batch {w.batch} x {int(w.seq_lens.max())} tokens, GQA "
            f"{w.num_q_heads}/{w.num_kv_heads} heads, {kv}, block "
            f"{w.block_size}, {w.num_blocks}-block randomly permuted pool, " +
            (f"cascade: {splits[0]} prefix + {splits[1]} suffix splits + merge"
             if isinstance(splits, tuple) else f"{splits} splits + lse_merge"))


def run_reference(args, world, rank):
    if rank != 0:
        return
    w = workloads.make(args.workload)
    cores = os.cpu_count()
    # Size the per-step sample so that warm-up + timed steps stay near a minute.
    probe_tokens = 512
    used, t = oracle_gbs(w, probe_tokens)
    per_token_s = t[0] / probe_tokens
    budget = 60.0 / max(1, args.steps + args.warmup)
    tokens = int(max(64, min(int(w.seq_lens.max()), budget / max(per_token_s, 1e-9))))
    for _ in range(args.warmup):
        oracle_gbs(w, tokens)
    times = []
    t0 = time.perf_counter()
    for _ in range(args.steps):
        used, tt = oracle_gbs(w, tokens)
        times.append(tt[0])
    wall = time.perf_counter() - t0
    gbs = used * args.steps / sum(times) / 1e9
    sample = (f"every (sequence, query head) row of {args.workload}, first {tokens} of "
              f"{int(w.seq_lens.max())} tokens per sequence, per step")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * wall / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload_desc(w, workload_splits(args)),
                   "oracle": "C, fp64, all host cores"},
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": cores,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }))


def staged(dev, tensors):
    """One pinned host buffer holding `tensors` (256-byte aligned segments),
    one device buffer of the same layout, and device views of each segment."""
    offs, at = {}, 0
    for n, t in tensors.items():
        offs[n] = at
        at += (t.numel() * t.element_size() + 255) // 256 * 256
    host = torch.empty(max(at, 1), dtype=torch.uint8).pin_memory()
    devb = torch.empty(max(at, 1), dtype=torch.uint8, device=dev)
    views = {}
    for n, t in tensors.items():
        nb = t.numel() * t.element_size()
        host[offs[n]:offs[n] + nb].view(t.dtype).copy_(t.contiguous().view(-1))
        views[n] = devb[offs[n]:offs[n] + nb].view(t.dtype).view(t.shape)
    return host, devb, views


def _events(n):
    return [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in range(n)]


def _stats(ms_list):
    return {"mean": round(statistics.fmean(ms_list), 5),
            "median": round(statistics.median(ms_list), 5), "min": round(min(ms_list), 5),
            "n": len(ms_list)}


def time_step(pkv, st, args, world, stream, sampler=None):
    """Warm-up, then K steps replayed from a CUDA graph (the headline timing),
    then the same K steps one by one with CUDA events around every step and
    around its split attention kernel, then the split kernel alone back to
    back.  Returns the figures as a dict (times in ms, max over ranks)."""
    for _ in range(args.warmup):
        st.run()
    torch.cuda.synchronize()
    if pkv.device_status(reset=True) != 0:
        raise RuntimeError("device status word set during warm-up")

    # Steps captured in a CUDA graph (the library's calls allocate nothing
    # and never synchronise with the host, so they capture as they are); the
    # timed steps replay it, as a serving loop replays its decode step.
    graph = None
    per_graph = max(1, args.graph_steps)
    if not args.eager:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for _ in range(per_graph):
                st.run()
        for _ in range(3):
            graph.replay()
        torch.cuda.synchronize()

    # eager steps (the calls made one by one from Python), for context
    ke = min(args.steps, 500)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(ke):
        st.run()
    e1.record(stream)
    torch.cuda.synchronize()
    eager_ms = max_over_ranks(e0.elapsed_time(e1) / ke, world)

    # ---- timed region: K steps back to back, events only at its two ends
    K = args.steps
    ev_start = torch.cuda.Event(enable_timing=True)
    ev_end = torch.cuda.Event(enable_timing=True)
    if sampler:
        sampler.wait_ready()
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.time()
    ev_start.record(stream)
    if graph is not None:
        for _ in range(K // per_graph):
            graph.replay()
        for _ in range(K % per_graph):
            st.run()
    else:
        for _ in range(K):
            st.run()
    ev_end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    t1 = time.time()
    clocks = sampler.summary(t0, t1) if sampler else None
    if sampler:
        sampler.stop()
    if pkv.device_status(reset=True) != 0:
        raise RuntimeError("device status word set during the timed steps")
    ms = max_over_ranks(ev_start.elapsed_time(ev_end) / K, world)

    # ---- the same K steps again, one by one, with events around every step
    # and around its split attention kernel (the kernel's average launch
    # duration is the roofline's; the step events give the per-step spread)
    ev_k, ev_s = _events(K), _events(K)
    barrier(world)
    torch.cuda.synchronize()
    # In batches of 64 steps, each behind a spin of the GPU (~0.3 ms of
    # clock cycles per step) during which the host enqueues the batch: the
    # steps of a batch then run back to back and no event bracket holds a
    # wait for the host's next launch (a short step's calls can take the
    # host longer than the GPU; a batch stays within the launch queue).
    spin = getattr(torch.cuda, "_sleep", None)   # torch's spin kernel (clock cycles)
    for i0 in range(0, K, 64):
        n = min(64, K - i0)
        if spin is not None:
            spin(int(n * 0.3e-3 * 2.0e9))
        for i in range(i0, i0 + n):
            ev_s[i][0].record(stream)
            st.run(*ev_k[i])
            ev_s[i][1].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    kern = [a.elapsed_time(b) for a, b in ev_k]
    steps = [a.elapsed_time(b) for a, b in ev_s]
    kms = max_over_ranks(statistics.fmean(kern), world)

    # ---- the split kernel alone, launched back to back (context only)
    torch.cuda.synchronize()
    a_ev, b_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    kb = min(K, 200)
    a_ev.record(stream)
    for _ in range(kb):
        st.kernel()
    b_ev.record(stream)
    torch.cuda.synchronize()
    kms_b2b = a_ev.elapsed_time(b_ev) / kb
    if pkv.device_status(reset=True) != 0:
        raise RuntimeError("device status word set")
    return {"ms": ms, "kms": kms, "kms_b2b": kms_b2b, "eager_ms": eager_ms, "eager_steps": ke,
            "graph": graph is not None, "per_graph": per_graph, "clocks": clocks,
            "step_events": _stats(steps), "kernel_events": _stats(kern)}


def time_cold_l2(pkv, st, reps, stream):
    """One step captured in a CUDA graph, replayed `reps` times, each replay
    preceded by a read of a 256 MiB buffer that evicts the 129 MB L2 (a read
    leaves no dirty lines to write back during the step) and bracketed by
    CUDA events: the step with nothing of its data in L2."""
    flush = torch.empty(64 << 20, dtype=torch.float32, device=st.q.device).fill_(1.0)
    sink = torch.empty((), dtype=torch.float32, device=st.q.device)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        st.run()
    g.replay()
    torch.cuda.synchronize()
    ev = _events(reps)
    for a, b in ev:
        torch.sum(flush, dim=0, out=sink)
        a.record(stream)
        g.replay()
        b.record(stream)
    torch.cuda.synchronize()
    if pkv.device_status(reset=True) != 0:
        raise RuntimeError("device status word set during the cold-L2 steps")
    del flush
    return _stats([a.elapsed_time(b) for a, b in ev])


def run_gpu(args, world, rank, local):
    import paged_kv_cache_93_gb300 as pkv
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = workloads.make(args.workload)
    splits = workload_splits(args)
    st = STEPS[args.workload](pkv, w, dev, splits)
    total_bytes, kernel_bytes = step_bytes(w, splits)
    stream = torch.cuda.current_stream()
    K = args.steps

    sampler = ClockSampler(local) if rank == 0 else None
    tm = time_step(pkv, st, args, world, stream, sampler)
    ms, kms, kms_b2b, clocks = tm["ms"], tm["kms"], tm["kms_b2b"], tm["clocks"]
    eager_ms, ke, per_graph = tm["eager_ms"], tm["eager_steps"], tm["per_graph"]
    graph = tm["graph"] or None
    cold = time_cold_l2(pkv, st, min(K, 200), stream)

    # ---- the same step at the library's own split choice (num_splits = 0)
    auto = None
    if args.workload in AUTO_SPLITS_ALSO and not args.splits:
        s_auto = pkv.decode_auto_splits(st.k, st.v, w.batch, w.num_q_heads,
                                        w.block_tables.shape[1] * w.block_size)
        st_a = STEPS[args.workload](pkv, w, dev, s_auto)
        ta = time_step(pkv, st_a, args, world, stream)
        tb, kb_ = step_bytes(w, s_auto)
        auto = {"num_splits": s_auto, "ms_per_step": round(ta["ms"], 5),
                "value": round(world * tb / (ta["ms"] * 1e-3) / 1e9, 2),
                "launch_ms": round(ta["kms"], 5),
                "kernel_gbs": round(kb_ / (ta["kms"] * 1e-3) / 1e9, 2),
                "ms_per_step_events": ta["step_events"]}
        del st_a

    value = world * total_bytes / (ms * 1e-3) / 1e9
    peak, peak_kind = load_peak()
    kernel_gbs = kernel_bytes / (kms * 1e-3) / 1e9
    if auto is not None:
        auto["frac"] = round(auto["kernel_gbs"] / peak, 4)
    if getattr(st, "bound", "hbm") == "tensor":
        # a math-bound launch inside seconds of back-to-back steps: the
        # sustained bf16 tensor throughput is the denominator
        tpeak, tkind = load_peak("bf16_tflops_sustained", FALLBACK_BF16_TFLOPS_SUSTAINED)
        flops = kernel_flops(w)
        tflops = flops / (kms * 1e-3) / 1e12
        roofline = {"bound": "tensor", "achieved": round(tflops, 2), "peak": tpeak,
                    "unit": "TFLOP/s", "frac": round(tflops / tpeak, 4), "traffic": None,
                    "algorithmic_flops_per_launch": flops,
                    "hbm_gbs_on_unique_bytes": round(kernel_gbs, 2),
                    "peak_kind": f"{tkind} bf16_tflops_sustained (MEASURED_PEAKS.json cuBLAS "
                                 f"bf16 GEMM, seconds-long loop)"}
    else:
        roofline = {"bound": "hbm", "achieved": round(kernel_gbs, 2), "peak": peak,
                    "unit": "GB/s", "frac": round(kernel_gbs / peak, 4), "traffic": None,
                    "algorithmic_bytes_per_launch": kernel_bytes,
                    "peak_kind": f"{peak_kind} hbm_gbs (MEASURED_PEAKS.json copy bandwidth)"}

    # ---- end to end through the public API, host buffers in pinned memory
    e2e = None
    if args.workload in ("long32k", "mix", "tiny"):
        # A serving loop's decode step through the public API: the step's
        # inputs staged in one pinned buffer (one copy in) and its outputs in
        # one device buffer (one copy out).  Two sets of buffers and a copy
        # stream: step i+1's inputs go in while step i computes, and step i's
        # results come back while step i+1 runs; events keep every buffer from
        # being reused before its copy or its step is done.
        names = ("q", "block_tables", "seq_lens", "new_seq", "new_pos", "k_new", "v_new")
        sets = []
        for _ in range(2):
            h_in, d_in, d = staged(dev, {n: getattr(w, n) for n in names})
            h_res, d_res, r = staged(dev, {"out": torch.empty(w.batch, w.num_q_heads,
                                                              w.head_dim_v),
                                           "lse": torch.empty(w.batch, w.num_q_heads)})
            ev = {k: torch.cuda.Event() for k in ("in", "done", "out")}
            sets.append((h_in, d_in, d, h_res, d_res, r, ev))
        ws = torch.zeros(max(1, pkv.decode_workspace_size(w.batch, w.num_q_heads, w.head_dim_v,
                                                          splits)), dtype=torch.uint8,
                         device=dev)
        h2d = sets[0][0].numel()
        d2h = sets[0][3].numel()
        d_slots = torch.empty(w.new_pos.numel(), dtype=torch.int64, device=dev)
        copy_stream = torch.cuda.Stream(device=dev)
        ke = max(per_graph, min(K, 400))

        def run_steps(n):
            """n pipelined steps.  The copy stream forks from the current
            stream at the start and joins it at the end, and only events
            recorded within the run are waited on, so a run also captures
            into a CUDA graph."""
            comp = torch.cuda.current_stream()
            seen = set()

            def wait(stream, i, key):
                if (i % 2, key) in seen:
                    stream.wait_event(sets[i % 2][6][key])

            def record(stream, i, key):
                sets[i % 2][6][key].record(stream)
                seen.add((i % 2, key))

            fork = torch.cuda.Event()
            fork.record(comp)
            copy_stream.wait_event(fork)

            def stage_in(i):
                h_in, d_in = sets[i % 2][0], sets[i % 2][1]
                with torch.cuda.stream(copy_stream):
                    wait(copy_stream, i, "done")            # step i-2 has read this set
                    d_in.copy_(h_in, non_blocking=True)
                    record(copy_stream, i, "in")

            stage_in(0)
            for i in range(n):
                _, _, d, h_res, d_res, r, ev = sets[i % 2]
                if i + 1 < n:
                    stage_in(i + 1)
                wait(comp, i, "in")
                wait(comp, i, "out")                        # step i-2's results are home
                pkv.slot_mapping(st.k, st.v, d["block_tables"], d["new_seq"], d["new_pos"],
                                 out=d_slots)
                pkv.kv_append(st.k, st.v, d["k_new"], d["v_new"], d_slots)
                pkv.paged_decode_attn(d["q"], st.k, st.v, d["block_tables"], d["seq_lens"],
                                      w.scale, num_splits=splits, workspace=ws, out=r["out"],
                                      lse=r["lse"])
                record(comp, i, "done")
                with torch.cuda.stream(copy_stream):
                    wait(copy_stream, i, "done")
                    h_res.copy_(d_res, non_blocking=True)
                    record(copy_stream, i, "out")
            for j in range(min(n, 2)):                      # join: every result is home
                wait(comp, n - 1 - j, "out")

        run_steps(3)
        e_graph = None
        if graph is not None:
            e_graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(e_graph):
                run_steps(per_graph)
            e_graph.replay()
        ke = ke // per_graph * per_graph if e_graph is not None else ke
        torch.cuda.synchronize()
        barrier(world)
        te = time.perf_counter()
        if e_graph is not None:
            for _ in range(ke // per_graph):
                e_graph.replay()
        else:
            run_steps(ke)
        torch.cuda.synchronize()
        e2e_s = max_over_ranks((time.perf_counter() - te) / ke, world)
        barrier(world)
        # the last step's results came home intact
        _, _, _, h_res, d_res, _, _ = sets[(ke - 1) % 2]
        if not torch.equal(h_res, d_res.cpu()):
            raise RuntimeError("end-to-end results differ between device and host buffers")
        e2e = {"value": round(total_bytes / e2e_s / 1e9 * world, 2), "unit": "GB/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": round(e2e_s * 1e3, 4), "steps": ke,
               "api": "pinned host inputs (one staging buffer, one copy per step) -> "
                      "slot_mapping + kv_append + paged_decode_attn -> pinned host out/lse "
                      "(one copy per step); two buffer sets and a copy stream overlap each "
                      "step's copies with the neighbouring steps' compute; " +
                      (f"{per_graph} such steps captured in a CUDA graph and replayed"
                       if e_graph is not None else "calls made one by one from Python") +
                      "; wall clock"}
    if pkv.device_status(reset=True) != 0:
        raise RuntimeError("device status word set")

    if rank != 0:
        return

    # ---- CPU baseline: the oracle on this host's cores (all of them, and one)
    tokens = None if (args.workload in ("long32k", "mix", "tiny") and not args.quick_cpu) else 2048
    used, times = oracle_gbs(w, tokens, repeats=1)
    cpu_gbs = used / min(times) / 1e9
    single = None
    if args.workload in SINGLE_THREAD_SAMPLE:
        t1_tokens = SINGLE_THREAD_SAMPLE[args.workload]
        if args.quick_cpu and t1_tokens is not None:
            t1_tokens = min(t1_tokens, 2048)
        used1, times1 = oracle_gbs(w, t1_tokens, repeats=1, num_threads=1)
        single = {"value": round(used1 / min(times1) / 1e9, 4), "unit": "GB/s", "cores": 1,
                  "kind": "oracle",
                  "sample": ("whole workload (every row, every token)" if t1_tokens is None else
                             f"every row, first {t1_tokens} tokens of each sequence") +
                            ", C fp64 oracle, one thread"}
    traffic = stored_traffic(args.workload)
    seq_tokens = int(w.seq_lens.sum())
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": round(ms, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3" if w.k_codes is not None else "bf16",
        "data": "synthetic",
        "config": {
            "workload": workload_desc(w, splits), "batch": w.batch,
            "context": int(w.seq_lens.max()), "num_q_heads": w.num_q_heads,
            "num_kv_heads": w.num_kv_heads, "head_dim_k": w.head_dim_k,
            "head_dim_v": w.head_dim_v, "block_size": w.block_size, "num_splits": splits,
            "step": st.desc,
            "launch": (f"CUDA graph of {per_graph} steps (captured once, replayed)"
                       if graph is not None else "calls made one by one from Python"),
            "l2": f"no flush: the {total_bytes / 1e9:.3f} GB a step reads exceeds the 129 MB "
                  f"L2 (steps back to back)",
            "parallelism": "replicas" if world > 1 else "single GPU",
            "compute": ("E4M3 codes expanded exactly to fp16 in shared memory, fp16 "
                        "tensor-core products (the fp32 query and probabilities split into "
                        "fp16 hi+lo), fp32 accumulate and softmax"
                        if w.k_codes is not None and w.num_q_heads // w.num_kv_heads >= 64 else
                        "E4M3 tensor-core products (K/V as stored; the fp32 query as 4 and the "
                        "probabilities as 5 E4M3 terms), fp32 accumulate and softmax"
                        if w.k_codes is not None else
                        "bf16 tensor-core products (fp32 query and probabilities split into bf16 "
                        "hi+lo), fp32 accumulate and softmax"),
            "bytes": "unique K/V bytes (shared blocks once) + q + tables + appends + out/lse",
        },
        "pct_of_peak": round(100 * value / world / peak, 2),
        "seq_tokens_per_s": round(world * seq_tokens / (ms * 1e-3), 1),
        "decode_steps_per_s": round(world * 1e3 / ms, 2),
        "roofline": dict(roofline, traffic=traffic, kernel=st.kernel_name,
                         launch_ms=round(kms, 5), launch_ms_back_to_back=round(kms_b2b, 5)),
        "cpu_baseline": {
            "value": round(cpu_gbs, 4), "unit": "GB/s", "cores": os.cpu_count(),
            "kind": "oracle",
            "sample": ("whole workload (every row, every token)" if tokens is None else
                       f"every row, first {tokens} tokens of each sequence") +
                      ", C fp64 oracle, all host cores",
            "single_thread": single,
        },
        "e2e": e2e,
        "ms_per_step_events": dict(
            tm["step_events"],
            how="CUDA events around every step, the step's calls made one by one"),
        "kernel_launch_ms_events": tm["kernel_events"],
        "cold_l2": dict(cold, value=round(world * total_bytes / (cold["median"] * 1e-3) / 1e9, 2),
                        how="one step replayed from a CUDA graph, each repetition after a "
                            "read of a 256 MiB buffer that evicts the 129 MB L2; CUDA events "
                            "around the step; value at the median"),
        "library_auto_splits": auto,
        "eager": {"ms_per_step": round(eager_ms, 5),
                  "value": round(world * total_bytes / (eager_ms * 1e-3) / 1e9, 2),
                  "steps": tm["eager_steps"]},
        "gpu_launches": st.launches * K,
        "clocks": clocks,
    }
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--workload", default="long32k", choices=sorted(STEPS))
    ap.add_argument("--splits", type=int, default=0, help="0 = the workload's default")
    ap.add_argument("--suffix-splits", type=int, default=0,
                    help="cascade workload: suffix split count (0 = the default)")
    ap.add_argument("--quick-cpu", action="store_true", help="smaller oracle sample")
    ap.add_argument("--eager", action="store_true",
                    help="time the calls made one by one instead of a CUDA-graph replay")
    ap.add_argument("--graph-steps", type=int, default=16,
                    help="steps captured in one CUDA graph")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_gpu(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
