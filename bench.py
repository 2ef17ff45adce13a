#!/usr/bin/env python
"""Benchmark of one paged decode step on GB300 (and of the oracle on the host cores).

Default workload: the Llama-3-8B-shaped layer (32 q / 8 kv heads, head_dim 128, bf16
cache, block 16, batch 64, context ~ U[512, 4096], pool 1.2x the blocks needed).
One step = kv_append of each sequence's new token + paged decode attention over the
whole cache (plan, attention and split-reduce kernels).  The printed line carries:

* value: KV-cache GB/s = algorithmic bytes of the step / device time of the step
  (CUDA events on the launch stream; inputs resident in HBM; every step reads 613 MB
  of K/V, 4.8x the 129 MB L2; steps smaller than 4x L2 get an L2 flush between them);
* e2e: the same metric through the public API with pinned host buffers, the
  host-to-device copies of the step's inputs and the device-to-host copy of the
  output inside the timed region;
* roofline: the attention call alone against the measured HBM copy bandwidth;
* cpu_baseline: the fp64 oracle on a bounded sample of the workload on host cores;
* by_config: the other workloads (70B-shaped with a shared prefix, MQA / MHA, RoPE
  shift of reused chunks, long-context INT4 cache), same method, fewer steps.

--impl reference times the oracle instead (each step a bounded sample).
Multi-GPU (torchrun): every rank runs its own replica of the workload (weak scaling,
no collective on the data path); the step time is the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import resource
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

L2_BYTES = 129 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0
METRIC = "paged GQA decode attn: KV-cache HBM GB/s (% of peak) and sequences/s"


# Batches above this many sequences get the library's one-CTA plan kernel before the
# attention kernel (smaller ones plan inside the attention kernel).
PLAN_KERNEL_ABOVE = 256

# ---------------------------------------------------------------------------------------------
# algorithmic bytes
def attended_blocks(w: workloads.Workload, s: int):
    """(logical block, attended rows) of sequence s: the blocks from the one its attention
    window starts in (block 0 without a window), with the rows of each that are attended."""
    c = int(w.context_lens[s])
    t0 = max(0, c - w.window) if w.window > 0 else 0
    out = []
    for i in range(t0 // w.block_size, -(-c // w.block_size)):
        lo, hi = max(t0, i * w.block_size), min(c, (i + 1) * w.block_size)
        out.append((i, hi - lo))
    return out


def kv_token_rows(w: workloads.Workload) -> int:
    """Unique (physical block, row) pairs the step must read (shared prefix blocks once)."""
    need = {}
    for s in range(w.batch):
        for i, rows in attended_blocks(w, s):
            p = int(w.block_tables[s, i])
            need[p] = max(need.get(p, 0), rows)
    return sum(need.values())


def logical_token_rows(w) -> int:
    return int(np.sum(w.context_lens))


def attention_bytes(w, int4=False) -> int:
    rows = kv_token_rows(w)
    if int4:
        # codes (K and V, half a byte per value) + V (scale, min) per token + K (scale, min)
        # per channel per full block + the bf16 K tail of each unfinished block
        full_blocks = {}
        tail_rows = 0
        for s in range(w.batch):
            c = int(w.context_lens[s])
            for i, _ in attended_blocks(w, s):
                if (i + 1) * w.block_size <= c:
                    full_blocks[int(w.block_tables[s, i])] = 1
            tail_rows += c % w.block_size
        kv = (rows * w.n_kv * w.head_dim + rows * w.n_kv * 4 + len(full_blocks) * w.n_kv * w.head_dim * 4
              + tail_rows * w.n_kv * w.head_dim * 2)
    else:
        kv = rows * w.n_kv * w.head_dim * 2 * 2
    q = w.batch * w.n_h * w.head_dim * 2
    out = w.batch * w.n_h * w.head_dim * 2
    tables = sum(len(attended_blocks(w, s)) for s in range(w.batch)) * 4
    return kv + q + out + tables + w.batch * 4


def append_bytes(w, int4=False) -> int:
    if int4:   # read k, v; write V codes + meta per token (K blocks that complete are rare)
        return w.batch * w.n_kv * (w.head_dim * 4 + w.head_dim // 2 + 4 + w.head_dim * 2) + w.batch * 12
    return w.batch * w.n_kv * w.head_dim * 2 * 2 * 2 + w.batch * 8


# ---------------------------------------------------------------------------------------------
class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 50 ms while running."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self) -> dict:
        rows = []
        try:
            for line in open(self.path):
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 7 and parts[0].replace(".", "").isdigit():
                    rows.append(parts)
        except OSError:
            pass
        finally:
            if self.path:
                os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm = [float(r[0]) for r in rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[3:7]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(float(r[1]) for r in rows),
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max(float(r[2]) for r in rows if r[2].replace(".", "").isdigit())
                if any(r[2].replace(".", "").isdigit() for r in rows) else None}


def measured_hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        return float(json.load(open(p))["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def bench_probes(dev, stream, nbytes=4 << 30, K=10, W=3):
    """The library's HBM ceiling probes on a buffer of nbytes (31x the L2 at the default):
    a read-only stream and a copy of half the buffer into the other half; best of K."""
    import paged_kv_cache_175_gb300 as pkv
    buf = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    buf.fill_(1)
    half = nbytes // 2
    src, dst = buf[:half], buf[half:]
    none = lambda: None
    t_read = min(time_steps(lambda: pkv.probe_read(buf), K, W, none, stream))
    t_copy = min(time_steps(lambda: pkv.probe_copy(src, dst), K, W, none, stream))
    del buf, src, dst
    torch.cuda.empty_cache()
    return {"read_gbs": round(nbytes / (t_read / 1e3) / 1e9, 1),
            "copy_gbs": round(2 * half / (t_copy / 1e3) / 1e9, 1),
            "bytes": nbytes, "best_of": K, "launches": 2 * (K + W)}


# the files each captured attention kernel is compiled from (the plan and split-reduce
# kernels live elsewhere and do not change its traffic)
KERNEL_SOURCES = {
    "bf16": ["decode_bf16.cu", "decode_common.cuh", "pkv_device.cuh"],
    "int4": ["int4.cu", "decode_common.cuh", "pkv_device.cuh"],
}


def source_hash(family: str = "bf16") -> str:
    """Hash of the sources the attention kernels of one family are built from."""
    h = hashlib.sha256()
    d = os.path.join(ROOT, "paged_kv_cache_175_gb300", "csrc")
    for f in KERNEL_SOURCES[family]:
        h.update(open(os.path.join(d, f), "rb").read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per launch of the dominant kernel from a committed ncu summary, if it was
    taken on the current kernel sources (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        rec = json.load(open(p))[workload]
    except (OSError, KeyError, ValueError):
        return None
    fam = "int4" if workload.startswith("int4") else "bf16"
    return rec["bytes_per_launch"] if rec.get("source_hash") == source_hash(fam) else None


# ---------------------------------------------------------------------------------------------
def l2_policy(step_bytes, flush_buf):
    """Steps that stream at least 4x the L2 need no flush (the data a step leaves in L2 is
    the tail of each CTA's piece, which the next step reaches last, after evicting it).
    Smaller steps get a flush between timed steps: a write of 2x L2, then a read of it, so
    the written lines are evicted (and written back) before the timed step rather than
    during it; the step starts from a cold, clean L2."""
    if step_bytes >= 4 * L2_BYTES:
        return (lambda: None), "no flush: each step streams >= 4x the L2 (inputs larger than L2)"

    def flush():
        flush_buf.zero_()
        flush_buf.view(torch.int32).max()

    return flush, "L2 flushed between steps (write of 2x L2, then read back; outside the events)"


def time_steps(step, K, W, flush, stream):
    """W untimed warm-up steps, then K steps each timed by CUDA events on `stream`,
    with `flush` (an L2 flush, or nothing for steps larger than L2) between them."""
    for _ in range(W):
        flush()
        step()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for a, b in evs:
        flush()
        a.record(stream)
        step()
        b.record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


class Bf16Step:
    def __init__(self, name, seed, dev):
        import paged_kv_cache_175_gb300 as pkv
        self.pkv = pkv
        self.w = w = workloads.make(name, seed)
        self.k_pool, self.v_pool = workloads.pools_bf16(w, seed, dev)
        self.q = workloads.queries(w, seed, dev)
        self.kn, self.vn = workloads.new_tokens(w, seed, dev)
        self.slots = torch.as_tensor(workloads.decode_slots(w), device=dev)
        self.bt = torch.as_tensor(w.block_tables, device=dev)
        self.ctx = torch.as_tensor(w.context_lens, device=dev)
        self.out = torch.empty_like(self.q)
        nbytes = pkv.decode_workspace_bytes(w.batch, w.n_h, w.n_kv, w.head_dim, w.block_size)
        self.ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        # append, attention, split-reduce; the library adds a plan kernel above 256 sequences
        self.launches_per_step = 3 + (w.batch > PLAN_KERNEL_ABOVE)
        self.attention_launches = self.launches_per_step - 1
        self.inputs = {"q": self.q, "kn": self.kn, "vn": self.vn, "slots": self.slots, "bt": self.bt,
                       "ctx": self.ctx}

    def attention(self, x=None):
        x = x or self.inputs
        if self.w.window:
            self.pkv.paged_decode_attn_window(x["q"], self.k_pool, self.v_pool, x["bt"], x["ctx"], self.w.scale,
                                              self.w.window, out=x.get("out", self.out), workspace=self.ws,
                                              err=self.err)
        else:
            self.pkv.paged_decode_attn(x["q"], self.k_pool, self.v_pool, x["bt"], x["ctx"], self.w.scale,
                                       out=x.get("out", self.out), workspace=self.ws, err=self.err)

    def step(self, x=None):
        x = x or self.inputs
        self.pkv.kv_append(x["kn"], x["vn"], x["slots"], self.k_pool, self.v_pool, err=self.err)
        self.attention(x)

    def bytes(self):
        return attention_bytes(self.w) + append_bytes(self.w), attention_bytes(self.w)


class Int4Step:
    def __init__(self, name, seed, dev):
        import paged_kv_cache_175_gb300 as pkv
        self.pkv = pkv
        self.w = w = workloads.make(name, seed)
        # the cache holds ctx-1 tokens of history; the step appends token ctx-1 and attends
        self.cache = pkv.alloc_int4_cache(w.num_blocks, w.n_kv, w.block_size, w.head_dim, w.batch, dev)
        ks, vs, sl, tl, newk, newv = [], [], [], [], [], []
        for s in range(w.batch):
            k, v = workloads.history_kv(w, s, seed, dev)
            slots = workloads.history_slots(w, s)
            ks.append(k[:-1]); vs.append(v[:-1]); sl.append(slots[:-1])
            tl.append(np.full(len(slots) - 1, s, np.int32))
            newk.append(k[-1]); newv.append(v[-1])
        pkv.kv_quant_append_int4(torch.cat(ks), torch.cat(vs), torch.as_tensor(np.concatenate(sl), device=dev),
                                 torch.as_tensor(np.concatenate(tl), device=dev), self.cache)
        torch.cuda.synchronize()
        del ks, vs
        torch.cuda.empty_cache()
        self.kn, self.vn = torch.stack(newk).contiguous(), torch.stack(newv).contiguous()
        self.slots = torch.as_tensor(workloads.decode_slots(w), device=dev)
        self.tails = torch.arange(w.batch, dtype=torch.int32, device=dev)
        self.q = workloads.queries(w, seed, dev)
        self.bt = torch.as_tensor(w.block_tables, device=dev)
        self.ctx = torch.as_tensor(w.context_lens, device=dev)
        self.out = torch.empty_like(self.q)
        nbytes = pkv.decode_workspace_bytes(w.batch, w.n_h, w.n_kv, w.head_dim, w.block_size, int4=True)
        self.ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        # quantize, tail update, attention, split-reduce (+ plan above 256 sequences)
        self.launches_per_step = 4 + (w.batch > PLAN_KERNEL_ABOVE)
        self.attention_launches = self.launches_per_step - 2
        self.inputs = {"q": self.q, "kn": self.kn, "vn": self.vn, "slots": self.slots, "tails": self.tails,
                       "bt": self.bt, "ctx": self.ctx}

    def attention(self, x=None):
        x = x or self.inputs
        if self.w.window:
            self.pkv.paged_decode_attn_int4_window(x["q"], self.cache, x["bt"], x["ctx"], self.w.scale,
                                                   self.w.window, out=x.get("out", self.out), workspace=self.ws,
                                                   err=self.err)
        else:
            self.pkv.paged_decode_attn_int4(x["q"], self.cache, x["bt"], x["ctx"], self.w.scale, out=x.get("out", self.out),
                                            workspace=self.ws, err=self.err)

    def step(self, x=None):
        x = x or self.inputs
        self.pkv.kv_quant_append_int4(x["kn"], x["vn"], x["slots"], x["tails"], self.cache, err=self.err)
        self.attention(x)

    def bytes(self):
        return attention_bytes(self.w, True) + append_bytes(self.w, True), attention_bytes(self.w, True)


class RopeStep:
    def __init__(self, name, seed, dev):
        import paged_kv_cache_175_gb300 as pkv
        self.pkv = pkv
        self.w = w = workloads.make(name, seed)
        self.k_pool, _ = workloads.pools_bf16(w, seed, dev)
        self.ids = torch.as_tensor(w.extra["rope_block_ids"], device=dev)
        self.deltas = torch.as_tensor(w.extra["rope_deltas"], device=dev)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        self.launches_per_step = 1
        self.attention_launches = 1
        self.out = None
        self.inputs = {"ids": self.ids, "deltas": self.deltas}

    def step(self, x=None):
        x = x or self.inputs
        self.pkv.rope_shift_k(self.k_pool, x["ids"], x["deltas"], err=self.err)

    attention = step

    def bytes(self):
        w = self.w
        nz = int(np.count_nonzero(w.extra["rope_deltas"]))
        b = nz * w.n_kv * w.block_size * w.head_dim * 2 * 2 + len(w.extra["rope_deltas"]) * 8
        return b, b


class BlendStep:
    """One layer of CacheBlend's model-free steps on the 64 reused 512-token chunks of a
    workload: KV deviation of every chunk token against its recomputed K/V (synthetic:
    the cached rows plus noise of a per-token scale), the 15% of each chunk with the
    largest deviation selected, their recomputed rows fused into the cache."""

    def __init__(self, name, seed, dev):
        import paged_kv_cache_175_gb300 as pkv
        self.pkv = pkv
        self.w = w = workloads.make(name, seed)
        bs = w.block_size
        self.k_pool, self.v_pool = workloads.pools_bf16(w, seed, dev)
        blocks = w.extra["rope_block_ids"].astype(np.int64)
        slots = (blocks[:, None] * bs + np.arange(bs)[None, :]).reshape(-1)
        self.n = n = len(slots)
        self.chunk = 512
        self.slots = torch.as_tensor(slots, device=dev)
        g = torch.Generator(device=dev).manual_seed(seed + 17)
        blk, row = self.slots // bs, self.slots % bs
        scale = torch.rand(n, 1, 1, generator=g, device=dev) ** 3
        shape = (n, w.n_kv, w.head_dim)
        self.kn = (self.k_pool[blk, :, row].float() + scale * torch.randn(*shape, generator=g, device=dev)).to(torch.bfloat16)
        self.vn = (self.v_pool[blk, :, row].float() + scale * torch.randn(*shape, generator=g, device=dev)).to(torch.bfloat16)
        n_seg = n // self.chunk
        self.k_sel = pkv.select_count(0.15, self.chunk)
        self.offs = torch.arange(0, n + 1, self.chunk, dtype=torch.int32, device=dev)
        self.counts = torch.full((n_seg,), self.k_sel, dtype=torch.int32, device=dev)
        self.dev_buf = torch.empty(n, dtype=torch.float32, device=dev)
        self.sel = torch.empty(n_seg * self.k_sel, dtype=torch.int32, device=dev)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        self.out = None
        self.launches_per_step = 3                 # deviation, selection, fuse
        self.attention_launches = 1                # deviation alone
        self.inputs = {}

    def attention(self, x=None):
        self.pkv.kv_deviation(self.k_pool, self.v_pool, self.slots, self.kn, self.vn, out=self.dev_buf, err=self.err)

    def step(self, x=None):
        self.attention()
        self.pkv.select_top(self.dev_buf, self.offs, self.counts, out=self.sel)
        self.pkv.kv_fuse(self.kn, self.vn, self.slots, self.sel, self.k_pool, self.v_pool, err=self.err)

    def bytes(self):
        w = self.w
        row = w.n_kv * w.head_dim * 2
        dev_b = 4 * self.n * row + self.n * 8 + self.n * 4          # pool and new rows, slots, dev out
        k = self.sel.numel()
        step_b = dev_b + self.n * 4 + k * 4 + k * (8 + 4 * row)      # dev in; ids; slots, new rows in, pool rows out
        return step_b, dev_b


def make_step(name, seed, dev):
    if name.startswith("int4"):
        return Int4Step(name, seed, dev)
    if name.startswith("rope_"):
        return RopeStep(name[5:], seed, dev)
    if name.startswith("blend_"):
        return BlendStep(name[6:], seed, dev)
    return Bf16Step(name, seed, dev)


# ---------------------------------------------------------------------------------------------
def cpu_samples(name, seed, n_seqs):
    """Host inputs for the oracle: n_seqs sequences of the workload, each with a compact
    pool holding just its blocks (same shapes and value distribution as the GPU arm)."""
    w = workloads.make(name, seed)
    order = np.random.default_rng(seed + 99).permutation(w.batch)[:n_seqs]
    f64 = lambda t: t.float().numpy().astype(np.float64)
    out = []
    for i, s in enumerate(int(x) for x in order):
        c = int(w.context_lens[s])
        nb = -(-c // w.block_size)
        shape = (nb, w.n_kv, w.block_size, w.head_dim)
        kb = f64(workloads.normal_bf16(shape, 1000 + 4 * i))
        vb = f64(workloads.normal_bf16(shape, 1001 + 4 * i))
        q = f64(workloads.normal_bf16((1, w.n_h, w.head_dim), 1002 + 4 * i))
        kv = f64(workloads.normal_bf16((2, 1, w.n_kv, w.head_dim), 1003 + 4 * i))
        sub = workloads.Workload(w.name, 1, w.n_h, w.n_kv, w.head_dim, w.block_size,
                                 w.context_lens[s:s + 1], np.arange(nb, dtype=np.int32)[None, :], nb, w.scale,
                                 window=w.window)
        out.append((sub, kb, vb, q, kv[0], kv[1], np.array([(c - 1)], dtype=np.int64)))
    return out


def blas_threads():
    """Threads numpy's BLAS runs with (threadpoolctl where installed, else the usual
    environment variables, else the host's core count, which OpenBLAS defaults to)."""
    try:
        from threadpoolctl import threadpool_info
        n = [int(i["num_threads"]) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return max(n)
    except Exception:
        pass
    for v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(v, "").isdigit():
            return int(os.environ[v])
    return os.cpu_count()


def time_cpu(samples, budget_s):
    """Run the oracle's decode step over the samples (cycling) until budget_s seconds."""
    import oracle
    done, nbytes, elapsed = 0, 0, 0.0
    ru = lambda: sum(resource.getrusage(resource.RUSAGE_SELF)[:2])
    cpu0, wall0 = ru(), time.perf_counter()
    while elapsed < budget_s:
        sub, kb, vb, q, kn, vn, slot = samples[done % len(samples)]
        t0 = time.perf_counter()
        k2, v2 = oracle.kv_append(kb, vb, kn, vn, slot, sub.block_size)
        oracle.paged_decode_attention(q, k2, v2, sub.block_tables, sub.context_lens, sub.scale, sub.block_size,
                                      window=sub.window)
        elapsed += time.perf_counter() - t0
        nbytes += attention_bytes(sub) + append_bytes(sub)
        done += 1
    util = (ru() - cpu0) / max(time.perf_counter() - wall0, 1e-9)
    info = {"sample": f"{done} sequence decode steps (append + attention, all heads) of the {samples[0][0].name} "
                      f"workload, {elapsed:.1f} s of oracle time", "cores": os.cpu_count(),
            "blas_threads": blas_threads(), "cpu_time_per_wall_time": round(util, 2), "kind": "oracle"}
    return nbytes / elapsed / 1e9, done / elapsed, elapsed, info


# ---------------------------------------------------------------------------------------------
def bench_offload(dev, stream, K, W, world, n_blocks=4096):
    """Offload and onload of n_blocks blocks of the 8B-shaped pool between HBM and
    page-locked host memory through pkv_copy_blocks, against one contiguous
    cudaMemcpyAsync of the same bytes each way (the copy engines' ceiling on this node)."""
    import paged_kv_cache_175_gb300 as pkv
    w = workloads.make("llama3_8b", 0)
    shape = (w.num_blocks, w.n_kv, w.block_size, w.head_dim)
    kp, vp = workloads.pools_bf16(w, 0, dev)
    hshape = (n_blocks,) + shape[1:]
    kh = torch.empty(hshape, dtype=torch.bfloat16).pin_memory()
    vh = torch.empty(hshape, dtype=torch.bfloat16).pin_memory()
    rng = np.random.default_rng(3)
    src = rng.permutation(w.num_blocks)[:n_blocks]
    dst = rng.permutation(w.num_blocks)[:n_blocks]
    off = np.stack([np.zeros(n_blocks, int), src, np.arange(n_blocks)], 1)
    on = np.stack([np.ones(n_blocks, int), np.arange(n_blocks), dst], 1)
    moved = 2 * n_blocks * int(np.prod(shape[1:])) * 2                  # K and V bytes per direction
    none = lambda: None
    t_off = reduce_max(statistics.mean(time_steps(lambda: pkv.copy_blocks(off, kp, vp, kh, vh), K, W, none, stream)), world)
    t_on = reduce_max(statistics.mean(time_steps(lambda: pkv.copy_blocks(on, kp, vp, kh, vh), K, W, none, stream)), world)
    flat_d = torch.empty(moved // 2, dtype=torch.uint8, device=dev)
    flat_h = torch.empty(moved // 2, dtype=torch.uint8).pin_memory()
    d2h = lambda: (flat_h.copy_(flat_d, non_blocking=True), flat_h.copy_(flat_d, non_blocking=True))
    h2d = lambda: (flat_d.copy_(flat_h, non_blocking=True), flat_d.copy_(flat_h, non_blocking=True))
    t_d2h = reduce_max(statistics.mean(time_steps(d2h, K, W, none, stream)), world)
    t_h2d = reduce_max(statistics.mean(time_steps(h2d, K, W, none, stream)), world)
    gb = lambda ms: moved / (ms / 1e3) / 1e9
    launches = -(-n_blocks // 480)                                       # one wave, 480 copies per launch
    return ({"blocks": n_blocks, "bytes_per_direction": moved,
             "offload_gbs": round(gb(t_off), 2), "onload_gbs": round(gb(t_on), 2),
             "memcpy_d2h_gbs": round(gb(t_d2h), 2), "memcpy_h2d_gbs": round(gb(t_h2d), 2),
             "offload_frac_of_memcpy": round(t_d2h / t_off, 4), "onload_frac_of_memcpy": round(t_h2d / t_on, 4),
             "steps": K}, 2 * launches * K)


def block_manager_trace(w, seed, decode_steps):
    """Prompts of the 70B-prefix workload (the sharers' first 2048 tokens identical), each
    then decoding `decode_steps` tokens: (prompts, decode token matrix)."""
    rng = np.random.default_rng(seed)
    prefix = rng.integers(0, 32000, size=w.shared_prefix_blocks * w.block_size)
    prompts = []
    for s in range(w.batch):
        n = int(w.context_lens[s]) - decode_steps
        own = rng.integers(0, 32000, size=n)
        if s < w.n_sharers:
            own[:len(prefix)] = prefix
        prompts.append(own.astype(np.int32))
    return prompts, rng.integers(0, 32000, size=(decode_steps, w.batch)).astype(np.int32)


def run_block_manager(bm, prompts, decode, add, append, release):
    """Admit every prompt, run the decode steps, release all, admit them again (prefix
    reuse); seconds of each phase."""
    t0 = time.perf_counter()
    for s, p in enumerate(prompts):
        add(bm, s, p)
    t1 = time.perf_counter()
    ids = np.arange(len(prompts), dtype=np.int64)
    for row in decode:
        append(bm, ids, row)
    t2 = time.perf_counter()
    for s in range(len(prompts)):
        release(bm, s)
    for s, p in enumerate(prompts):
        add(bm, len(prompts) + s, p)
    t3 = time.perf_counter()
    return t1 - t0, t2 - t1, t3 - t2


def bench_block_manager(rank, decode_steps=16):
    """Host cost of the native block manager on a serving trace shaped like the 70B-prefix
    workload, with the oracle's restatement timed on a bounded sample of it."""
    import paged_kv_cache_175_gb300 as pkv
    w = workloads.make("llama2_70b_prefix", rank)
    prompts, decode = block_manager_trace(w, rank, decode_steps)
    need = sum(-(-int(c) // w.block_size) for c in w.context_lens)
    N = int(need * 1.2)
    for rep in range(2):                              # the first pass warms caches and allocators
        nat = pkv.BlockManager(N, w.block_size, host_blocks=N // 4)
        ta, td, tr = run_block_manager(nat, prompts, decode, lambda b, s, p: b.add_sequence(s, p),
                                       lambda b, i, r: b.append_tokens(i, r), lambda b, s: b.release(s))
    reused = nat.counts()["reused_tokens"]
    tokens = int(sum(len(p) for p in prompts))
    out = {"requests": w.batch, "prompt_tokens": tokens, "decode_steps": decode_steps, "pool_blocks": N,
           "admit_tokens_per_s": round(tokens / ta, 1), "decode_step_us": round(td / decode_steps * 1e6, 2),
           "decode_appends_per_s": round(w.batch * decode_steps / td, 1),
           "readmit_tokens_per_s": round(tokens / tr, 1), "reused_tokens": reused}
    # the oracle (linear scans) on the first 16 requests and 8 decode steps, smaller pool
    import oracle
    sub_p, sub_d = prompts[:16], decode[:8, :16]
    need_s = sum(-(-(len(p) + 8) // w.block_size) for p in sub_p)
    ref = oracle.BlockManager(int(need_s * 1.2), w.block_size, host_blocks=need_s // 4)
    ra, rd, rr = run_block_manager(ref, sub_p, sub_d, lambda b, s, p: b.add_sequence(s, p),
                                   lambda b, i, r: [b.append_token(int(s), int(t)) for s, t in zip(i, r)],
                                   lambda b, s: b.release(s))
    st = int(sum(len(p) for p in sub_p))
    out["cpu_baseline"] = {"kind": "oracle", "sample": "first 16 requests, 8 decode steps",
                           "admit_tokens_per_s": round(st / ra, 1),
                           "decode_appends_per_s": round(16 * 8 / rd, 1)}
    return out


# ---------------------------------------------------------------------------------------------
def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def reduce_max(x: float, world: int) -> float:
    """Max of a per-rank scalar over all ranks (the slowest rank sets the job's time)."""
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(per_rank_bytes: float, per_rank_seqs: int, max_ms_total: float, world: int, steps: int) -> dict:
    """Whole-job throughput: every rank processes its own replica (weak scaling)."""
    secs = max_ms_total / 1e3
    return {"gbs": per_rank_bytes * world * steps / secs / 1e9, "seqs_per_s": per_rank_seqs * world * steps / secs,
            "ms_per_step": max_ms_total / steps}


def run_config(name, K, W, seed, dev, stream, flush_buf, world):
    st = make_step(name, seed, dev)
    step_bytes, attn_bytes = st.bytes()
    flush, _ = l2_policy(step_bytes, flush_buf)
    torch.cuda.synchronize()
    barrier(world)
    ms = time_steps(st.step, K, W, flush, stream)
    total = reduce_max(sum(ms), world)
    agg = aggregate(step_bytes, st.w.batch, total, world, K)
    ams = time_steps(st.attention, K, min(W, 3), flush, stream)
    attn_ms = reduce_max(statistics.mean(ams), world)
    assert int(st.err.item()) == 0, f"{name}: device error flag {int(st.err.item())}"
    return st, step_bytes, attn_bytes, agg, attn_ms


STEP_NAMES = {"Bf16Step": "kv_append + paged_decode_attn",
              "Int4Step": "kv_quant_append_int4 + paged_decode_attn_int4",
              "RopeStep": "rope_shift_k",
              "BlendStep": "kv_deviation + select_top + kv_fuse"}


def step_class_name(name):
    if name.startswith("int4"):
        return "Int4Step"
    if name.startswith("rope_"):
        return "RopeStep"
    if name.startswith("blend_"):
        return "BlendStep"
    return "Bf16Step"


def workload_config(name, world):
    """The `config` object of the JSON line (both arms print the same one)."""
    import workloads as wl
    cls = step_class_name(name)
    w = wl.make(name[5:] if cls == "RopeStep" else name[6:] if cls == "BlendStep" else name, 0)
    if cls == "Bf16Step":
        step_bytes = attention_bytes(w) + append_bytes(w)
    elif cls == "Int4Step":
        step_bytes = attention_bytes(w, True) + append_bytes(w, True)
    else:
        step_bytes = None
    l2 = ("no flush: each step streams >= 4x the L2 (inputs larger than L2)"
          if step_bytes is not None and step_bytes >= 4 * L2_BYTES else
          "L2 flushed between steps (write of 2x L2, then read back; outside the events)")
    return {"workload": f"{name}: {w.n_h} q / {w.n_kv} kv heads, head_dim {w.head_dim}, block "
                        f"{w.block_size}, batch {w.batch}, ctx mean {float(np.mean(w.context_lens)):.0f}",
            "step": STEP_NAMES[cls], "parallelism": f"replicas x{world}", "l2": l2,
            "algorithmic_bytes_per_step": step_bytes}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="pkv", choices=["pkv", "reference"])
    ap.add_argument("--workload", default="llama3_8b")
    ap.add_argument("--configs", default="all", choices=["all", "main"])
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle time for cpu_baseline")
    ap.add_argument("--probe-only", action="store_true", help="only the HBM ceiling probes (one JSON line)")
    ap.add_argument("--kernel-only", action="store_true",
                    help="only W + K steps of --workload, no end-to-end, probe or other workloads (for profilers)")
    ap.add_argument("--probe-bytes", type=int, default=4 << 30, help="buffer of the ceiling probes")
    args = ap.parse_args()
    K, W = args.steps, max(args.warmup, 0)
    world, rank, local = dist_setup(args.gpus)

    if args.impl == "reference":
        if rank != 0:
            return
        # each step: the oracle on a bounded sample, sized so the whole run takes about two minutes
        per_step = max(0.05, min(10.0, 120.0 / max(1, K + W)))
        samples = cpu_samples(args.workload, 0, 4)
        for _ in range(W):
            time_cpu(samples, per_step)
        gbs, sps, tot = [], [], 0.0
        info = None
        for _ in range(K):
            g, s, el, info = time_cpu(samples, per_step)
            gbs.append(g); sps.append(s); tot += el
        v = statistics.mean(gbs)
        print(json.dumps({
            "impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": "GB/s", "n_gpus": 1, "steps": K,
            "warmup": W, "ms_per_step": round(tot / K * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(args.workload, 1),
            "seqs_per_s": round(statistics.mean(sps), 3),
            "cpu_baseline": {"value": round(v, 4), "unit": "GB/s", "cores": info["cores"], "kind": "oracle",
                             "sample": f"each step: {info['sample']}", "blas_threads": info["blas_threads"],
                             "cpu_time_per_wall_time": info["cpu_time_per_wall_time"]},
            "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}))
        return

    import paged_kv_cache_175_gb300 as pkv
    from paged_kv_cache_175_gb300._build import build_library
    if rank == 0:
        build_library()
    barrier(world)
    pkv.lib()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    flush_buf = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)
    peak, peak_src = measured_hbm_peak()
    if args.probe_only:
        pr = bench_probes(dev, stream, args.probe_bytes, K, W)
        if rank == 0:
            print(json.dumps({"probes": pr, "measured_copy_gbs": peak}))
        return

    # ---- main workload: timed steps with clocks sampled during the timed region ----
    main_step = make_step(args.workload, rank, dev)
    step_bytes, attn_bytes = main_step.bytes()
    flush, l2_note = l2_policy(step_bytes, flush_buf)
    if args.kernel_only:
        ms = time_steps(main_step.step, K, W, flush, stream)
        assert int(main_step.err.item()) == 0, f"device error flag {int(main_step.err.item())}"
        if rank == 0:
            print(json.dumps({"workload": args.workload, "steps": K, "warmup": W,
                              "ms_per_step": round(statistics.mean(ms), 5),
                              "step_gbs": round(step_bytes / (statistics.mean(ms) / 1e3) / 1e9, 2)}))
        return
    torch.cuda.synchronize()
    barrier(world)
    with ClockSampler(local) as clk:
        ms = time_steps(main_step.step, K, W, flush, stream)
    clocks = clk.summary()
    total_ms = reduce_max(sum(ms), world)
    agg = aggregate(step_bytes, main_step.w.batch, total_ms, world, K)
    ams = time_steps(main_step.attention, K, min(W, 3), flush, stream)
    attn_ms = reduce_max(statistics.mean(ams), world)
    assert int(main_step.err.item()) == 0, f"device error flag {int(main_step.err.item())}"

    # ---- end to end through the public API: pinned host inputs in, output back out ----
    # Every step copies its inputs in from pinned host memory and its result back out,
    # double-buffered on a second stream: step j+1's inputs go in while step j's kernels run,
    # and step j's result comes out while step j+1's kernels run (the pipelining of a serving
    # loop).  The inputs travel packed in one pinned buffer per step (one copy; the
    # device-side tensors are views of one device buffer); the launches of G steps are one
    # CUDA graph.
    w = main_step.w
    layout, off = {}, 0
    for k, v in main_step.inputs.items():
        layout[k] = (off, v.dtype, v.shape, v.numel() * v.element_size())
        off += -(-layout[k][3] // 256) * 256
    h_pack = torch.empty(max(off, 256), dtype=torch.uint8).pin_memory()
    for k, v in main_step.inputs.items():
        o, _, _, nb = layout[k]
        h_pack[o:o + nb].copy_(v.contiguous().view(-1).view(torch.uint8).cpu())
    d_pack = [torch.empty_like(h_pack, device=dev) for _ in range(2)]
    d = [{k: d_pack[b][o:o + nb].view(dt).view(shp) for k, (o, dt, shp, nb) in layout.items()} for b in range(2)]
    has_out = main_step.out is not None
    out_d = [torch.empty_like(main_step.out) for _ in range(2)] if has_out else [None, None]
    out_h = [torch.empty(main_step.out.shape, dtype=main_step.out.dtype).pin_memory() for _ in range(2)] \
        if has_out else [None, None]
    h2d = sum(nb for (_, _, _, nb) in layout.values())
    d2h = out_h[0].numel() * out_h[0].element_size() if has_out else 0
    copy_stream = torch.cuda.Stream(device=dev)

    def step_args(b):
        x = dict(d[b])
        if has_out:
            x["out"] = out_d[b]
        return x

    def one_step(b):                                      # a step on its own, copies in order
        d_pack[b].copy_(h_pack, non_blocking=True)
        flush()
        main_step.step(step_args(b))
        if has_out:
            out_h[b].copy_(out_d[b], non_blocking=True)

    # G steps per graph launch: the double-buffered pipeline below runs inside each graph,
    # so G only sets how often the first input copy and the last result copy are exposed
    # (measured on the 8B line: 8 / 16 / 32 steps per graph gave 97.5 / 99.1 / 99.6% of the
    # device-timed rate); the K % G steps left over run as a second, shorter graph
    G = max(1, min(32, K))
    ev_k = [torch.cuda.Event() for _ in range(G)]
    ev_in = [torch.cuda.Event() for _ in range(G)]
    ev_out = [torch.cuda.Event() for _ in range(G)]

    def group_steps(ng=G):                                # steps j = 0..ng-1 on buffers j % 2
        cs = torch.cuda.current_stream()
        copy_stream.wait_stream(cs)
        d_pack[0].copy_(h_pack, non_blocking=True)
        for j in range(ng):
            if j + 1 < ng:                                # step j+1's inputs, once step j-1 is done with the buffer
                with torch.cuda.stream(copy_stream):
                    if j >= 1:
                        copy_stream.wait_event(ev_k[j - 1])
                    d_pack[(j + 1) % 2].copy_(h_pack, non_blocking=True)
                    ev_in[j + 1].record(copy_stream)
            if j >= 1:
                cs.wait_event(ev_in[j])
            if j >= 2 and has_out:
                cs.wait_event(ev_out[j - 2])              # step j-2's result has left out_d[j % 2]
            flush()                                       # as between the device-timed steps
            main_step.step(step_args(j % 2))
            ev_k[j].record(cs)
            if has_out:                                   # step j's result, beside step j+1's kernels
                with torch.cuda.stream(copy_stream):
                    copy_stream.wait_event(ev_k[j])
                    out_h[j % 2].copy_(out_d[j % 2], non_blocking=True)
                    ev_out[j].record(copy_stream)
        cs.wait_stream(copy_stream)

    R = K % G

    def e2e_run(n):
        for _ in range(n // G):
            if graph is not None:
                graph.replay()
            else:
                group_steps()
        if n % G:
            if graph_rem is not None and n % G == R:
                graph_rem.replay()
            else:
                for _ in range(n % G):
                    one_step(0)

    graph = graph_rem = None
    e2e_run(max(W, G))                                    # eager warm-up (sets up the library's kernels)
    torch.cuda.synchronize()
    try:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            group_steps()
        graph = g
        if R:
            g2 = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g2):
                group_steps(R)
            graph_rem = g2
        e2e_run(G + R)
        torch.cuda.synchronize()
        e2e_mode = f"one CUDA graph per group of {G} steps, replayed" + (f", and one of {R} steps" if R else "")
    except Exception as ex:                               # eager launches if capture is refused
        graph = graph_rem = None
        torch.cuda.synchronize()
        e2e_mode = f"eager launches (graph capture failed: {type(ex).__name__})"
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    copy_stream.wait_stream(stream)
    e2e_run(K)
    stream.wait_stream(copy_stream)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_total = reduce_max(e0.elapsed_time(e1), world)
    e2e = aggregate(step_bytes, w.batch, e2e_total, world, K)

    probes = bench_probes(dev, stream)
    ceiling = max(probes["read_gbs"], peak)
    achieved = attn_bytes / (attn_ms / 1e3) / 1e9

    line = {
        "metric": METRIC, "value": round(agg["gbs"], 2), "unit": "GB/s", "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": round(agg["ms_per_step"], 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": workload_config(args.workload, world),
        "seqs_per_s": round(agg["seqs_per_s"], 1),
        "frac_of_hbm_peak": round(agg["gbs"] / world / peak, 4),
        "e2e": {"value": round(e2e["gbs"], 2), "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "launch": e2e_mode,
                "copies": "inputs packed in one pinned buffer per step; double-buffered on a second stream: "
                          "step j+1's inputs go in and step j's result comes out beside the kernels",
                "ms_per_step": round(e2e["ms_per_step"], 5)},
        "roofline": {"bound": "hbm", "kernel": {"Bf16Step": "paged_decode_attn (attention + split-reduce)",
                                                "Int4Step": "paged_decode_attn_int4 (attention + split-reduce)",
                                                "RopeStep": "rope_shift_k",
                                                "BlendStep": "kv_deviation"}[type(main_step).__name__],
                     "achieved": round(attn_bytes / (attn_ms / 1e3) / 1e9, 2), "peak": peak,
                     "peak_source": f"{peak_src} (HBM copy, MEASURED_PEAKS.json)" if peak_src == "measured"
                     else "fallback 6.8 TB/s",
                     "unit": "GB/s", "frac": round(attn_bytes / (attn_ms / 1e3) / 1e9 / peak, 4),
                     "traffic": recorded_traffic(args.workload),
                     "algorithmic_bytes_per_launch": attn_bytes, "ms_per_launch": round(attn_ms, 5),
                     # the library's own ceiling probes, measured in this run: the attention
                     # kernels almost only read, so the read stream is their ceiling
                     "read_ceiling": {"kernel": "pkv_probe_read", "gbs": probes["read_gbs"],
                                      "copy_probe_gbs": probes["copy_gbs"],
                                      "denominator": round(ceiling, 1),
                                      "denominator_is": "max(read probe, measured copy)",
                                      "frac": round(achieved / ceiling, 4)}},
        # the timed loops: steps, attention alone, end to end; the probes
        "gpu_launches": main_step.launches_per_step * 2 * K + main_step.attention_launches * K + probes["launches"],
        "clocks": clocks,
    }

    # ---- other workloads ----
    if args.configs == "all":
        by = {}
        kk, ww = max(5, min(K, 30)), max(3, min(W, 5))
        for name in ["llama2_70b_prefix", "mqa_bs16", "mqa_bs32", "mha_bs16", "mha_bs32", "rope_mqa_bs16",
                     "rope_mha_bs32", "int4_long", "int4_long_bs64", "llama3_8b_window256", "blend_mqa_bs16",
                     "blend_mha_bs32"]:
            if name == args.workload:
                continue
            st, sb, ab, ag, am = run_config(name, kk, ww, rank, dev, stream, flush_buf, world)
            by[name] = {"gbs": round(ag["gbs"], 2), "frac_of_hbm_peak": round(ag["gbs"] / world / peak, 4),
                        "seqs_per_s": round(ag["seqs_per_s"], 1), "ms_per_step": round(ag["ms_per_step"], 5),
                        "bytes_per_step": sb, "attn_gbs": round(ab / (am / 1e3) / 1e9, 2),
                        "attn_frac": round(ab / (am / 1e3) / 1e9 / peak, 4), "attn_ms": round(am, 5),
                        "steps": kk}
            line["gpu_launches"] += (st.launches_per_step + st.attention_launches) * kk
            del st
            torch.cuda.empty_cache()
        off, n_launch = bench_offload(dev, stream, kk, ww, world)
        by["offload_llama3_8b"] = off
        line["gpu_launches"] += n_launch
        by["block_manager_llama2_70b_prefix"] = bench_block_manager(rank)
        line["by_config"] = by
        # compact per-workload fractions of the attention call (of the measured copy / of the
        # read ceiling), printed last so that a tail of the line still shows them
        fr = {args.workload: (round(achieved / peak, 4), round(achieved / ceiling, 4))}
        for k, v in by.items():
            if "attn_gbs" in v:
                fr[k] = (v["attn_frac"], round(v["attn_gbs"] / ceiling, 4))

    # ---- oracle on the host cores (rank 0, one GPU only) ----
    if rank == 0 and world == 1 and args.cpu_budget > 0 and isinstance(main_step, Bf16Step):
        g, s, el, info = time_cpu(cpu_samples(args.workload, 0, 8), args.cpu_budget)
        line["cpu_baseline"] = {"value": round(g, 4), "unit": "GB/s", "cores": info["cores"], "kind": "oracle",
                                "sample": info["sample"], "seqs_per_s": round(s, 3),
                                "blas_threads": info["blas_threads"],
                                "cpu_time_per_wall_time": info["cpu_time_per_wall_time"]}
    if args.configs == "all":
        line["attn_frac_of_copy_and_read_ceiling"] = fr
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
