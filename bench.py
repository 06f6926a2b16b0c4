#!/usr/bin/env python
"""Benchmark of the attention hot path on one GB300 (or N, one process each).

One step is one pass over every hot-path kernel on its workload:
  * causal GQA prefill   B=2, S=8192, H_q=32, H_kv=8, D=128   (headline: TFLOP/s,
    causal FLOPs counted as 2*B*H_q*S^2*D)
  * the same shape without the mask (the unmasked tensor-core ceiling)
  * causal GQA prefill at the Qwen3-0.6B attention shape, B=4, S=1024, H 16/8
    (L2 flushed before each launch: its inputs would otherwise stay in L2)
  * one layer's chunked step from raw projections (4 sequences, 6144 cached +
    2048 new tokens each, H 32/8), with its QK-norm + RoPE + KV append
    prologue, unfused (separate query pass) and fused (queries normalised and
    rotated inside the prefill kernel)
  * the chunked prefill alone (FLOPs over each query's visible keys); it runs
    just before the decode legs, as it leaves the least dirty data in L2
  * paged decode          256 sequences, lengths uniform on [128, 2048], H 16/8
  * the 256-sequence decode step together with its KV append (two launches)
  * paged decode          8 sequences x 32768 tokens, H 16/8
  * paged decode          256 sequences as above, H 64/8 (eight query heads per
    kv head in one tensor-core tile)
    (decode: GB/s of K/V bytes of the valid tokens; split-K + combine kernels)
  * the attention-input prologue (QK-norm, RoPE, KV append) of 2 x 8192 new
    tokens, H 32/8 (GB/s of the bytes it must move)
Each kernel launch is bracketed by CUDA events on the stream it runs on; the
K timed steps are bracketed by a barrier and a device synchronisation.  All
inputs are resident in HBM; every leg's inputs are larger than L2 (129 MB)
except the Qwen3-0.6B-shaped prefill's, for which a 256 MB buffer is rewritten
before each launch, outside its events.

--impl reference times the FP64 CPU oracle instead (bounded row samples of the
same prefill workload on the host cores): a deliberately slow baseline.

Prints one JSON line (rank 0).  Under torchrun each rank runs the same work on
its own GPU (weak scaling, no collective on the data path).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "prefill attn TFLOP/s; paged-decode KV-read GB/s (fraction of GB300 peak)"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
KERNEL_SOURCES = {
    "prefill_kernel": ["prefill.cu", "ptx.cuh"],
    "decode_mma_kernel": ["decode.cu"],
    "qk_norm_rope_kernel": ["rope.cu", "ptx.cuh"],
}


# ------------------------------------------------------------------ helpers

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def dist_init(world: int, use_cuda: bool):
    if world <= 1:
        return None
    import torch.distributed as dist
    os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
    dist.init_process_group("nccl" if use_cuda else "gloo")
    return dist


def reduce_max(dist, x: float, use_cuda: bool) -> float:
    """Max of a float over ranks (identity without a process group)."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if use_cuda else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {k: float(p[k]) for k in FALLBACK_PEAKS}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def code_tokens(text: str) -> str:
    """C/C++/CUDA source with comments and whitespace removed (string literals kept)."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        elif c == '"':
            j = i + 1
            while j < n and text[j] != '"':
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        else:
            if not c.isspace():
                out.append(c)
            i += 1
    return "".join(out)


def source_hash(kernel: str) -> str:
    """Identifies the kernel's code: a comment or layout edit leaves it unchanged."""
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "attention_gqa_causal_gb300", "csrc", f)) as fh:
            h.update(code_tokens(fh.read()).encode())
    return h.hexdigest()[:16]


def dram_traffic(kernel: str, workload: str):
    """Per-launch DRAM bytes from the committed ncu summary, if it was taken
    on the current kernel source; else None."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            t = json.load(f)
        e = t[kernel][workload]
        return e["bytes_per_launch"] if e.get("source_hash") == source_hash(kernel) else None
    except (OSError, KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons while running.  Rows carry
    nvidia-smi's own timestamp, so stop() can keep those taken inside the timed region."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(index), f"--query-gpu={self.FIELDS}",
                                       "--format=csv,noheader,nounits", "-lms", "20"],
                                      stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.p = None

    def wait_ready(self, timeout: float = 5.0):
        """Block until the first sample is written (nvidia-smi takes a moment to start)."""
        end = time.time() + timeout
        while self.p is not None and time.time() < end and self.p.poll() is None:
            if os.path.getsize(self.f.name) > 0:
                return
            time.sleep(0.01)

    @staticmethod
    def _epoch(stamp: str):
        import datetime
        try:
            return datetime.datetime.strptime(stamp.strip(), "%Y/%m/%d %H:%M:%S.%f").timestamp()
        except ValueError:
            return None

    def stop(self, window=None):
        """Summarise the samples; with window = (t0, t1) in epoch seconds, only those
        stamped inside it (all of them if none fall inside)."""
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.p.terminate()
        self.p.wait()
        self.f.seek(0)
        rows = [r.split(",") for r in self.f.read().strip().splitlines() if r.strip()]
        os.unlink(self.f.name)
        inside = rows
        if window is not None:
            t0, t1 = window
            inside = [r for r in rows if (lambda t: t is not None and t0 <= t <= t1)(self._epoch(r[0]))]
            if not inside:
                inside = rows
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in inside:
            try:
                sm.append(float(r[1]))
                mx = float(r[2])
                for name, v in zip(names, r[5:9]):
                    if v.strip().lower() == "active":
                        reasons.add(name)
            except (ValueError, IndexError):
                continue
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "samples": len(sm), "samples_run": len(rows),
                "window": "timed region" if inside is not rows else "whole run",
                "reasons": sorted(reasons)}


# ------------------------------------------------------------------ GPU legs

class Leg:
    """One hot-path call on one workload.  bind(ins, out) returns a closure that
    runs it on the given device buffers (ins shaped like dev_in); out_alias is the
    index of the input that is also the output (in place), else None."""
    def __init__(self, name, kind, work, unit, launches):
        self.name, self.kind, self.work, self.unit, self.launches = name, kind, work, unit, launches
        self.times = []
        self.out_alias = None

    def set_buffers(self, bind, dev_in, dev_out):
        self.bind, self.dev_in, self.dev_out = bind, dev_in, dev_out
        self.run = bind(dev_in, dev_out)

    def value(self, ms):
        return self.work / (ms * 1e-3) / (1e12 if self.unit == "TFLOP/s" else 1e9)


def build_legs(torch, ag, which):
    legs = []
    if which in ("all", "prefill", "prefill_full"):
        Q, K, V = W.prefill_inputs(W.PREFILL_LONG, seed=0)
        dQ, dK, dV = (torch.from_numpy(x).cuda() for x in (Q, K, V))
        dO = torch.empty_like(dQ)
        host = {"Q": Q, "K": K, "V": V}
        for cfg in ((W.PREFILL_LONG,) if which == "prefill" else (W.PREFILL_LONG_FULL,)
                    if which == "prefill_full" else (W.PREFILL_LONG, W.PREFILL_LONG_FULL)):
            leg = Leg(cfg.name, "prefill", cfg.flops(), "TFLOP/s", 1)
            leg.cfg = cfg
            leg.set_buffers(lambda ins, out, c=cfg: (lambda: ag.attn_prefill(*ins, out, causal=c.causal)),
                            (dQ, dK, dV), dO)
            leg.host = host
            leg.config = {"B": cfg.B, "S": cfg.S, "H_q": cfg.H_q, "H_kv": cfg.H_kv, "D": cfg.D,
                          "causal": cfg.causal}
            legs.append(leg)
    if which in ("all", "qwen"):
        # the Qwen3-0.6B attention shape (B=4, S=1024, H 16/8, causal): its 50 MB of inputs
        # and outputs fit in L2, so L2 is flushed before each timed launch (and with
        # --workload qwen it is also timed as is, L2 warm)
        cfg = W.PREFILL_QWEN
        Q, K, V = W.prefill_inputs(cfg, seed=0)
        dQ, dK, dV = (torch.from_numpy(x).cuda() for x in (Q, K, V))
        dO = torch.empty_like(dQ)
        for flush in ((True,) if which == "all" else (False, True)):
            leg = Leg(cfg.name + ("_l2flush" if flush else ""), "prefill", cfg.flops(), "TFLOP/s", 1)
            leg.set_buffers(lambda ins, out: (lambda: ag.attn_prefill(*ins, out, causal=True)), (dQ, dK, dV), dO)
            leg.host = {"Q": Q, "K": K, "V": V}
            leg.flush = flush
            leg.config = {"B": cfg.B, "S": cfg.S, "H_q": cfg.H_q, "H_kv": cfg.H_kv, "D": cfg.D,
                          "causal": True, "l2": "flushed before each launch" if flush else "warm"}
            legs.append(leg)
    if which in ("all", "layer"):
        # One layer's attention step on the chunked workload, from raw projections:
        # QK-norm + RoPE + KV append of the 4 x 2048 new tokens, then the chunked
        # prefill.  Unfused: the prologue rewrites q in place and the prefill reads
        # it back.  Fused: the prologue handles keys and values only and the
        # prefill normalises and rotates each query row as it loads it.  Both are
        # timed over their two launches, as TFLOP/s of the attention FLOPs.
        cfg = W.CHUNKED_PREFILL
        L = W.chunked_layer_inputs(cfg, seed=0)
        cs = torch.empty((L["max_pos"], cfg.D), dtype=torch.float32, device="cuda")
        ag.attn_rope_cos_sin_table(cs, W.PROLOGUE.base)
        keys = ["Q", "k_cache", "v_cache", "cu_seqlens_q", "seq_lens_kv", "block_tables", "K", "V",
                "q_weight", "k_weight", "positions", "slot_mapping"]
        t = tuple(torch.from_numpy(L[k]).cuda() for k in keys)
        Op = torch.empty_like(t[0])
        for fused in (False, True):
            name = f"layer_{cfg.name}_{'fused' if fused else 'unfused'}"
            leg = Leg(name, "prefill", cfg.flops(), "TFLOP/s", 2)

            def bind(t, o, fused=fused, c=cfg, cs=cs):
                if fused:
                    return lambda: (ag.attn_qk_norm_rope_append(
                        None, t[6], t[7], None, t[9], cs, t[10], t[11], t[1], t[2], eps=1e-6, H_q=c.H_q),
                        ag.attn_prefill_paged_qk_norm_rope(t[0], t[1], t[2], o, t[3], t[4], t[5], t[8], cs,
                                                           c.chunk, eps=1e-6, causal=c.causal))
                return lambda: (ag.attn_qk_norm_rope_append(
                    t[0], t[6], t[7], t[8], t[9], cs, t[10], t[11], t[1], t[2], eps=1e-6),
                    ag.attn_prefill_paged(t[0], t[1], t[2], o, t[3], t[4], t[5], c.chunk, causal=c.causal))
            leg.set_buffers(bind, t, Op)
            leg.host = {k: L[k] for k in keys}
            leg.config = {"num_seqs": cfg.num_seqs, "prefix": cfg.prefix, "chunk": cfg.chunk,
                          "H_q": cfg.H_q, "H_kv": cfg.H_kv, "D": cfg.D, "causal": cfg.causal,
                          "rope_base": W.PROLOGUE.base, "eps": 1e-6,
                          "query_prologue": "inside the prefill kernel" if fused else "separate pass"}
            legs.append(leg)
    if which in ("all", "prefill_paged"):
        cfg = W.CHUNKED_PREFILL
        Qp, kc, vc, cu, skv, tables = W.chunked_prefill_inputs(cfg, seed=0)
        t = [torch.from_numpy(x).cuda() for x in (Qp, kc, vc, cu, skv, tables)]
        Op = torch.empty_like(t[0])
        leg = Leg(cfg.name, "prefill", cfg.flops(), "TFLOP/s", 1)
        leg.set_buffers(lambda t, o, c=cfg: (lambda: ag.attn_prefill_paged(
            t[0], t[1], t[2], o, t[3], t[4], t[5], c.chunk, causal=c.causal)), tuple(t), Op)
        leg.host = {"Q": Qp, "k_cache": kc, "v_cache": vc, "cu_seqlens_q": cu, "seq_lens_kv": skv,
                    "block_tables": tables}
        leg.config = {"num_seqs": cfg.num_seqs, "prefix": cfg.prefix, "chunk": cfg.chunk,
                      "H_q": cfg.H_q, "H_kv": cfg.H_kv, "D": cfg.D, "causal": cfg.causal,
                      "block_size": 16, "num_blocks": int(kc.shape[0])}
        legs.append(leg)
    for cfg, key in ((W.DECODE_MIX, "decode"), (W.DECODE_LONG, "decode_long"), (W.DECODE_GQA8, "decode_gqa8")):
        if which not in ("all", key) and not (key == "decode" and which == "decode_append"):
            continue
        inp = W.decode_inputs(cfg, seed=0)
        t = [torch.from_numpy(x).cuda() for x in (inp.q, inp.k_cache, inp.v_cache,
                                                  inp.block_tables, inp.seq_lens)]
        out = torch.empty_like(t[0])
        leg = Leg(cfg.name, "decode", float(inp.kv_bytes()), "GB/s", 2)
        leg.set_buffers(lambda t, o: (lambda: ag.attn_decode_paged(t[0], t[1], t[2], o, t[3], t[4])),
                        tuple(t), out)
        leg.host = {"q": inp.q, "k_cache": inp.k_cache, "v_cache": inp.v_cache,
                    "block_tables": inp.block_tables, "seq_lens": inp.seq_lens}
        leg.config = {"num_seqs": cfg.num_seqs, "H_q": cfg.H_q, "H_kv": cfg.H_kv, "D": cfg.D,
                      "block_size": cfg.block_size, "seq_len": [cfg.len_lo, cfg.len_hi],
                      "max_blocks_per_seq": cfg.max_blocks_per_seq,
                      "num_blocks": inp.num_blocks, "kv_bytes": inp.kv_bytes()}
        if which != "decode_append":
            legs.append(leg)
        if cfg is W.DECODE_MIX and which in ("all", "decode_append"):
            # one decode step with its KV append: each sequence's new token goes to
            # its last position (rewritten every step, so steps are idempotent)
            N, H_kv = cfg.num_seqs, cfg.H_kv
            Ls = inp.seq_lens.astype(np.int64)
            slots = inp.block_tables[np.arange(N), (Ls - 1) // 16].astype(np.int64) * 16 + (Ls - 1) % 16
            kn = W.normal_fp16(0, 7, (N, H_kv, cfg.D))
            vn = W.normal_fp16(0, 8, (N, H_kv, cfg.D))
            dkn, dvn, dsl = (torch.from_numpy(x).cuda() for x in (kn, vn, slots))
            app_bytes = 2 * kn.nbytes
            leg2 = Leg(cfg.name + "_append", "decode", float(inp.kv_bytes() + app_bytes), "GB/s", 3)
            leg2.set_buffers(lambda t, o: (lambda: ag.attn_decode_paged_append(
                t[0], t[5], t[6], t[1], t[2], o, t[7], t[3], t[4])), tuple(t) + (dkn, dvn, dsl), out)
            leg2.host = dict(leg.host, k_new=kn, v_new=vn, slot_mapping=slots)
            leg2.config = dict(leg.config, append_bytes=app_bytes)
            legs.append(leg2)
    if which in ("all", "prologue"):
        # QK-norm + RoPE + KV append of the prefill workload's 2 x 8192 new tokens:
        # q rotated in place (repeated steps re-normalise it, so values stay bounded),
        # k and v written to a permutation of the cache slots.  Last in the step:
        # the ~100 MB it leaves dirty in L2 are written back during the next
        # (compute-bound) prefill rather than during a bandwidth-bound decode.
        cfg = W.PROLOGUE
        Q, K, V, qw, kw, pos, slots, nb = W.prologue_inputs(cfg, seed=0)
        t = [torch.from_numpy(x).cuda() for x in (Q, K, V, qw, kw, pos, slots)]
        kc = torch.zeros((nb, cfg.H_kv, 16, cfg.D), dtype=torch.float16, device="cuda")
        vc = torch.zeros_like(kc)
        cs = torch.empty((cfg.seq_len, cfg.D), dtype=torch.float32, device="cuda")
        ag.attn_rope_cos_sin_table(cs, cfg.base)
        leg = Leg(cfg.name, "prologue", cfg.bytes(), "GB/s", 1)
        leg.set_buffers(lambda t, o, kc=kc, vc=vc, cs=cs: (lambda: ag.attn_qk_norm_rope_append(
            t[0], t[1], t[2], t[3], t[4], cs, t[5], t[6], kc, vc, eps=1e-6)), tuple(t), t[0])
        leg.out_alias = 0   # q is rotated in place: the step's result is its q
        leg.host = {"Q": Q, "K": K, "V": V, "q_weight": qw, "k_weight": kw, "positions": pos,
                    "slot_mapping": slots}
        leg.config = {"tokens": cfg.tokens, "seq_len": cfg.seq_len, "H_q": cfg.H_q,
                      "H_kv": cfg.H_kv, "D": cfg.D, "rope_base": cfg.base, "eps": 1e-6,
                      "block_size": 16, "num_blocks": nb, "bytes": cfg.bytes()}
        legs.append(leg)
    return legs


def time_device(torch, legs, steps, warmup, dist, use_cuda):
    stream = torch.cuda.current_stream()
    # a buffer larger than L2 (129 MB), rewritten outside the timed events of legs
    # that ask for a cold L2
    flush_buf = torch.empty(256 << 20, dtype=torch.uint8, device="cuda") \
        if any(getattr(leg, "flush", False) for leg in legs) else None
    for _ in range(warmup):
        for leg in legs:
            leg.run()
    torch.cuda.synchronize()
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in legs] for _ in range(steps)]
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    time_device.window = (time.time(), None)
    for s in range(steps):
        for i, leg in enumerate(legs):
            if getattr(leg, "flush", False):
                flush_buf.fill_(s & 0xff)
            ev[s][i][0].record(stream)
            leg.run()
            ev[s][i][1].record(stream)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    wall = time.perf_counter() - t0
    time_device.window = (time_device.window[0], time.time())
    for i, leg in enumerate(legs):
        leg.times = [ev[s][i][0].elapsed_time(ev[s][i][1]) for s in range(steps)]
    return wall


def time_e2e(torch, leg, steps, warmup):
    """Same leg through the public API with pinned host buffers: every step copies
    its inputs host-to-device, makes the C-ABI call and copies its result back, all
    inside the timed region.  Steps are pipelined the way a serving loop would run
    them: two device buffer sets and three streams (copies in, kernels, copies out),
    so the copies of one step overlap the kernels of its neighbours; events keep a
    buffer set from being refilled before its previous step's kernels and result
    copy are done."""
    pinned_in = [torch.from_numpy(np.ascontiguousarray(x)).pin_memory() for x in leg.host.values()]
    pinned_out = [torch.empty(leg.dev_out.shape, dtype=leg.dev_out.dtype).pin_memory() for _ in range(2)]
    second_in = tuple(torch.empty_like(x) for x in leg.dev_in)
    second_out = second_in[leg.out_alias] if leg.out_alias is not None else torch.empty_like(leg.dev_out)
    sets = [(leg.dev_in, leg.dev_out), (second_in, second_out)]
    runs = [leg.bind(ins, out) for ins, out in sets]
    s_in, s_run, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_run = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def step(i):
        b = i % 2
        ins, out = sets[b]
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(ev_run[b])      # its previous kernels have read the inputs
            for h, d in zip(pinned_in, ins):
                d.copy_(h, non_blocking=True)
            ev_in[b].record(s_in)
        with torch.cuda.stream(s_run):
            s_run.wait_event(ev_in[b])
            if i >= 2:
                s_run.wait_event(ev_out[b])     # its previous result has been copied out
            runs[b]()
            ev_run[b].record(s_run)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_run[b])
            pinned_out[b].copy_(out, non_blocking=True)
            ev_out[b].record(s_out)

    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(s_in)
    for i in range(steps):
        step(i)
    s_in.wait_event(ev_out[(steps - 1) % 2])
    b.record(s_in)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    bi = sum(x.numel() * x.element_size() for x in pinned_in)
    bo = pinned_out[0].numel() * pinned_out[0].element_size()
    return {"value": leg.value(ms), "unit": leg.unit, "ms": ms,
            "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
            "pipeline": "2 buffer sets, 3 streams (copy in / kernels / copy out)"}


# ------------------------------------------------------------------ CPU oracle

def cpu_model() -> str:
    try:   # lscpu names Arm cores too (/proc/cpuinfo on Arm has no model name)
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key = line.split(":")[0].strip().lower()
                if key in ("model name", "cpu model", "hardware"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine()


def oracle_sample(seconds: float, seed: int = 0, cfg=None):
    """Time the FP64 oracle on random rows of a causal prefill workload (the
    long one by default) until about `seconds` of CPU time; returns (TFLOP/s,
    rows, wall seconds, threads)."""
    import oracle
    cfg = cfg or W.PREFILL_LONG
    Q, K, V = W.prefill_inputs(cfg, seed=0)
    rng = np.random.default_rng(seed)
    threads = oracle.num_threads()

    def rows(n):
        return np.stack([rng.integers(cfg.B, size=n), rng.integers(cfg.S, size=n),
                         rng.integers(cfg.H_q, size=n)], 1).astype(np.int32)

    def flops(r):  # QK^T and PV over the i+1 allowed keys of each row
        return float(np.sum(4.0 * cfg.D * (r[:, 1].astype(np.float64) + 1)))

    n = 2 * threads
    r = rows(n)
    t = time.perf_counter()
    oracle.prefill_rows(Q, K, V, r, causal=True)
    dt = time.perf_counter() - t
    total_f, total_t, total_n = flops(r), dt, n
    while total_t < seconds:
        n = int(min(max(n, (seconds - total_t) / max(dt, 1e-3) * n * 0.5), 200000)) or 1
        r = rows(n)
        t = time.perf_counter()
        oracle.prefill_rows(Q, K, V, r, causal=True)
        dt = time.perf_counter() - t
        total_f += flops(r)
        total_t += dt
        total_n += n
    return total_f / total_t / 1e12, total_n, total_t, threads


def oracle_decode_sample(seconds: float, seed: int = 0, n_seqs: int = 16):
    """Time the FP64 oracle on the decode mix: `n_seqs` sequences drawn with
    the workload's length distribution, every query head of each, repeated
    until about `seconds`; returns (GB/s of valid K/V bytes, sequences, wall
    seconds, threads)."""
    import oracle
    cfg = W.DECODE_MIX
    small = W.DecodeConfig(cfg.name, n_seqs, cfg.H_q, cfg.H_kv, cfg.D, cfg.block_size,
                           cfg.len_lo, cfg.len_hi, cfg.max_blocks_per_seq)
    d = W.decode_inputs(small, seed=seed)
    total_b, total_t, total_n = 0.0, 0.0, 0
    while total_t < seconds:
        t = time.perf_counter()
        oracle.decode_paged(d.q, d.k_cache, d.v_cache, d.block_tables, d.seq_lens)
        total_t += time.perf_counter() - t
        total_b += d.kv_bytes()
        total_n += n_seqs
    return total_b / total_t / 1e9, total_n, total_t, oracle.num_threads()


def cpu_baseline_extras(seconds: float):
    """Two further oracle figures: the Qwen3-0.6B-shaped prefill on one core,
    and the decode mix on every core (GB/s of K/V)."""
    import oracle
    with oracle.threads(1):
        tf, n, secs, _ = oracle_sample(seconds, cfg=W.PREFILL_QWEN)
    one = {"workload": W.PREFILL_QWEN.name, "value": tf, "unit": "TFLOP/s", "cores": 1,
           "sample": f"{n} random rows (b,i,h), FP64, {secs:.1f} s"}
    gbs, n, secs, threads = oracle_decode_sample(seconds)
    dec = {"workload": W.DECODE_MIX.name, "value": gbs, "unit": "GB/s", "cores": threads,
           "sample": f"{n} sequences drawn with the workload's lengths, all heads, FP64, {secs:.1f} s"}
    return [one, dec]


# ------------------------------------------------------------------ arms

def run_ours(args):
    import torch
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dist = dist_init(world, True)
    import attention_gqa_causal_gb300 as ag
    ag.load()
    legs = build_legs(torch, ag, args.workload)
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.wait_ready()
    wall = time_device(torch, legs, args.steps, args.warmup, dist, True)
    clk = clocks.stop(time_device.window)
    wall = reduce_max(dist, wall, True)
    err = ag.attn_get_device_error(reset=True)
    peaks, peak_src = load_peaks()

    parts = []
    for leg in legs:
        ms = reduce_max(dist, sum(leg.times) / len(leg.times), True)
        val = leg.value(ms) * world
        part = {"workload": leg.name, "value": val, "unit": leg.unit, "ms": ms,
                "ms_min": min(leg.times), "config": leg.config}
        if leg.kind == "prefill":
            peak = peaks["bf16_tflops"]
            part["roofline"] = {"bound": "tensor", "achieved": leg.value(ms), "peak": peak,
                                "unit": "TFLOP/s", "frac": leg.value(ms) / peak,
                                "peak_kind": f"{peak_src} dense bf16 burst (fp16 runs at the same tensor rate)",
                                "traffic": dram_traffic("prefill_kernel", leg.name)}
        else:
            peak = peaks["hbm_gbs"]
            kernel = "qk_norm_rope_kernel" if leg.kind == "prologue" else "decode_mma_kernel"
            part["roofline"] = {"bound": "hbm", "achieved": leg.value(ms), "peak": peak,
                                "unit": "GB/s", "frac": leg.value(ms) / peak,
                                "peak_kind": f"{peak_src} copy bandwidth",
                                "traffic": dram_traffic(kernel, leg.name)}
        parts.append(part)

    e2e = None
    if not args.no_e2e:
        e2e_parts = {}
        for leg in legs:
            e2e_parts[leg.name] = time_e2e(torch, leg, max(2, min(args.steps, 10)), 2)
        head = legs[0].name
        e2e = dict(e2e_parts[head])
        e2e["workload"] = head
        for p in parts:
            p["e2e"] = e2e_parts[p["workload"]]

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        tf, n, secs, threads = oracle_sample(args.cpu_seconds)
        cpu = {"value": tf, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
               "cpu": cpu_model(), "nproc": os.cpu_count(),
               "sample": f"{n} random rows (b,i,h) of {W.PREFILL_LONG.name}, FP64, {secs:.1f} s",
               "also": cpu_baseline_extras(max(1.0, args.cpu_seconds / 5))}

    head = parts[0]
    launches = sum(leg.launches for leg in legs) * args.steps
    line = {
        "metric": METRIC, "value": head["value"], "unit": head["unit"], "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": wall * 1e3 / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16", "data": "synthetic: seeded N(0,1) FP16 "
        "(splitmix64 + Box-Muller), seq_lens uniform, block tables a seeded permutation",
        "config": {"workload": " + ".join(leg.name for leg in legs), **head["config"],
                   "l2": "inputs larger than L2 (129 MB), except the Qwen3-0.6B-shaped prefill: "
                         "L2 flushed (256 MB written) before each of its launches",
                   "parallelism": f"replicated weak scaling x{world}" if world > 1 else "single GPU"},
        "roofline": head["roofline"], "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": launches, "clocks": clk, "device_error": err, "parts": parts,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    secs = max(1.0, args.cpu_seconds / max(1, args.steps + args.warmup) * 3)
    vals = []
    n_tot = 0
    t_tot = 0.0
    threads = 1
    for s in range(args.warmup + args.steps):
        tf, n, t, threads = oracle_sample(secs, seed=s)
        if s >= args.warmup:
            vals.append(tf)
            n_tot += n
            t_tot += t
    val = statistics.mean(vals)
    sample = f"{n_tot} random rows (b,i,h) of {W.PREFILL_LONG.name} over {args.steps} steps, FP64, {t_tot:.1f} s"
    line = {
        "impl": "reference", "metric": METRIC, "value": val, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_tot * 1e3 / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic: seeded N(0,1) FP16 inputs, FP64 CPU oracle",
        "config": {"workload": W.PREFILL_LONG.name, "B": 2, "S": 8192, "H_q": 32, "H_kv": 8,
                   "D": 128, "causal": True},
        "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "cpu": cpu_model(), "nproc": os.cpu_count(), "sample": sample},
        "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=["all", "prefill", "prefill_full", "prefill_paged", "layer", "prologue", "qwen",
                                           "decode", "decode_long", "decode_append", "decode_gqa8"],
                    default="all")
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="CPU time budget of the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
