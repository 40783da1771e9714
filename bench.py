#!/usr/bin/env python
"""Decode-attention benchmark over a 2-/4-bit affine-quantized KV cache on GB300.

Metric: decode-attention µs per call and achieved HBM GB/s (fraction of the
measured peak), INT2 and INT4. One step = one call of lbkv_decode_attn (the
whole hot path: split-KV decode with affine folding and the merge of the
partials, one kernel launch; two when a bf16 window is present) over one batch
of seeded synthetic inputs already resident in HBM. Headline workload: INT2
token-wise K/V, group 128, 32 query / 8 KV heads, head_dim 128, batch 32, 32K
context. The other workloads run as a sweep.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl {lbkv,reference}] [--no-sweep]
       python bench.py --micro   (tensor-core operation rates, bit_kv_cache_split_gb300/micro)
       python bench.py --profile [--bits B] [--batch N] [--ctx T] [--workload NAME] [--steps K] [--warmup W]
(--profile: only eager calls of one workload, for ncu captures)
Under torchrun (N > 1) every rank runs its own replica on its GPU (the path
shards by sequence and KV head with no exchange); rank 0 prints one JSON line.
"""

from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from bit_kv_cache_split_gb300 import inputs  # noqa: E402

METRIC = "decode-attn µs/call and achieved HBM GB/s (% of GB300 peak), INT2/INT4"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0
HEADLINE = dict(batch=32, ctx=32768)


# ------------------------------------------------------------------ bytes

def algorithmic_bytes(wl: inputs.Workload) -> int:
    """Bytes one call must move at minimum: codes, scales, offsets, Q, output, lengths
    (and the bf16 window). Split-workspace traffic is not counted."""
    D, Hkv, g = wl.head_dim, wl.num_kv_heads, wl.group
    total = 0
    for L in wl.lens:
        codes = 2 * L * D * wl.bits // 8
        sz = 0
        for layout in (wl.k_layout, wl.v_layout):
            if layout == inputs.TOKENWISE:
                sz += L * (D // g) * 4
            else:
                sz += math.ceil(L / g) * D * 4
        total += Hkv * (codes + sz)
    total += 2 * wl.batch * wl.num_q_heads * D * 2 + 4 * wl.batch
    if wl.window:
        total += wl.batch * Hkv * wl.window * D * 2 * 2 + 4 * wl.batch
    return total


def measured_hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def source_hash() -> str:
    """Hash of the split-decode kernel's device sources, comments and blank space left out
    (its traffic depends on the code alone: not on comments, the other kernels, the opt-in
    tensor-core kernel or the host entry points)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "bit_kv_cache_split_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        # the split-decode kernel: its header, its instantiations and the device helpers
        if not (f in ("lbkv_decode.cuh", "lbkv_device.cuh") or f.startswith("lbkv_decode_int")):
            continue
        with open(os.path.join(csrc, f)) as fh:
            text = fh.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)  # block comments
        text = re.sub(r"//[^\n]*", " ", text)                # line comments
        code = " ".join(text.split())
        h.update(f.encode() + code.encode())
    return h.hexdigest()[:16]


def profiled_counters(workload: str) -> dict:
    """Counters of one launch of `workload` from a committed ncu summary (DRAM bytes, SASS
    instructions), if it was taken on the current decode-kernel sources; else {}."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            rec = json.load(f).get(workload)
    except (OSError, ValueError):
        return {}
    if not rec or rec.get("source_hash") != source_hash():
        return {}
    return rec


def issue_budget(sm_count: int, sm_mhz, hbm_gbs: float):
    """Lane-slots the GPU can issue per byte streamed at the HBM peak: SMs x 4 schedulers x
    32 lanes x SM clock / bandwidth (the explainer's instruction-budget arithmetic, which
    gives 9.99 for H100 and 4.65 for B200)."""
    if not sm_mhz:
        return None
    return sm_count * 4 * 32 * sm_mhz * 1e6 / (hbm_gbs * 1e9)


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi samples (200 ms) taken while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.samples = []
        self.proc = None
        self.idx = device_index

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200",
                 "-i", str(self.idx)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 8:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        rows = [p for (t, p) in self.samples if t0 <= t <= t1] or [p for (_, p) in self.samples]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(r[0]) for r in rows if num(r[0]) is not None]
        mx = [num(r[1]) for r in rows if num(r[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in rows for k in range(4) if r[4 + k].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max((num(r[2]) or 0.0) for r in rows)}


# ------------------------------------------------------------------ device timing

class Case:
    """Device-resident replicas of one workload plus output and workspace."""

    def __init__(self, wl: inputs.Workload, device, min_footprint=4 * L2_BYTES, max_replicas=256):
        import bit_kv_cache_split_gb300 as pkg

        self.pkg, self.wl = pkg, wl
        self.bytes = algorithmic_bytes(wl)
        r = max(2, math.ceil(min_footprint / max(self.bytes, 1)))
        self.replicas = []
        for i in range(min(r, max_replicas)):
            w = inputs.Workload(**{**wl.__dict__, "seed": wl.seed + 1000 * i})
            self.replicas.append(inputs.generate(w, device))
        self.out = torch.empty((wl.batch, wl.num_q_heads, wl.head_dim), dtype=torch.bfloat16, device=device)
        n = pkg.workspace_bytes(wl.batch, wl.num_q_heads, wl.num_kv_heads, wl.t_cap, wl.bits, wl.k_layout,
                                wl.v_layout, wl.group, window=bool(wl.window))
        self.ws = pkg._binding.alloc_workspace(n, device)
        self.footprint = sum(sum(x.numel() * x.element_size() for x in rep.values()) for rep in self.replicas)

    def call(self, i, stream=None):
        t = self.replicas[i % len(self.replicas)]
        win = {}
        if "k_win" in t:
            win = dict(k_win=t["k_win"], v_win=t["v_win"], win_lens=t["win_lens"])
        self.pkg.decode_attn(t["q"], t["k_codes"], t["k_scale"], t["k_off"], t["v_codes"], t["v_scale"], t["v_off"],
                             t["seq_lens"], bits=self.wl.bits, k_layout=self.wl.k_layout, v_layout=self.wl.v_layout,
                             group=self.wl.group, sm_scale=self.wl.sm_scale, out=self.out, workspace=self.ws,
                             stream=stream, **win)

    def time(self, steps, warmup, barrier=None):
        """Average ms per call over exactly `steps` calls: the calls are captured once in a
        CUDA graph (no host launch overhead between them) and the replay is timed with CUDA
        events on the launching stream. L2 is flushed before the timed replay, and
        consecutive calls read different replicas."""
        for i in range(warmup):
            self.call(i)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            with torch.cuda.graph(graph, stream=side):
                for i in range(steps):
                    self.call(warmup + i)
        torch.cuda.current_stream().wait_stream(side)
        graph.replay()  # untimed: the graph's first launch uploads it
        torch.cuda.synchronize()
        flush = torch.empty(4 * L2_BYTES, dtype=torch.uint8, device=self.out.device)
        flush.zero_()
        del flush
        if barrier:
            barrier()
        torch.cuda.synchronize()
        s = torch.cuda.current_stream()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        graph.replay()
        e1.record(s)
        torch.cuda.synchronize()
        if barrier:
            barrier()
        del graph
        return e0.elapsed_time(e1) / steps

    def free(self):
        self.replicas.clear()
        self.out = self.ws = None


def time_e2e(wl, steps, warmup, device):
    """Same metric through the public API from pinned host buffers: every step copies the
    step's inputs host->device, decodes, and reads the output back. The copies of step i + 1
    (on a copy stream, into the other of two device buffer sets) overlap the decode of step i,
    as a serving loop would run it; the timed region still holds every step's copies."""
    import bit_kv_cache_split_gb300 as pkg

    host = {k: v.pin_memory() for k, v in inputs.generate(wl, "cpu").items()}
    bufs = [{k: torch.empty_like(v, device=device) for k, v in host.items()} for _ in range(2)]
    out_h = torch.empty((wl.batch, wl.num_q_heads, wl.head_dim), dtype=torch.bfloat16).pin_memory()
    out_d = torch.empty_like(out_h, device=device)
    n = pkg.workspace_bytes(wl.batch, wl.num_q_heads, wl.num_kv_heads, wl.t_cap, wl.bits, wl.k_layout, wl.v_layout,
                            wl.group, window=bool(wl.window))
    ws = pkg._binding.alloc_workspace(n, device)
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = out_h.numel() * out_h.element_size()
    compute = torch.cuda.current_stream()
    copier = torch.cuda.Stream()
    ready = [torch.cuda.Event(), torch.cuda.Event()]  # a buffer set holds its step's inputs
    done = [torch.cuda.Event(), torch.cuda.Event()]   # the decode that read a buffer set ended

    def copy_in(i, start=None):
        b = i % 2
        with torch.cuda.stream(copier):
            if start is not None:
                copier.wait_event(start)
            copier.wait_event(done[b])
            for k in host:
                bufs[b][k].copy_(host[k], non_blocking=True)
            ready[b].record(copier)

    def decode(i):
        b = i % 2
        dev = bufs[b]
        compute.wait_event(ready[b])
        win = {}
        if "k_win" in dev:
            win = dict(k_win=dev["k_win"], v_win=dev["v_win"], win_lens=dev["win_lens"])
        pkg.decode_attn(dev["q"], dev["k_codes"], dev["k_scale"], dev["k_off"], dev["v_codes"], dev["v_scale"],
                        dev["v_off"], dev["seq_lens"], bits=wl.bits, k_layout=wl.k_layout, v_layout=wl.v_layout,
                        group=wl.group, out=out_d, workspace=ws, **win)
        done[b].record(compute)
        out_h.copy_(out_d, non_blocking=True)

    def run(n_steps, start=None):
        copy_in(0, start)
        for i in range(n_steps):
            if i + 1 < n_steps:
                copy_in(i + 1)
            decode(i)

    run(warmup)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(compute)
    run(steps, start=e0)
    e1.record(compute)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    return ms, h2d, d2h


# ------------------------------------------------------------------ CPU oracle

def oracle_throughput(wl, target_s=12.0, max_units=None, threads=0):
    """The fp64 oracle on a bounded sample of `wl`: whole (sequence, KV head) units, all
    their query heads. Returns (GB/s of algorithmic bytes, seconds, units, threads, rows)."""
    import oracle

    oracle.build()
    hq = wl.hq_per_kv
    per_unit = max(1, algorithmic_bytes(wl) // max(1, wl.batch * wl.num_kv_heads))

    def sample(n_units):
        b_needed = math.ceil(n_units / wl.num_kv_heads)
        w = inputs.Workload(**{**wl.__dict__, "batch": b_needed,
                               "seq_lens": wl.lens[:b_needed] if not isinstance(wl.seq_lens, int) else wl.seq_lens})
        t = inputs.generate(w, "cpu")
        x = oracle.inputs_from_tensors(t, bits=w.bits, k_layout=w.k_layout, v_layout=w.v_layout, group=w.group,
                                       Hkv=w.num_kv_heads, T_cap=w.t_cap, sm_scale=w.sm_scale)
        rows = [(u // w.num_kv_heads, (u % w.num_kv_heads) * hq + i) for u in range(n_units) for i in range(hq)]
        nthreads = threads or os.cpu_count() or 1
        t0 = time.perf_counter()
        oracle.decode_ref(x, rows=rows, n_threads=nthreads)
        return time.perf_counter() - t0, min(nthreads, len(rows)), len(rows)

    cores = os.cpu_count() or 1
    n = max(1, cores // hq)
    if max_units is not None:
        n = min(n, max_units)
    dt, used, rows = sample(n)
    total_units = wl.batch * wl.num_kv_heads
    if dt < target_s / 4:
        cap = total_units if max_units is None else max_units
        n2 = min(cap, max(n, int(n * target_s / max(dt, 1e-3))))
        if n2 > n:
            n = n2
            dt, used, rows = sample(n)
    return n * per_unit / dt / 1e9, dt, n, used, rows


# ------------------------------------------------------------------ main

def sweep_workloads():
    ws = []
    for b in inputs.BATCHES:
        for ctx in inputs.CONTEXTS:
            ws.append(inputs.decode_int2(b, ctx))
    for b in inputs.BATCHES:
        for ctx in inputs.CONTEXTS:
            ws.append(inputs.decode_int4(b, ctx))
    for bits in (2, 4):  # all four K/V layout pairs on the same ragged lengths
        for kl, vl in ((0, 0), (1, 0), (0, 1), (1, 1)):
            ws.append(inputs.mixed_layout(bits, kl, vl))
    for b in (1, 16, 64):
        ws.append(inputs.long_context(b))
    for g in (32, 64, 128):
        for hq in (1, 2, 4, 8):
            ws.append(inputs.long_context(16, group=g, hq_per_kv=hq))
    return ws


def run_sweep(device, peak):
    import bit_kv_cache_split_gb300 as pkg

    rows = []
    for wl in sweep_workloads():
        try:
            case = Case(wl, device)
            ms = case.time(steps=20, warmup=3)
        except pkg.LbkvError as e:
            rows.append({"workload": wl.name, "unsupported": str(e)})
            torch.cuda.empty_cache()
            continue
        gbs = case.bytes / (ms * 1e-3) / 1e9
        row = {"workload": wl.name, "us_per_call": round(ms * 1e3, 2), "gbs": round(gbs, 1),
               "frac": round(gbs / peak, 3), "bytes": case.bytes,
               "launch": pkg.decode_launch_info(wl.batch, wl.num_q_heads, wl.num_kv_heads, wl.t_cap, wl.bits,
                                                wl.k_layout, wl.v_layout, wl.group, window=bool(wl.window))}
        rec = profiled_counters(wl.name)
        if rec:  # ncu counters of this workload on the current kernel sources
            row["traffic"] = rec["dram_bytes_per_launch"]
            row["lane_slots_per_byte"] = round(32 * rec["inst_per_launch"] / case.bytes, 2)
        if wl.window:
            # scale/offset operations per stored value under folding: 2 h_q / g (explainer,
            # break-even paragraph: folding wins while this is below 1, i.e. g > 2 h_q)
            row["fold_ops_per_value"] = round(2 * wl.hq_per_kv / wl.group, 4)
        rows.append(row)
        case.free()
        torch.cuda.empty_cache()
    return rows


def append_bytes(B, Hkv, bits, group, k_layout, v_layout) -> float:
    """Algorithmic bytes of one lbkv_append call, a group's flush spread over its calls.

    Token-wise sides: the new K/V read, its codes and scales/offsets written, the lengths
    read and written. With a channel-wise side: the token written to the window; every
    `group`-th call reads the window's group of tokens and writes its codes and scales."""
    D = 128
    new = B * Hkv * 2 * D * 2
    codes = B * Hkv * 2 * D * bits // 8
    if k_layout == 0 and v_layout == 0:
        return new + codes + B * Hkv * 2 * (D // group) * 2 * 2 + B * 4 * 2
    sz = 0
    for layout in (k_layout, v_layout):
        sz += B * Hkv * (group * (D // group) * 2 * 2 if layout == 0 else D * 2 * 2)  # per group of tokens
    flush = B * Hkv * 2 * group * D * 2 + group * codes + sz
    return new + new + flush / group + B * 4 * 4  # read + window write, flush share, both lengths


def time_append(device, peak, calls=256):
    """µs per lbkv_append call (one new token for every sequence and KV head), B = 32,
    8 KV heads: a CUDA graph of `calls` appends, replayed once untimed and once timed."""
    import bit_kv_cache_split_gb300 as pkg

    rows = []
    for bits, kl, vl in ((2, 0, 0), (4, 0, 0), (2, 1, 0)):
        B, Hkv, g, D = 32, 8, 128, 128
        T = 2 * calls
        tag = {(0, 0): "tokenwise", (1, 0): "cwK-twV"}[(kl, vl)]
        name = f"append-int{bits}-{tag}-b{B}-kv{Hkv}"
        gen = torch.Generator(device=device).manual_seed(7)
        k_new = torch.randn((B, Hkv, D), generator=gen, device=device).to(torch.bfloat16)
        v_new = torch.randn((B, Hkv, D), generator=gen, device=device).to(torch.bfloat16)
        sides = []
        for layout in (kl, vl):
            sshape = (B, Hkv, T, D // g) if layout == 0 else (B, Hkv, T // g, D)
            sides.append((torch.zeros((B, Hkv, T, D * bits // 8), dtype=torch.uint8, device=device),
                          torch.zeros(sshape, dtype=torch.float16, device=device),
                          torch.zeros(sshape, dtype=torch.float16, device=device)))
        lens = torch.zeros((B,), dtype=torch.int32, device=device)
        kw = {}
        if kl or vl:
            kw = dict(k_win=torch.zeros((B, Hkv, 128, D), dtype=torch.bfloat16, device=device),
                      v_win=torch.zeros((B, Hkv, 128, D), dtype=torch.bfloat16, device=device),
                      win_lens=torch.zeros((B,), dtype=torch.int32, device=device))
        ws = torch.zeros(64, dtype=torch.int32, device=device)

        def one():
            pkg.append(k_new, v_new, lens, *sides[0], *sides[1], bits=bits, k_layout=kl, v_layout=vl, group=g,
                       workspace=ws, **kw)

        one()  # loads the kernel before capture
        torch.cuda.synchronize()
        lens.zero_()
        if kw:
            kw["win_lens"].zero_()
        side = torch.cuda.Stream(device)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            with torch.cuda.graph(graph, stream=side):
                for _ in range(calls):
                    one()
        torch.cuda.synchronize()
        graph.replay()  # untimed
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        graph.replay()
        e1.record()
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / calls
        ok = int(lens[0].item()) == 2 * calls and pkg.device_status(ws) == 0
        nbytes = append_bytes(B, Hkv, bits, g, kl, vl)
        gbs = nbytes / (us * 1e-6) / 1e9
        rows.append({"workload": name, "us_per_call": round(us, 2), "gbs": round(gbs, 1), "frac": round(gbs / peak, 4),
                     "bytes": int(nbytes), "lengths_ok": ok})
        del graph
        torch.cuda.empty_cache()
    return rows


def time_bf16(device, peak, int2_us, calls=5):
    """The BF16 comparator (lbkv_decode_bf16) on the headline's shape (batch 32, 32K context,
    32q/8kv, head_dim 128) over a bf16 cache (4.3 GB, far larger than L2): a CUDA graph of
    `calls` calls, replayed once untimed and once timed."""
    import bit_kv_cache_split_gb300 as pkg

    B, Hq, Hkv, T, D = HEADLINE["batch"], 32, 8, HEADLINE["ctx"], 128
    gen = torch.Generator(device=device).manual_seed(11)
    q = torch.randn((B, Hq, D), generator=gen, device=device, dtype=torch.bfloat16)
    k = torch.randn((B, Hkv, T, D), generator=gen, device=device, dtype=torch.bfloat16)
    v = torch.randn((B, Hkv, T, D), generator=gen, device=device, dtype=torch.bfloat16)
    lens = torch.full((B,), T, dtype=torch.int32, device=device)
    out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=device)
    d = pkg._binding.make_desc(B, Hq, Hkv, T, D)
    ws = torch.zeros(pkg._binding.load().lbkv_bf16_workspace_bytes(ctypes.byref(d)), dtype=torch.uint8, device=device)
    for _ in range(2):
        pkg.decode_bf16(q, k, v, lens, out=out, workspace=ws)
    torch.cuda.synchronize()
    side = torch.cuda.Stream(device)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            for _ in range(calls):
                pkg.decode_bf16(q, k, v, lens, out=out, workspace=ws)
    torch.cuda.synchronize()
    graph.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    graph.replay()
    e1.record()
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / calls
    nbytes = B * Hkv * T * D * 2 * 2 + 2 * B * Hq * D * 2 + B * 4
    gbs = nbytes / (us * 1e-6) / 1e9
    status = pkg.device_status(ws)
    del graph, k, v
    torch.cuda.empty_cache()
    return {"workload": f"bf16-b{B}-ctx{T}", "us_per_call": round(us, 2), "gbs": round(gbs, 1),
            "frac": round(gbs / peak, 4), "bytes": nbytes, "int2_speedup": round(us / int2_us, 2),
            "device_status": status}


def time_paged(device, peak, contiguous_us, page_tokens=128, calls=20):
    """The headline workload (INT2 token-wise, batch 32, 32K context) stored in a paged
    cache: pools of `page_tokens`-token pages in shuffled order behind a page table. Two
    replicas alternate (each larger than L2); a CUDA graph of `calls` calls is replayed
    once untimed and, after an L2 flush, once timed."""
    import bit_kv_cache_split_gb300 as pkg

    wl = inputs.decode_int2(HEADLINE["batch"], HEADLINE["ctx"])
    reps = []
    for i in range(2):
        w = inputs.Workload(**{**wl.__dict__, "seed": wl.seed + 1000 * i})
        t = inputs.generate(w, device)
        table, n_pages = inputs.page_table(w.lens, page_tokens, w.t_cap // page_tokens, seed=40 + i)
        pool = {k: inputs.to_pages(t[k], table, n_pages, page_tokens)
                for k in ("k_codes", "k_scale", "k_off", "v_codes", "v_scale", "v_off")}
        reps.append((t["q"], pool, t["seq_lens"], table.to(device)))
        del t
    n = pkg.workspace_bytes(wl.batch, wl.num_q_heads, wl.num_kv_heads, wl.t_cap, wl.bits, wl.k_layout,
                            wl.v_layout, wl.group)
    ws = pkg._binding.alloc_workspace(n, device)
    out = torch.empty((wl.batch, wl.num_q_heads, wl.head_dim), dtype=torch.bfloat16, device=device)

    def call(i):
        q, c, lens, table = reps[i % 2]
        pkg.decode_attn(q, c["k_codes"], c["k_scale"], c["k_off"], c["v_codes"], c["v_scale"], c["v_off"], lens,
                        bits=2, group=128, page_table=table, max_seq_len=wl.t_cap, out=out, workspace=ws)

    for i in range(3):
        call(i)
    torch.cuda.synchronize()
    side = torch.cuda.Stream(device)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            for i in range(calls):
                call(i)
    torch.cuda.synchronize()
    graph.replay()
    torch.cuda.synchronize()
    flush = torch.empty(4 * L2_BYTES, dtype=torch.uint8, device=device)
    flush.zero_()
    del flush
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    graph.replay()
    e1.record()
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / calls
    nbytes = algorithmic_bytes(wl) + wl.batch * (wl.t_cap // page_tokens) * 4  # + the page table
    gbs = nbytes / (us * 1e-6) / 1e9
    status = pkg.device_status(ws)
    del graph, reps
    torch.cuda.empty_cache()
    return {"workload": f"{wl.name}-paged{page_tokens}", "us_per_call": round(us, 2), "gbs": round(gbs, 1),
            "frac": round(gbs / peak, 4), "bytes": nbytes, "paged_over_contiguous": round(us / contiguous_us, 3),
            "device_status": status}


def time_rotation(device, peak, contiguous_us, calls=20):
    """A cache stored rotated: the headline workload decoded with both rotation flags (the
    query rotated in the prologue, the output rotated back at the end), and lbkv_rotate over
    the rows of one bf16 K side of the headline (batch 32, 8 KV heads, 32K tokens: 2.1 GB)."""
    import bit_kv_cache_split_gb300 as pkg

    wl = inputs.decode_int2(HEADLINE["batch"], HEADLINE["ctx"])
    reps = [inputs.generate(inputs.Workload(**{**wl.__dict__, "seed": wl.seed + 1000 * i}), device) for i in range(2)]
    n = pkg.workspace_bytes(wl.batch, wl.num_q_heads, wl.num_kv_heads, wl.t_cap, wl.bits, wl.k_layout,
                            wl.v_layout, wl.group)
    ws = pkg._binding.alloc_workspace(n, device)
    out = torch.empty((wl.batch, wl.num_q_heads, wl.head_dim), dtype=torch.bfloat16, device=device)
    keys = ("k_codes", "k_scale", "k_off", "v_codes", "v_scale", "v_off")

    def graph_time(call, n_calls):
        for i in range(3):
            call(i)
        torch.cuda.synchronize()
        side = torch.cuda.Stream(device)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            with torch.cuda.graph(graph, stream=side):
                for i in range(n_calls):
                    call(i)
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        flush = torch.empty(4 * L2_BYTES, dtype=torch.uint8, device=device)
        flush.zero_()
        del flush
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        graph.replay()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1e3 / n_calls

    def decode(i):
        t = reps[i % 2]
        pkg.decode_attn(t["q"], *[t[k] for k in keys], t["seq_lens"], bits=2, group=128, rotation=3, out=out,
                        workspace=ws)

    us = graph_time(decode, calls)
    status = pkg.device_status(ws)
    del reps
    torch.cuda.empty_cache()
    x = torch.randn((wl.batch * wl.num_kv_heads * wl.t_cap, 128), device=device, dtype=torch.bfloat16)
    y = torch.empty_like(x)
    rot_us = graph_time(lambda i: pkg.rotate(x, out=y), 5)
    rot_bytes = 2 * x.numel() * 2
    del x, y
    torch.cuda.empty_cache()
    return {"workload": f"{wl.name}-rotated", "us_per_call": round(us, 2), "rotated_over_plain": round(us / contiguous_us, 3),
            "device_status": status,
            "rotate": {"rows": wl.batch * wl.num_kv_heads * wl.t_cap, "us_per_call": round(rot_us, 2),
                       "gbs": round(rot_bytes / (rot_us * 1e-6) / 1e9, 1),
                       "frac": round(rot_bytes / (rot_us * 1e-6) / 1e9 / peak, 4), "bytes": rot_bytes}}


def time_pack(device, peak, calls=5):
    """lbkv_pack (the prefill quantizer) of one bf16 side of the headline (batch 32, 8 KV heads,
    32K tokens: 2.1 GB) into INT2 g128 codes, token-wise and channel-wise."""
    import bit_kv_cache_split_gb300 as pkg

    B, Hkv, T = HEADLINE["batch"], 8, HEADLINE["ctx"]
    x = torch.randn((B, Hkv, T, 128), device=device, dtype=torch.bfloat16)
    lens = torch.full((B,), T, dtype=torch.int32, device=device)
    rows = []
    for layout in (0, 1):
        codes, scale, off = pkg.pack(x, lens, bits=2, layout=layout, group=128)
        for _ in range(2):
            pkg.pack(x, lens, bits=2, layout=layout, group=128, codes=codes, scale=scale, off=off)
        torch.cuda.synchronize()
        side = torch.cuda.Stream(device)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            with torch.cuda.graph(graph, stream=side):
                for _ in range(calls):
                    pkg.pack(x, lens, bits=2, layout=layout, group=128, codes=codes, scale=scale, off=off)
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        graph.replay()
        e1.record()
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / calls
        nbytes = x.numel() * 2 + codes.numel() + 2 * scale.numel() * 2
        rows.append({"workload": f"pack-int2-{'channelwise' if layout else 'tokenwise'}-b{B}-ctx{T}",
                     "us_per_call": round(us, 2), "gbs": round(nbytes / (us * 1e-6) / 1e9, 1),
                     "frac": round(nbytes / (us * 1e-6) / 1e9 / peak, 4), "bytes": nbytes})
        del graph, codes, scale, off
    del x
    torch.cuda.empty_cache()
    return rows


def time_batch1_launches(device, peak, launches=200):
    """Per-launch CUDA-event times of INT2 token-wise decode at batch 1, 32K context (eager
    launches, each bracketed by its own events, replicas rotated so that the cache is read
    from HBM): median, 10th and 90th percentiles."""
    wl = inputs.decode_int2(1, HEADLINE["ctx"])
    case = Case(wl, device)
    for i in range(10):
        case.call(i)
    torch.cuda.synchronize()
    s = torch.cuda.current_stream()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(launches)]
    for i, (a, b) in enumerate(ev):
        a.record(s)
        case.call(i)
        b.record(s)
    torch.cuda.synchronize()
    us = sorted(a.elapsed_time(b) * 1e3 for a, b in ev)
    med = statistics.median(us)
    gbs = case.bytes / (med * 1e-6) / 1e9
    case.free()
    torch.cuda.empty_cache()
    return {"workload": wl.name, "launches": launches, "median_us": round(med, 2),
            "p10_us": round(us[len(us) // 10], 2), "p90_us": round(us[(9 * len(us)) // 10], 2),
            "gbs_at_median": round(gbs, 1), "frac_at_median": round(gbs / peak, 4), "bytes": case.bytes}


def quantization_error(device, units=((0, 0), (3, 5), (7, 7))):
    """Quantize-then-decode at the INT4 decode shape (batch 8, 8 KV heads, 32 query heads,
    32K context): bf16 K/V ~ N(0, 1) through lbkv_pack (token-wise, g128) and
    lbkv_decode_attn, compared on sampled (sequence, KV head) units with attention over the
    unquantized bf16 K/V computed in fp64 (torch). This is the error of 4-bit quantization
    itself on Gaussian data; the explainer's accuracy paragraph quotes an L2 distance of about
    0.5-0.6 for INT2 on the paper's own stress test, a different input."""
    import bit_kv_cache_split_gb300 as pkg

    B, Hkv, Hq, T, g = 8, 8, 32, HEADLINE["ctx"], 128
    hq = Hq // Hkv
    rows = []
    for bits in (4, 2):
        k, lens = inputs.generate_pack_source(B, Hkv, T, seed=2, device=device)
        v, _ = inputs.generate_pack_source(B, Hkv, T, seed=12, device=device)
        q = torch.randn((B, Hq, 128), generator=torch.Generator().manual_seed(22)).to(torch.bfloat16).to(device)
        kc, ks, kz = pkg.pack(k, lens, bits=bits, layout=0, group=g)
        vc, vs, vz = pkg.pack(v, lens, bits=bits, layout=0, group=g)
        out = pkg.decode_attn(q, kc, ks, kz, vc, vs, vz, lens, bits=bits, group=g).double()
        num = den = 0.0
        mx = 0.0
        for b, kvh in units:
            qq = q[b, kvh * hq:(kvh + 1) * hq].double()
            kk, vv = k[b, kvh].double(), v[b, kvh].double()
            p = torch.softmax((qq @ kk.T) / math.sqrt(128.0), dim=-1)
            ref = p @ vv
            d = out[b, kvh * hq:(kvh + 1) * hq] - ref
            num += float((d * d).sum())
            den += float((ref * ref).sum())
            mx = max(mx, float(d.abs().max()))
        rows.append({"workload": f"packed-int{bits}-tokenwise-b{B}-ctx{T}", "bits": bits,
                     "units": [list(u) for u in units], "rel_l2_vs_unquantized": round(math.sqrt(num / den), 4),
                     "l2_vs_unquantized": round(math.sqrt(num / len(units)), 4),
                     "max_abs_vs_unquantized": round(mx, 4)})
        del k, v, kc, vc, ks, kz, vs, vz
        torch.cuda.empty_cache()
    return rows


def run_micro():
    """Builds and runs the tensor-core microbenchmarks under bit_kv_cache_split_gb300/micro
    (one JSON line per measurement):
    - tc_rates.cu: cycles per tcgen05 product (kind::f8f6f4, M = 128, N = 16..256, A in tensor
      memory) and per tensor-memory store and load, with 1, 4 and 16 warps per SM;
    - mma_sync_rates.cu: SM cycles per warp-level product (f16 m16n8k16, e4m3 and u8 x s8
      m16n8k32, loop-variant A operands) with 4, 8 and 16 warps per SM."""
    from bit_kv_cache_split_gb300 import build as libbuild

    os.makedirs(libbuild.BUILD, exist_ok=True)
    for name in ("tc_rates", "mma_sync_rates"):
        src = os.path.join(ROOT, "bit_kv_cache_split_gb300", "micro", name + ".cu")
        exe = os.path.join(libbuild.BUILD, name)
        subprocess.run([libbuild.nvcc(), *libbuild.ARCH, "-O2", src, "-o", exe], check=True)
        r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
        sys.stdout.write(r.stdout)
        if r.returncode != 0:
            raise SystemExit(f"microbenchmark {name} failed: {r.stderr.strip()}")


def max_over_ranks(ms: float, world: int, device=None) -> float:
    """The slowest rank's time: every rank's timed region is one step of its own replica,
    and the job is done when the last one is (weak scaling, one process per GPU)."""
    if world <= 1:
        return ms
    import torch.distributed as dist

    t = torch.tensor([ms], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(step_bytes: int, ms: float, world: int) -> float:
    """Whole-job GB/s: all ranks' algorithmic bytes over the slowest rank's time."""
    return world * step_bytes / (ms * 1e-3) / 1e9


def dist_info():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def reference_arm(args, world, rank):
    """The CPU oracle as the reference arm, timed on the host cores."""
    if rank != 0:
        return
    wl = inputs.decode_int2(**HEADLINE)
    hq = wl.hq_per_kv
    cores = os.cpu_count() or 1
    units = max(1, cores // hq)
    vals, secs, used = [], [], 1
    for i in range(args.warmup + args.steps):
        gbs, dt, n, used, rows = oracle_throughput(wl, target_s=0.0, max_units=units)
        if i >= args.warmup:
            vals.append(gbs)
            secs.append(dt)
    value = statistics.mean(vals) if vals else 0.0
    ms = statistics.mean(secs) * 1e3 if secs else 0.0
    sample = f"{units} of {wl.batch * wl.num_kv_heads} (sequence, KV head) units of {wl.name}, all {hq} query heads"
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": wl.name, "batch": wl.batch, "ctx": HEADLINE["ctx"], "q_heads": wl.num_q_heads,
                       "kv_heads": wl.num_kv_heads, "head_dim": wl.head_dim, "bits": wl.bits, "group": wl.group,
                       "layout": "token-wise K / token-wise V", "sample": sample},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": used, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="lbkv", choices=["lbkv", "reference"])
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--profile", action="store_true", help="eager calls of one workload only (for ncu)")
    ap.add_argument("--bits", type=int, default=2)
    ap.add_argument("--batch", type=int, default=HEADLINE["batch"])
    ap.add_argument("--ctx", type=int, default=HEADLINE["ctx"])
    ap.add_argument("--workload", default=None, help="--profile: a sweep workload by name instead")
    ap.add_argument("--micro", action="store_true",
                    help="the tensor-core microbenchmark (tcgen05 product, TMEM store and load rates) only")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    world, rank, local = dist_info()

    if args.impl == "reference":
        reference_arm(args, world, rank)
        return
    if args.micro:
        run_micro()
        return

    import bit_kv_cache_split_gb300 as pkg

    pkg.build.build()
    pkg.load()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    barrier = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=device)
        barrier = dist.barrier

    if args.profile:
        wl = (inputs.decode_int2 if args.bits == 2 else inputs.decode_int4)(args.batch, args.ctx)
        if args.workload:
            named = {w.name: w for w in sweep_workloads()}
            if args.workload not in named:
                raise SystemExit(f"unknown workload {args.workload}; one of {sorted(named)}")
            wl = named[args.workload]
        case = Case(wl, device, min_footprint=0)
        for i in range(args.warmup + args.steps):
            case.call(i)
        torch.cuda.synchronize()
        print(json.dumps({"profile": wl.name, "calls": args.warmup + args.steps, "bytes_per_call": case.bytes,
                          "replicas": len(case.replicas)}), flush=True)
        return

    peak, peak_kind = measured_hbm_peak()
    wl = inputs.decode_int2(**HEADLINE)
    case = Case(wl, device)
    sampler = ClockSampler(local)
    sampler.start()
    t_pre = time.time()
    end = time.time() + 1.0  # untimed load so that clock samples fall under load
    i = 0
    while time.time() < end:
        case.call(i)
        i += 1
        if i % 64 == 0:
            torch.cuda.synchronize()
    torch.cuda.synchronize()
    ms = case.time(args.steps, args.warmup, barrier)
    t_end = time.time()
    time.sleep(0.3)
    sampler.stop()
    ms = max_over_ranks(ms, world, device)
    status = pkg.device_status(case.ws)
    footprint = case.footprint
    n_rep = len(case.replicas)
    case.free()
    torch.cuda.empty_cache()

    step_bytes = algorithmic_bytes(wl)
    value = job_throughput(step_bytes, ms, world)
    achieved = step_bytes / (ms * 1e-3) / 1e9
    clocks = sampler.summary(t_pre, t_end)

    e2e_ms, h2d, d2h = time_e2e(wl, max(3, min(args.steps, 20)), 2, device)
    e2e_ms = max_over_ranks(e2e_ms, world, device)
    e2e_val = job_throughput(step_bytes, e2e_ms, world)

    sweep = append = bf16 = paged = rotation = pack = batch1 = quant = None
    if not args.no_sweep and rank == 0:
        batch1 = time_batch1_launches(device, peak)
        quant = quantization_error(device)
        sweep = run_sweep(device, peak)
        append = time_append(device, peak)
        bf16 = time_bf16(device, peak, ms * 1e3)
        paged = time_paged(device, peak, ms * 1e3)
        rotation = time_rotation(device, peak, ms * 1e3)
        pack = time_pack(device, peak)

    cpu = None
    if rank == 0 and not args.no_cpu:
        gbs, dt, n, used, rows = oracle_throughput(wl, target_s=12.0)
        cpu = {"value": round(gbs, 4), "unit": "GB/s", "cores": used, "kind": "oracle",
               "sample": f"{n} of {wl.batch * wl.num_kv_heads} (sequence, KV head) units of {wl.name} "
                         f"({rows} query rows, {dt:.1f} s), generated on the host with the same recipe"}

    counters = profiled_counters(wl.name)
    lane_slots = None
    if counters.get("inst_per_launch"):
        lane_slots = round(counters["inst_per_launch"] * 32 / step_bytes, 3)
    sm_count = torch.cuda.get_device_properties(device).multi_processor_count
    budget = issue_budget(sm_count, clocks.get("sm_mhz"), peak)

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms, 5), "us_per_call": round(ms * 1e3, 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16 x f16 -> f32",
            "data": "synthetic (seeded; codes uniform, s~U[0.01,0.1], z~U[-0.2,0.2], Q~N(0,1) bf16)",
            "config": {"workload": wl.name, "batch": wl.batch, "ctx": HEADLINE["ctx"], "q_heads": wl.num_q_heads,
                       "kv_heads": wl.num_kv_heads, "head_dim": wl.head_dim, "bits": wl.bits, "group": wl.group,
                       "layout": "token-wise K / token-wise V", "parallelism": f"replicas x{world}",
                       "l2": f"inputs larger than L2: {n_rep} rotating replicas, {footprint / 1e9:.2f} GB, "
                             f"L2 flushed before the timed graph replay"},
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(achieved / peak, 4), "traffic": counters.get("dram_bytes_per_launch"),
                         "peak_kind": f"{peak_kind} copy bandwidth", "kernel": "split_decode_kernel INT2 token-wise",
                         "bytes_per_launch": step_bytes,
                         "lane_slots_per_byte": lane_slots,
                         "issue_budget": None if budget is None else round(budget, 3),
                         "issue_budget_how": "SMs x 4 schedulers x 32 lanes x median sampled SM clock / peak",
                         "counters_from": counters.get("capture")},
            "clocks": clocks,
            "e2e": {"value": round(e2e_val, 1), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4)},
            "gpu_launches": args.steps,
            "device_status": status,
            "cpu_baseline": cpu,
            "batch1_launches": batch1,
            "quantization_error": quant,
            "sweep": sweep,
            "append": append,
            "bf16_comparator": bf16,
            "paged": paged,
            "rotation": rotation,
            "pack": pack,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
