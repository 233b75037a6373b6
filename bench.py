"""Benchmark: decode-attention effective HBM GB/s and query-heads/s on GB300.

One step = one fused decode call (split-K kernel + combine) over one batch of
synthetic input of the chosen workload (default: the largest one that fits one
GPU, the large-batch workload B=256 H=40 D=128 S=8192 current_pos=8191 with
outlier key channels, 40 GiB of K+V).  Prints ONE JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                  [--impl ours|reference] [--no-sweep] [--cpu-seconds T]

Timing: W untimed warm-up steps, a ~1 s untimed load soak (so clocks settle and
can be sampled), then exactly K steps bracketed by a barrier and
torch.cuda.synchronize() with CUDA events on the launching stream; max over
ranks.  Workloads whose K/V fit in L2 rotate through enough independent input
sets that their total exceeds 4x L2, so no step reads inputs left in L2 by the
previous one.  N > 1 runs one independent replica per GPU (weak scaling): the
path shards by sequence with no data exchange.

--impl reference times the CPU oracle (the plain fp64 restatement of the
method) on this host's cores, on the same workload, metric and unit; each step
is one pass over a bounded sample of the workload's sequences (same recipe).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from token_decode_attention_gb300.workloads import (  # noqa: E402
    WORKLOADS, algorithmic_bytes, draw_current_pos, make_inputs)

METRIC = "decode-attention effective HBM GB/s (% of GB300 peak) and query-heads/s"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
GB300_L2_BYTES = 129 * 2**20  # used when no device is visible
# Sequences of a workload the CPU oracle takes per pass when the whole workload
# would take it more than a few seconds (the oracle streams ~6 GB/s): 16 of the
# outlier workload's 256 sequences are 2.7 GB.
CPU_SAMPLE_SEQUENCES = {"outlier": 16}


def input_sets(kv_bytes: int, l2_bytes: int) -> int:
    """Independent input sets a step rotates through so that no step reads inputs
    left in L2 by the previous one: one when K+V alone exceed 4x L2."""
    return 1 if kv_bytes >= 4 * l2_bytes else min(4096, math.ceil(4 * l2_bytes / kv_bytes) + 1)


def l2_note(kv_bytes: int, l2_bytes: int) -> str:
    n = input_sets(kv_bytes, l2_bytes)
    if n == 1:
        return f"inputs larger than L2 ({kv_bytes / 2**30:.2f} GiB K+V)"
    return f"rotating {n} input sets, {n * kv_bytes / 2**30:.2f} GiB K+V in total (> 4x L2)"


def workload_config(w, world: int, l2_bytes: int) -> dict:
    """The `config` object of the JSON line: the workload only, identical for
    both arms (the kernel plan is reported beside it)."""
    return {"workload": f"{w.name}: {w.description}", "batch": w.batch,
            "n_heads": w.n_heads, "head_dim": w.head_dim, "seq_len": w.seq_len,
            "current_pos": "per-sequence" if w.current_pos is None else w.current_pos,
            "l2": l2_note(w.kv_bytes(), l2_bytes), "parallelism": f"replicas x{world}"}


def device_l2_bytes() -> int:
    try:
        if torch.cuda.is_available():
            props = torch.cuda.get_device_properties(torch.cuda.current_device())
            return int(getattr(props, "L2_cache_size", 0) or GB300_L2_BYTES)
    except Exception:
        pass
    return GB300_L2_BYTES


def log(*a):
    print(*a, file=sys.stderr, flush=True)


# ------------------------------------------------------------------ helpers

def hbm_peak() -> tuple[float, str]:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# the sources of the decode call whose DRAM traffic profiles/ncu_traffic.json records
DECODE_SOURCES = ("decode_kernel.cuh", "decode_streamk.cu", "decode_cluster.cu",
                  "decode_cluster_paged.cu", "combine.cu", "merge.cuh", "streamk.h", "ptx.cuh",
                  "dattn_internal.h", "dattn_api.cpp")


def _code_only(text: str) -> str:
    """C/C++ source without comments, trailing blanks and blank lines: what the
    compiler sees, so that editing a comment keeps a recorded capture valid."""
    out, i, n = [], 0, len(text)
    while i < n:
        if text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        elif text[i] == '"':  # string literal (PTX in asm statements): copied as is
            j = i + 1
            while j < n and text[j] != '"':
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        else:
            out.append(text[i])
            i += 1
    lines = (line.rstrip() for line in "".join(out).splitlines())
    return "\n".join(line for line in lines if line)


def kernel_source_hash() -> str:
    """Hash of the decode path's sources (code only, comments stripped)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "token_decode_attention_gb300", "csrc")
    for name in DECODE_SOURCES:
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            h.update(name.encode() + _code_only(f.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per call of the decode kernel from a committed ncu capture
    (profiles/ncu_traffic.json), if it was taken on these kernel sources."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except Exception:
        return None
    entry = rec.get(workload)
    if not entry or entry.get("kernel_source_hash") != kernel_source_hash():
        return None
    # a capture of part of a large workload (its first sequences) scales to a full call
    return entry.get("dram_bytes_per_call") * entry.get("scale", 1)


class ClockSampler:
    """nvidia-smi clock/throttle sampling in the background."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.dev}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(smax)),
                "samples": len(sm), "reasons": sorted(reasons)}


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def whole_job(ms_local: float, steps: int, bytes_per_step_local: int, heads_per_step_local: int,
              world: int, device) -> dict:
    """Aggregate one replica's timing into the whole-job figures.

    Every rank runs its own replica (weak scaling); the job takes as long as
    the slowest rank, and the work is the sum over ranks.  Collective on every
    rank when world > 1.
    """
    ms_max = max_over_ranks(ms_local, world, device)
    t_step = ms_max * 1e-3 / steps
    total_bytes = all_ranks_sum(bytes_per_step_local, world, device)
    total_heads = all_ranks_sum(heads_per_step_local, world, device)
    return {"ms_per_step": ms_max / steps, "t_step": t_step,
            "value_gbs": total_bytes / t_step / 1e9, "query_heads_per_s": total_heads / t_step,
            "total_bytes_per_step": total_bytes}


def all_ranks_sum(x: int, world: int, device) -> int:
    if world == 1:
        return int(x)
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.int64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return int(t.item())


# ------------------------------------------------------------- our arm

def to_pages(x: dict, page_size: int, seed: int) -> dict:
    """The same cache held in pages of `page_size` positions, in a seeded random
    order of the page pool, with the block table that maps it back."""
    B, S, H, D = x["k"].shape
    if S % page_size:
        raise ValueError(f"seq_len {S} is not a multiple of page_size {page_size}")
    maxp = S // page_size
    perm = torch.from_numpy(np.random.default_rng(seed).permutation(B * maxp)).to(x["k"].device)
    out = {"q": x["q"], "cur_pos": x["cur_pos"],
           "table": perm.view(B, maxp).to(torch.int32).contiguous()}
    for key in ("k", "v"):
        pages = torch.empty((B * maxp, page_size, H, D), dtype=x[key].dtype, device=x[key].device)
        pages[perm] = x[key].view(B * maxp, page_size, H, D)
        out[key] = pages
        x[key] = None  # the dense copy is no longer needed
    return out


class Replica:
    """Input sets, outputs and workspace of one workload on one GPU."""

    def __init__(self, name: str, device, l2_bytes: int, partitions: int = 0,
                 batch: int = 0, page_size: int = 0, current_pos: int | None = None):
        import dataclasses

        import token_decode_attention_gb300 as dattn
        self.dattn = dattn
        self.w = w = WORKLOADS[name]
        if batch:
            # same per-sequence recipe, fewer sequences (small ncu captures)
            self.w = w = dataclasses.replace(w, batch=batch,
                                             description=w.description + f", batch {batch}")
        if current_pos is not None:
            # same recipe, another live length (every sequence)
            self.w = w = dataclasses.replace(w, current_pos=current_pos,
                                             description=w.description + f", current_pos {current_pos}")
        self.device = device
        kv = w.kv_bytes()
        self.sets_n = input_sets(kv, l2_bytes)
        base = make_inputs(w, device, batch=w.batch)
        self.cp_host = base["cur_pos_host"]
        self.page_size = page_size
        if page_size:
            base = to_pages(base, page_size, w.seed)
        self.sets = [base]
        for i in range(1, self.sets_n):
            self.sets.append({key: (val.clone() if key in ("q", "k", "v") else val)
                              for key, val in base.items()})
        self.outs = [torch.empty((w.batch, w.n_heads, w.head_dim), dtype=torch.float16,
                                 device=device) for _ in range(self.sets_n)]
        self.partitions = partitions
        if page_size:
            pages = int(base["k"].shape[0])
            self.plan = dattn.dattn_decode_paged_plan(w.batch, w.n_heads, w.head_dim, page_size,
                                                      w.seq_len // page_size, pages, partitions)
        else:
            self.plan = dattn.dattn_decode_plan(w.batch, w.n_heads, w.head_dim, w.seq_len,
                                                partitions)
        # enough for the dense and the paged call of this shape
        nbytes = max(16, dattn.dattn_decode_workspace_bytes(w.batch, w.n_heads, w.head_dim,
                                                            w.seq_len, partitions))
        self.ws = torch.empty((nbytes,), dtype=torch.uint8, device=device)
        self.bytes_per_step = algorithmic_bytes(w.batch, w.n_heads, w.head_dim, w.seq_len,
                                                self.cp_host)
        # the decode kernel, plus the merge kernel of a split plan
        self.launches_per_step = 1 + (1 if self.plan["partitions"] > 1 and
                                      self.plan["cluster_size"] == 0 else 0)
        # Everything above ran on the default stream; the steps run on a side
        # stream.  Finish it here so no buffer freed by the set-up (and reused
        # by the allocator) is still being read when the side stream writes.
        torch.cuda.synchronize(device)
        self.l2_note = l2_note(kv, l2_bytes)

    def step(self, i: int, stream):
        x = self.sets[i % self.sets_n]
        if self.page_size:
            self.dattn.dattn_decode_paged_f16(x["q"], x["k"], x["v"], self.outs[i % self.sets_n],
                                              x["table"], x["cur_pos"], self.ws, self.partitions,
                                              stream)
        else:
            self.dattn.dattn_decode_f16_ex(x["q"], x["k"], x["v"], self.outs[i % self.sets_n],
                                           x["cur_pos"], self.ws, self.partitions, stream)

    def timed(self, steps: int, warmup: int, stream, world: int, soak_s: float = 1.0,
              sampler: ClockSampler | None = None, graph: bool = True):
        """Device time of exactly `steps` consecutive steps, in ms.

        With graph=True the K steps (rotating input sets) are captured once into
        a CUDA graph, outside the timed region, and the timed region replays it
        once: the GPU runs the K decode calls back to back, as a decode loop
        under graph submission does.  With graph=False the calls are issued
        eagerly from Python, so host overhead per call is included."""
        stream.wait_stream(torch.cuda.current_stream(self.device))
        with torch.cuda.stream(stream):
            for i in range(warmup):
                self.step(i, stream)
            torch.cuda.synchronize()
            g = None
            if graph:
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    for i in range(steps):
                        self.step(i, stream)
                g.replay()
                torch.cuda.synchronize()

            def run_once():
                if g is not None:
                    g.replay()
                else:
                    for i in range(steps):
                        self.step(i, stream)

            # untimed load soak: clocks settle, and the sampler sees the GPU busy
            if sampler is not None:
                sampler.start()
            t_end = time.time() + soak_s
            while time.time() < t_end:
                run_once()
                stream.synchronize()
            barrier(world)
            torch.cuda.synchronize()
            start = torch.cuda.Event(enable_timing=True)
            end = torch.cuda.Event(enable_timing=True)
            start.record(stream)
            run_once()
            end.record(stream)
            torch.cuda.synchronize()
            barrier(world)
        clocks = sampler.stop() if sampler is not None else None
        ms = start.elapsed_time(end)
        del g
        return ms, clocks

    def step_percentiles(self, samples: int, stream) -> dict:
        """Latency of one isolated step: one single-step graph per input set
        (rotating, as in the timed region), each replay bracketed by its own
        events, so a step neither overlaps its predecessor nor hides its launch;
        p10 / p50 / p90 in microseconds over `samples` replays.  The headline
        figure is the back-to-back throughput of the timed region instead."""
        stream.wait_stream(torch.cuda.current_stream(self.device))
        graphs = []
        n = min(self.sets_n, 512)  # 512 of the small workload's sets are 256 MB, 2x L2
        with torch.cuda.stream(stream):
            for i in range(n):
                self.step(i, stream)
            torch.cuda.synchronize()
            for i in range(n):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    self.step(i, stream)
                graphs.append(g)
            for g in graphs:
                g.replay()
            torch.cuda.synchronize()
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(samples)]
            for k, (a, b) in enumerate(ev):
                a.record(stream)
                graphs[k % len(graphs)].replay()
                b.record(stream)
            torch.cuda.synchronize()
        t = np.array([a.elapsed_time(b) * 1e3 for a, b in ev])
        del graphs
        return {"p10": float(np.percentile(t, 10)), "p50": float(np.percentile(t, 50)),
                "p90": float(np.percentile(t, 90)), "samples": samples,
                "note": "each step its own graph launch (not overlapped with the previous one)"}

    def e2e(self, steps: int, warmup: int, stream):
        """Same metric through the public API with host buffers.  Each step takes
        the new token's inputs (q, k, v rows and current_pos, packed in one pinned
        host buffer) from the host, rotates q and k at current_pos and appends k,
        v to the cache (dattn_rope_append_f16), runs the decode and returns out
        into pinned host memory.  The kernels read and write the pinned buffers
        themselves over the CPU-GPU link (unified addressing): every step moves
        the inputs host-to-device and the output device-to-host without a
        copy-engine transfer.  The same step with cudaMemcpyAsync copies in and
        out is measured beside it ('copy_engine').  The KV cache itself is
        device-resident state."""
        if self.page_size:
            return None  # measured on the dense layout only
        w = self.w
        x = self.sets[0]
        B, H, D = w.batch, w.n_heads, w.head_dim
        n = B * H * D
        # one pinned staging buffer: q | k_new | v_new (f16) | current_pos (u32)
        pack_h = torch.empty((3 * n * 2 + 4 * B,), dtype=torch.uint8).pin_memory()
        last = np.minimum(self.cp_host.astype(np.int64), w.seq_len - 1)
        k_rows = torch.stack([x["k"][b, int(last[b])] for b in range(B)]).cpu()
        v_rows = torch.stack([x["v"][b, int(last[b])] for b in range(B)]).cpu()
        halves = pack_h[: 6 * n].view(torch.float16)
        halves[:n].copy_(x["q"].cpu().reshape(-1))
        halves[n:2 * n].copy_(k_rows.reshape(-1))
        halves[2 * n:].copy_(v_rows.reshape(-1))
        pack_h[6 * n:].view(torch.int32).copy_(x["cur_pos"].cpu())
        qh, kh, vh = (halves[i * n:(i + 1) * n].view(B, H, D) for i in range(3))
        cph = pack_h[6 * n:].view(torch.int32)
        out_h = torch.empty((B, H, D), dtype=torch.float16).pin_memory()
        q_rot = torch.empty((B, H, D), dtype=torch.float16, device=self.device)
        out_d = self.outs[0]
        # the copy-engine variant's device-side buffers
        pack_d = torch.empty(pack_h.shape, dtype=torch.uint8, device=self.device)
        dh = pack_d[: 6 * n].view(torch.float16)
        q_d, knew_d, vnew_d = (dh[i * n:(i + 1) * n].view(B, H, D) for i in range(3))
        cp_d = pack_d[6 * n:].view(torch.int32)
        h2d = pack_h.numel()
        d2h = out_h.numel() * 2

        stream.wait_stream(torch.cuda.current_stream(self.device))

        def one():
            self.dattn.dattn_rope_append_f16(qh, kh, vh, q_rot, x["k"], x["v"], cph, stream=stream)
            self.dattn.dattn_decode_f16_ex(q_rot, x["k"], x["v"], out_h, cph, self.ws,
                                           self.partitions, stream)

        def one_ce():
            pack_d.copy_(pack_h, non_blocking=True)
            self.dattn.dattn_rope_append_f16(q_d, knew_d, vnew_d, q_d, x["k"], x["v"], cp_d,
                                             stream=stream)
            self.dattn.dattn_decode_f16_ex(q_d, x["k"], x["v"], out_d, cp_d, self.ws,
                                           self.partitions, stream)
            out_h.copy_(out_d, non_blocking=True)

        def timed(step):
            start = torch.cuda.Event(enable_timing=True)
            end = torch.cuda.Event(enable_timing=True)
            t0 = time.perf_counter()
            start.record(stream)
            for _ in range(steps):
                step()
            end.record(stream)
            torch.cuda.synchronize()
            return start.elapsed_time(end) / steps, (time.perf_counter() - t0) * 1e3 / steps

        def median_of(windows):
            # three timing windows of `steps` steps each: report the median
            # window and list all three
            runs = sorted(windows, key=lambda r: r[0])
            return runs[len(runs) // 2], [r[0] * 1e3 for r in windows]

        def batched(fn):
            # the step recorded once with the library's batch API (outside the
            # timed region) and submitted as one batch per step
            self.dattn.dattn_batch_begin(stream)
            fn()
            batch = self.dattn.dattn_batch_end(stream)
            for _ in range(warmup):
                batch.launch(stream)
            torch.cuda.synchronize()
            res = median_of([timed(lambda: batch.launch(stream)) for _ in range(3)])
            nodes = batch.nodes
            batch.close()
            return res, nodes

        with torch.cuda.stream(stream):
            for _ in range(warmup):
                one()
                one_ce()
            torch.cuda.synchronize()
            (eager_ms, eager_wall), eager_windows = median_of([timed(one) for _ in range(3)])
            ((ms, wall), windows), nodes = batched(one)
            ((ce_ms, _), ce_windows), ce_nodes = batched(one_ce)
        return {"value": self.bytes_per_step / (ms * 1e-3) / 1e9, "unit": "GB/s",
                "ms_per_step": ms, "wall_ms_per_step": wall,
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                "launches_per_step": 1 + self.launches_per_step,
                "submission": f"one dattn_batch_launch per step ({nodes} recorded operations)",
                "windows_us_per_step": [round(w, 2) for w in windows],
                "eager": {"value": self.bytes_per_step / (eager_ms * 1e-3) / 1e9,
                          "ms_per_step": eager_ms, "wall_ms_per_step": eager_wall,
                          "windows_us_per_step": [round(w, 2) for w in eager_windows]},
                "copy_engine": {"value": self.bytes_per_step / (ce_ms * 1e-3) / 1e9,
                                "ms_per_step": ce_ms,
                                "windows_us_per_step": [round(w, 2) for w in ce_windows],
                                "submission": f"one batch per step ({ce_nodes} recorded "
                                              "operations: H2D copy, rope/append, decode, "
                                              "D2H copy)"},
                "note": "the rope/append kernel reads the new token's q, k, v rows and "
                        "current_pos from one pinned host buffer and the decode writes out "
                        "into pinned host memory, over the CPU-GPU link (unified "
                        "addressing; no copy-engine transfer); 'eager' issues the same "
                        "calls from Python each step; 'copy_engine' moves the same bytes "
                        "with cudaMemcpyAsync before and after the kernels; the KV cache is "
                        "device-resident state; value counts the decode's bytes only; the "
                        "median of three timing windows"}


def graph_time_us(fn, steps: int, warmup: int, stream, graph: bool = True) -> float:
    """Device time per call of `fn(i, stream)`: `steps` calls captured in one
    CUDA graph, replayed once between two events on `stream` (or, with
    graph=False, issued eagerly between the events)."""
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        for i in range(warmup):
            fn(i, stream)
        torch.cuda.synchronize()
        g = None
        if graph:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for i in range(steps):
                    fn(i, stream)
            g.replay()
            torch.cuda.synchronize()
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        start.record(stream)
        if g is not None:
            g.replay()
        else:
            for i in range(steps):
                fn(i, stream)
        end.record(stream)
        torch.cuda.synchronize()
    return start.elapsed_time(end) * 1e3 / steps


OPS = ["rope_append_7b", "rope_append_ragged", "rope_append_outlier", "softmax_10240x8192",
       "softmax_65536x1024", "softmax_2048x128256"]


def sweep_ops(device, stream, steps: int, warmup: int, peak: float, only: str | None = None,
              graph: bool = True) -> dict:
    """The two other kernels of a decode step, each timed alone.

    rope_append: rotate the new q and k and append k, v at current_pos, for the
    decode shapes of the 7b, ragged and outlier workloads; algorithmic bytes
    3 B H D halves read + 3 B H D halves written + current_pos.  The inputs are
    small and L2-resident: these are launch/latency figures.
    softmax: f32 row softmax, 8 bytes per element (one read, one write), inputs
    larger than L2, rotating two input sets."""
    import token_decode_attention_gb300 as dattn
    res = {}
    for name in ("7b", "ragged", "outlier"):
        if only is not None and only != f"rope_append_{name}":
            continue
        w = WORKLOADS[name]
        B, H, D, S = w.batch, w.n_heads, w.head_dim, w.seq_len
        try:
            g = torch.Generator(device=device).manual_seed(w.seed)
            new = [torch.empty((B, H, D), dtype=torch.float16, device=device).normal_(
                generator=g) for _ in range(3)]
            qo = torch.empty_like(new[0])
            # a cache of 8 positions per sequence is enough: only row cp is touched
            cache_s = 8
            K = torch.zeros((B, cache_s, H, D), dtype=torch.float16, device=device)
            V = torch.zeros_like(K)
            cp = torch.from_numpy(
                (draw_current_pos(w) % cache_s).astype(np.int64)).to(torch.int32).to(device)
            torch.cuda.synchronize()
            us = graph_time_us(lambda i, st: dattn.dattn_rope_append_f16(
                new[0], new[1], new[2], qo, K, V, cp, stream=st), steps, warmup, stream, graph)
            nbytes = 6 * B * H * D * 2 + 4 * B
            res[f"rope_append_{name}"] = {"us_per_call": us, "GB/s": nbytes / us / 1e3,
                                          "algorithmic_bytes": nbytes,
                                          "shape": f"B={B} H={H} D={D}"}
            del new, qo, K, V
        except Exception as e:
            import traceback
            traceback.print_exc(file=sys.stderr)
            res[f"rope_append_{name}"] = {"error": f"{type(e).__name__}: {e}"}
    for rows, cols in ((10240, 8192), (65536, 1024), (2048, 128256)):
        key = f"softmax_{rows}x{cols}"
        if only is not None and only != key:
            continue
        try:
            g = torch.Generator(device=device).manual_seed(rows + cols)
            xs = [torch.empty((rows, cols), dtype=torch.float32, device=device).normal_(
                0.0, 3.0, generator=g) for _ in range(2)]
            ys = [torch.empty_like(x) for x in xs]
            torch.cuda.synchronize()
            us = graph_time_us(lambda i, st: dattn.dattn_softmax_f32(xs[i % 2], ys[i % 2], st),
                               steps, warmup, stream, graph)
            nbytes = 8 * rows * cols
            gbs = nbytes / us / 1e3
            res[key] = {"us_per_call": us, "GB/s": gbs, "frac_of_measured": gbs / peak,
                        "algorithmic_bytes": nbytes,
                        "l2": f"2 input sets of {rows * cols * 4 / 2**20:.0f} MiB"}
            del xs, ys
        except Exception as e:
            import traceback
            traceback.print_exc(file=sys.stderr)
            res[key] = {"error": f"{type(e).__name__}: {e}"}
        torch.cuda.empty_cache()
    return res


def cpu_baseline(name: str, budget_s: float, max_reps: int = 1000, batch: int = 0,
                 device: str = "cuda") -> dict:
    """The CPU oracle, as it stands, on a bounded sample of the workload
    (`batch` > 0: that many sequences of the same recipe)."""
    import oracle
    w = WORKLOADS[name]
    if batch:
        import dataclasses
        w = dataclasses.replace(w, batch=batch)
    x = make_inputs(WORKLOADS[name], device, batch=w.batch)
    q, k, v = (x[n].cpu().numpy() for n in ("q", "k", "v"))
    cp = x["cur_pos_host"]
    del x
    nbytes = algorithmic_bytes(w.batch, w.n_heads, w.head_dim, w.seq_len, cp)
    reps, t0 = 0, time.perf_counter()
    while reps < max_reps:
        oracle.decode_f64(q, k, v, cp)
        reps += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    el = time.perf_counter() - t0
    return {"value": nbytes * reps / el / 1e9, "unit": "GB/s", "cores": oracle.max_threads(),
            "kind": "oracle", "seconds": el,
            "query_heads_per_s": w.batch * w.n_heads * reps / el,
            "sample": f"{reps} full passes of the {name} workload ({w.description})"
                      + (f", {w.batch} of its sequences" if batch else "")
                      + ", fp64 C oracle with OpenMP"}


def cpu_sweep(budget_s: float) -> dict:
    """The oracle on every workload: small to long whole, outlier on 16 of its
    256 sequences (40 GiB of K/V would not fit a bounded run)."""
    res = {}
    for name in ("small", "7b", "ragged", "long", "outlier"):
        try:
            r = cpu_baseline(name, budget_s, batch=CPU_SAMPLE_SEQUENCES.get(name, 0))
            res[name] = {k: r[k] for k in ("value", "unit", "query_heads_per_s", "seconds",
                                           "cores", "sample")}
        except Exception as e:
            res[name] = {"error": f"{type(e).__name__}: {e}"}
        torch.cuda.empty_cache()
    return res


def sweep(device, stream, l2_bytes: int, steps: int, warmup: int, peak: float) -> dict:
    res = {}
    runs = [(n, 0, None) for n in ("small", "7b", "ragged", "long", "outlier")]
    # a live length whose CTA ranges end inside a stage (most lengths do)
    runs += [("7b", 0, 3332)]
    runs += [(n, 16, None) for n in ("7b", "ragged", "long", "outlier")]
    runs += [("7b", 128, None)]  # pages large enough for the cluster plan
    for name, ps, cp in runs:
        key = name + (f"_paged{ps}" if ps else "") + (f"_cp{cp}" if cp is not None else "")
        try:
            r = Replica(name, device, l2_bytes, page_size=ps, current_pos=cp)
            ms, _ = r.timed(steps, warmup, stream, 1, soak_s=0.2)
            pct = r.step_percentiles(max(20, steps), stream)
            t = ms * 1e-3 / steps
            gbs = r.bytes_per_step / t / 1e9
            res[key] = {"us_per_step": t * 1e6, "GB/s": gbs, "frac_of_measured": gbs / peak,
                         "frac_of_nominal_8TBs": gbs / NOMINAL_HBM_GBS,
                         "query_heads_per_s": r.w.batch * r.w.n_heads / t,
                         "isolated_step_us_p10_p50_p90": [pct["p10"], pct["p50"], pct["p90"]],
                         "plan": "cluster" if r.plan["cluster_size"] else "split",
                         "partitions": r.plan["partitions"],
                         "algorithmic_bytes": r.bytes_per_step, "l2": r.l2_note}
            del r
        except Exception as e:  # report, keep going
            import traceback
            traceback.print_exc(file=sys.stderr)
            res[key] = {"error": f"{type(e).__name__}: {e}"}
        torch.cuda.empty_cache()
    return res


# ---------------------------------------------------------------- main

def run_reference(args, world, rank):
    """The oracle, as it stands, on this host's cores: each step one pass over
    the workload, or over a bounded sample of its sequences (same recipe)
    where the whole workload would take minutes."""
    if rank != 0:
        return
    import dataclasses

    import oracle
    full = WORKLOADS[args.workload]
    sample = CPU_SAMPLE_SEQUENCES.get(full.name, 0)
    w = dataclasses.replace(full, batch=sample) if sample else full
    # drawn on the GPU when there is one (the host's float16 sampler is
    # single-threaded: ~1 min for this sample), then copied to the host
    x = make_inputs(full, "cuda" if torch.cuda.is_available() else "cpu", batch=w.batch)
    q, k, v = (x[n].cpu().numpy() for n in ("q", "k", "v"))
    cp = x["cur_pos_host"]
    del x
    nbytes = algorithmic_bytes(w.batch, w.n_heads, w.head_dim, w.seq_len, cp)
    for _ in range(args.warmup):
        oracle.decode_f64(q, k, v, cp)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.decode_f64(q, k, v, cp)
    el = time.perf_counter() - t0
    val = nbytes * args.steps / el / 1e9
    what = (f"each step one pass over {sample} of the {full.batch} sequences of the {full.name} "
            f"workload (same recipe)" if sample else
            f"each step one full pass of the {full.name} workload")
    line = {"metric": METRIC, "value": val, "unit": "GB/s", "impl": "reference",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": el * 1e3 / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(full, world, device_l2_bytes()),
            "query_heads_per_s": w.batch * w.n_heads * args.steps / el,
            "cpu_baseline": {"value": val, "unit": "GB/s", "cores": oracle.max_threads(),
                             "kind": "oracle", "sample": what + ", fp64 C oracle with OpenMP"},
            "e2e": {"value": val, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="outlier", choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--eager", action="store_true",
                    help="issue the timed steps from Python instead of a CUDA graph")
    ap.add_argument("--partitions", type=int, default=0,
                    help="force the number of decode partitions (0 = library choice)")
    ap.add_argument("--paged", type=int, default=0,
                    help="hold the cache in pages of this many positions (0 = dense)")
    ap.add_argument("--batch", type=int, default=0,
                    help="with --profile: fewer sequences of the same recipe")
    ap.add_argument("--profile", action="store_true",
                    help="only warm-up and timed steps of one workload (for ncu captures)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--op", default="", choices=[""] + OPS,
                    help="with --profile: time this other kernel of the decode step instead")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    world, rank, local = dist_env()

    if args.impl == "reference":
        run_reference(args, world, rank)
        return

    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)

    from token_decode_attention_gb300 import build
    if rank == 0:
        build.build()
    barrier(world)
    import token_decode_attention_gb300 as dattn
    dattn.load()

    props = torch.cuda.get_device_properties(device)
    l2 = int(getattr(props, "L2_cache_size", 0) or 129 * 2**20)
    peak, peak_kind = hbm_peak()
    stream = torch.cuda.Stream(device=device)

    if args.profile and args.op:
        r = sweep_ops(device, stream, args.steps, args.warmup, peak, only=args.op,
                      graph=not args.eager)
        print(json.dumps({"profile": args.op, **r[args.op]}), flush=True)
        if "error" in r[args.op]:
            raise SystemExit(1)
        return
    rep = Replica(args.workload, device, l2, args.partitions,
                  args.batch if args.profile else 0, args.paged)
    sampler = ClockSampler(local)
    if args.profile:
        ms, _ = rep.timed(args.steps, args.warmup, stream, world, soak_s=0.0,
                          graph=not args.eager)
        t = ms * 1e-3 / args.steps
        print(json.dumps({"profile": args.workload, "ms_per_step": t * 1e3,
                          "GB/s": rep.bytes_per_step / t / 1e9, "plan": rep.plan}), flush=True)
        return
    ms, clocks = rep.timed(args.steps, args.warmup, stream, world, sampler=sampler,
                           graph=not args.eager)
    eager_ms, _ = rep.timed(args.steps, 1, stream, world, soak_s=0.0, graph=False)
    eager_ms = max_over_ranks(eager_ms, world, device)
    job = whole_job(ms, args.steps, rep.bytes_per_step, rep.w.batch * rep.w.n_heads, world,
                    device)
    t_step = job["t_step"]
    value = job["value_gbs"]
    per_call = rep.bytes_per_step / t_step / 1e9
    pct = rep.step_percentiles(max(20, args.steps), stream)
    e2e = rep.e2e(args.steps, args.warmup, stream)
    if dattn.dattn_device_error(clear=True) != 0:
        raise RuntimeError("device error word set: a kernel gave up on a pipeline wait")

    if rank != 0:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return

    w = rep.w
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_step * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "data": "synthetic",
        "config": workload_config(w, world, l2),
        "query_heads_per_s": job["query_heads_per_s"],
        "frac_of_nominal_8TBs": per_call / NOMINAL_HBM_GBS,
        "roofline": {"bound": "hbm", "achieved": per_call, "peak": peak, "unit": "GB/s",
                     "frac": per_call / peak, "peak_source": f"{peak_kind} hbm_gbs",
                     "traffic": recorded_traffic(w.name),
                     "kernel": "one dattn_decode_f16_ex call: decode_streamk_kernel "
                               "(dominant) + combine_kernel launched with PDL",
                     "algorithmic_bytes_per_call": rep.bytes_per_step},
        "e2e": e2e,
        "submission": "eager Python calls" if args.eager else
                      "one CUDA graph of the K steps, captured before the timed region",
        "eager_ms_per_step": eager_ms / args.steps,
        "isolated_step_us": pct,
        "gpu_launches": rep.launches_per_step * args.steps,
        "clocks": clocks,
        "plan": rep.plan,
    }
    del rep
    torch.cuda.empty_cache()
    if world == 1:
        line["cpu_baseline"] = cpu_baseline(args.workload, args.cpu_seconds,
                                            batch=CPU_SAMPLE_SEQUENCES.get(args.workload, 0))
        if not args.no_sweep:
            line["sweep"] = sweep(device, stream, l2, 20, 3, peak)
            line["sweep_ops"] = sweep_ops(device, stream, 20, 3, peak)
            line["cpu_sweep"] = cpu_sweep(min(3.0, args.cpu_seconds))
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
