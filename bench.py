"""Benchmark of the paged-KV attention hot path on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl pkv|reference]

One step = one pass of the hot path over the 128-sequence Qwen3-0.6B-like
decode batch (16 q / 8 KV heads, head_dim 128, contexts U[100, 1024], 256-token
blocks in a 1024-block pool): the store of the new K/V row of every sequence
and the decode attention over the cache, done by pkv_decode_attention_append in
one split-K kernel (contexts cut across blocks are merged in-kernel by
log-sum-exp).  The timed step is that call captured once as a CUDA graph and
replayed, as a serving engine replays its decode step; the eager (uncaptured)
time and the same step as two calls (pkv_store_kvcache, then
pkv_decode_attention) are reported beside it.
The metric is KV GB/s (algorithmic bytes / step time) with decode tokens/s per
layer beside it.  The long-context decode, prefix-sharing decode, chunked
prefill and INT8-cache (decode and prefill) workloads are measured too and
reported under "other_workloads", with
the host cost of the block manager that produces the decode step's block
tables and slot mapping.

Timing: W untimed warm-up steps, then K steps bracketed by a barrier and
cudaDeviceSynchronize; L2 (126 MB) is flushed before every step by a 256 MiB
write followed by a 256 MiB read of another buffer (so that the write-backs of
the flush land before the step, not inside it), and each step is timed alone
with CUDA events on the launching stream.
A second timed pass with the library's kernel profiler on gives per-kernel
durations for the roofline.  Under torchrun each rank runs an independent
replica on its own GPU (no collective on the data path); value = bytes of all
ranks / max over ranks of the time.

--impl reference times the fp64 CPU oracle on the host cores instead (a
bounded sample of each step) and prints the same JSON line with
"impl": "reference".
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from paged_kv_cache_493_b300 import workloads as W  # noqa: E402

METRIC = "paged decode attention KV GB/s (% of HBM peak) and decode tokens/s/layer"
MAIN_WORKLOAD = "qwen_decode_b128"
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
# DRAM bytes (read + write) of one launch of a kernel on a workload, from an
# ncu capture, keyed by the SHA-256 of the kernel's source files at the time
# of the capture: the figure is reported only while the sources still hash to
# that value (any change to the kernel makes it null until captured again).
KERNEL_SOURCES = {
    "decode_append": ("decode_attention.cu", "pkv_device.cuh", "pkv_internal.h", "pkv_pair_gap.h"),
}
TRAFFIC_CAPTURES = {
    # kernel: (sha256 of its sources, workload, dram bytes per launch)
    "decode_append": ("c50eda2520f3cade45e0bb2510ec34cc8665aead7cf845c126939f89758649f2", MAIN_WORKLOAD,
                      324840192 + 4035072),
}


def sources_digest(kernel: str) -> str:
    import hashlib
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "paged_kv_cache_493_b300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def captured_traffic(kernel: str, workload: str):
    digest, wl, dram = TRAFFIC_CAPTURES.get(kernel, (None, None, None))
    if digest is None or wl != workload or dram is None:
        return None
    return dram if sources_digest(kernel) == digest else None


# ----------------------------------------------------------------------------- ranks
def dist_setup():
    """(rank, world, local_rank); initialises torch.distributed when WORLD_SIZE > 1."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1 and not torch.distributed.is_initialized():
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        torch.distributed.init_process_group(backend)
    return rank, world, local


def barrier():
    if torch.distributed.is_available() and torch.distributed.is_initialized():
        torch.distributed.barrier()


def reduce_max(x: float) -> float:
    if torch.distributed.is_available() and torch.distributed.is_initialized():
        dev = "cuda" if torch.distributed.get_backend() == "nccl" else "cpu"
        t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        return float(t.item())
    return float(x)


def replica_seed(base: int, rank: int) -> int:
    """Each rank draws its own batch: weak scaling over independent replicas."""
    return base + 7919 * rank


# ----------------------------------------------------------------------------- work model
def decode_kv_bytes(case) -> int:
    c = case.cache
    hkv, d = int(c.k_cache.shape[2]), int(c.k_cache.shape[3])
    return int(c.context_lens.sum()) * hkv * d * 2 * 2


def decode_step_bytes(case) -> dict:
    """Algorithmic bytes of one decode step: every cached K/V row read once, q
    read, out written, new rows read and written, metadata read."""
    kv = decode_kv_bytes(case)
    q = case.q.numel() * 2  # q read; the bf16 output written is the same size
    new = (case.k_new.numel() + case.v_new.numel()) * 2
    meta = (case.cache.block_tables.numel() + case.cache.context_lens.numel() +
            case.slot_mapping.numel()) * 4
    return {"kv": kv, "split_kernel": kv + 2 * q + meta, "step": kv + 2 * q + 2 * new + meta}


def unique_kv_bytes(case) -> int:
    """K/V bytes of distinct physical token slots (shared prefix blocks counted once)."""
    c = case.cache
    hkv, d = int(c.k_cache.shape[2]), int(c.k_cache.shape[3])
    per_block = {}
    for s, ctx in enumerate(c.context_lens.tolist()):
        row = c.block_tables[s].tolist()
        for b in range((ctx + 255) // 256):
            n = min(256, ctx - b * 256)
            per_block[row[b]] = max(per_block.get(row[b], 0), n)
    return sum(per_block.values()) * hkv * d * 2 * 2


def prefill_flops(case) -> int:
    c = case.cache
    hq, d = int(case.q.shape[1]), int(case.q.shape[2])
    cu = case.cu_seqlens_q.tolist()
    total = 0
    for s, ctx in enumerate(c.context_lens.tolist()):
        lq = cu[s + 1] - cu[s]
        # query i sees ctx - lq + i + 1 keys; QK^T and PV are 2 * d flops per key each
        keys = lq * (ctx - lq) + lq * (lq + 1) // 2
        total += keys * hq * d * 4
    return total


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples during the timed region (200 ms period)."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, ValueError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, max_mhz_hint: float) -> dict:
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
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
            return {"sm_mhz": None, "sm_max_mhz": max_mhz_hint, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax) if smax else max_mhz_hint,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- helpers
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        p = json.load(open(path))
        return {k: float(p[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained")}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def to_dev(t):
    return t.to("cuda", non_blocking=False)


class Flusher:
    """Evicts the L2 (126 MB) between steps: writes 256 MiB, then reads another
    256 MiB so that the written lines are drained to HBM before the next timed
    step starts (otherwise up to 126 MB of write-backs of the flush itself
    would land inside the timed region)."""

    def __init__(self):
        self.buf = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
        self.rbuf = torch.ones(64 << 20, dtype=torch.int32, device="cuda")
        self.k = 0

    def __call__(self):
        self.k = (self.k + 1) & 0xFF
        self.buf.fill_(self.k)
        self.sink = self.rbuf.sum()


def time_steps(step, steps: int, flush: Flusher):
    stream = torch.cuda.current_stream()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(steps):
        flush()
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    barrier()
    wall = time.perf_counter() - t0
    per = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    return per, wall


# ----------------------------------------------------------------------------- GPU arm
class DecodeBench:
    def __init__(self, case, pkv, shared_blocks: int = 0):
        self.case, self.pkv = case, pkv
        self.shared_blocks = int(shared_blocks)
        c = case.cache
        self.kc, self.vc = to_dev(c.k_cache), to_dev(c.v_cache)
        self.bt, self.cl = to_dev(c.block_tables), to_dev(c.context_lens)
        self.q, self.kn, self.vn = to_dev(case.q), to_dev(case.k_new), to_dev(case.v_new)
        self.sm = to_dev(case.slot_mapping)
        self.out = torch.empty_like(self.q)
        pkv.pkv_reserve_workspace(case.num_seqs, int(case.q.shape[1]), int(case.q.shape[2]),
                                  int(c.block_tables.shape[1]))

    def fused_step(self):
        """The decode step as one kernel: store of the new rows and attention."""
        self.pkv.pkv_decode_attention_append(self.q, self.kn, self.vn, self.sm, self.kc, self.vc,
                                             self.bt, self.cl, self.case.scale, self.out)

    def step(self):
        p = self.pkv
        p.pkv_store_kvcache(self.kn, self.vn, self.sm, self.kc, self.vc)
        if self.shared_blocks > 0:
            p.pkv_decode_attention_shared_prefix(self.q, self.kc, self.vc, self.bt, self.cl,
                                                 self.case.scale, self.shared_blocks, self.out)
        else:
            p.pkv_decode_attention(self.q, self.kc, self.vc, self.bt, self.cl, self.case.scale,
                                   self.out)

    def e2e_setup(self):
        """A step's inputs (q, new K/V rows, slot mapping, block tables,
        context lengths) packed into one pinned host buffer and one device
        buffer of the same layout (each tensor at a 256-byte-aligned offset),
        so a step makes one host-to-device copy and one device-to-host copy
        of the output."""
        c = self.case
        srcs = [c.q, c.k_new, c.v_new, c.slot_mapping, c.cache.block_tables, c.cache.context_lens]
        offs, total = [], 0
        for t in srcs:
            offs.append(total)
            total += -(-t.numel() * t.element_size() // 256) * 256
        self.h_buf = torch.empty(total, dtype=torch.uint8).pin_memory()
        self.d_buf = torch.empty(total, dtype=torch.uint8, device="cuda")

        def view(buf, off, t):
            n = t.numel() * t.element_size()
            return buf[off:off + n].view(t.dtype).view(t.shape)

        for t, off in zip(srcs, offs):
            view(self.h_buf, off, t).copy_(t)
        self.d_in = [view(self.d_buf, off, t) for t, off in zip(srcs, offs)]
        self.h_out = torch.empty(self.out.shape, dtype=self.out.dtype).pin_memory()
        return total, self.h_out.numel() * self.h_out.element_size()

    def e2e_step(self):
        p = self.pkv
        self.d_buf.copy_(self.h_buf, non_blocking=True)
        q, kn, vn, sm, bt, cl = self.d_in
        p.pkv_decode_attention_append(q, kn, vn, sm, self.kc, self.vc, bt, cl, self.case.scale,
                                      self.out)
        self.h_out.copy_(self.out, non_blocking=True)

    def e2e_phases(self, steps: int, flush) -> dict:
        """Per-phase device time of the eager end-to-end step (CUDA events on
        the stream): input copy, the two library calls, output copy."""
        stream = torch.cuda.current_stream()
        tot = {"h2d": 0.0, "calls": 0.0, "d2h": 0.0}
        p = self.pkv
        for _ in range(steps):
            flush()
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
            ev[0].record(stream)
            self.d_buf.copy_(self.h_buf, non_blocking=True)
            ev[1].record(stream)
            q, kn, vn, sm, bt, cl = self.d_in
            p.pkv_decode_attention_append(q, kn, vn, sm, self.kc, self.vc, bt, cl,
                                          self.case.scale, self.out)
            ev[2].record(stream)
            self.h_out.copy_(self.out, non_blocking=True)
            ev[3].record(stream)
            torch.cuda.synchronize()
            tot["h2d"] += ev[0].elapsed_time(ev[1])
            tot["calls"] += ev[1].elapsed_time(ev[2])
            tot["d2h"] += ev[2].elapsed_time(ev[3])
        return {k + "_ms": round(v / steps, 5) for k, v in tot.items()}


def capture_graph(step):
    """The step captured once as a CUDA graph (how a serving engine replays its
    decode step); the step's library calls are capturable once the decode
    workspace is reserved.  Returns the replay function."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    torch.cuda.synchronize()
    return graph.replay


def kernel_times(pkv, step, steps, flush, names):
    pkv.pkv_profiler_reset()
    pkv.pkv_profiler_enable(True)
    try:
        time_steps(step, steps, flush)
        res = {n: pkv.pkv_profiler_read(n) for n in names}
    finally:
        pkv.pkv_profiler_enable(False)
        pkv.pkv_profiler_reset()
    return res


def run_gpu(args, rank, world, local):
    import paged_kv_cache_493_b300 as pkv
    from paged_kv_cache_493_b300 import _build
    _build.build()
    pkv.load_library()
    torch.cuda.set_device(local)
    peaks, peak_src = load_peaks()
    flush = Flusher()

    case = W.qwen_decode(seed=replica_seed(1002, rank))
    bytes_ = decode_step_bytes(case)
    bench = DecodeBench(case, pkv)
    for _ in range(args.warmup):
        bench.step()
    torch.cuda.synchronize()

    # The step: pkv_decode_attention_append (store of the new rows and the
    # split-K decode in one kernel), captured once as a graph and replayed;
    # the two-call step (pkv_store_kvcache + pkv_decode_attention) beside it.
    for _ in range(args.warmup):
        bench.fused_step()
    replay = capture_graph(bench.fused_step)
    replay2 = capture_graph(bench.step)
    for _ in range(args.warmup):
        replay()
        replay2()
    with ClockSampler(local) as clk:
        per, wall = time_steps(replay, args.steps, flush)
        eager_per, _ = time_steps(bench.fused_step, args.steps, flush)
        kt = kernel_times(pkv, bench.fused_step, args.steps, flush, ["decode_append"])
        two_per, _ = time_steps(replay2, args.steps, flush)
        kt2 = kernel_times(pkv, bench.step, args.steps, flush, ["store_kvcache", "decode"])
    step_ms = reduce_max(sum(per) / len(per))
    eager_ms = reduce_max(sum(eager_per) / len(eager_per))
    two_ms = reduce_max(sum(two_per) / len(two_per))
    value = world * bytes_["step"] / (step_ms * 1e-3) / 1e9
    split_ms = kt["decode_append"][0] / max(kt["decode_append"][1], 1)
    achieved = bytes_["step"] / (split_ms * 1e-3) / 1e9
    launches_per_step = sum(n for _, n in kt.values()) / args.steps

    # End to end through the C ABI from pinned host buffers: one packed
    # host-to-device copy of the step's inputs, the two calls, the output
    # copied back; timed as a captured graph (how an engine replays its decode
    # step, copies included) and eagerly (one Python call per operation).
    h2d, d2h = bench.e2e_setup()
    for _ in range(args.warmup):
        bench.e2e_step()
    e2e_eager_per, _ = time_steps(bench.e2e_step, args.steps, flush)
    e2e_replay = capture_graph(bench.e2e_step)
    for _ in range(args.warmup):
        e2e_replay()
    e2e_per, _ = time_steps(e2e_replay, args.steps, flush)
    e2e_ms = reduce_max(sum(e2e_per) / len(e2e_per))
    e2e_eager_ms = reduce_max(sum(e2e_eager_per) / len(e2e_eager_per))
    phases = bench.e2e_phases(args.steps, flush)
    torch.cuda.synchronize()
    e2e_ok = torch.equal(bench.h_out.to("cuda"), bench.out)

    other = {}
    if not args.only_main:
        other = other_workloads(pkv, args, rank, flush, peaks)

    code, site = pkv.pkv_get_device_error()
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(step_ms, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {
            "workload": MAIN_WORKLOAD, "num_seqs": case.num_seqs, "context_lens": "U[100,1024] seeded",
            "mean_context": round(float(case.cache.context_lens.float().mean()), 1),
            "num_q_heads": 16, "num_kv_heads": 8, "head_dim": 128, "block_size": 256,
            "num_blocks": case.cache.num_blocks, "step": "pkv_decode_attention_append: store of the new K/V rows + split-K decode with in-kernel merge, one kernel, replayed as a CUDA graph",
            "l2": "flushed before every step (256 MiB write, then a 256 MiB read of another buffer that drains the written lines), step timed alone",
            "parallelism": f"replicas{world}",
        },
        "tokens_per_s_per_layer": round(world * case.num_seqs / (step_ms * 1e-3), 1),
        "kv_gbs": round(world * bytes_["kv"] / (step_ms * 1e-3) / 1e9, 2),
        "frac_of_hbm_peak": round(value / world / peaks["hbm_gbs"], 4),
        "frac_of_nominal_8tbs": round(value / world / 8000.0, 4),
        "wall_s_timed_region": round(wall, 4),
        "eager_ms_per_step": round(eager_ms, 5),
        "two_call_step": {"calls": "pkv_store_kvcache + pkv_decode_attention (graph)",
                          "ms_per_step": round(two_ms, 5),
                          "kernel_ms": {n: round(v[0] / max(v[1], 1), 5) for n, v in kt2.items()}},
        "roofline": {
            "kernel": "decode_split (fused store: pkv_decode_attention_append)",
            "bound": "hbm",
            "achieved": round(achieved, 2),
            "peak": peaks["hbm_gbs"],
            "peak_source": f"{peak_src} hbm_gbs (burst copy)",
            "unit": "GB/s",
            "frac": round(achieved / peaks["hbm_gbs"], 4),
            "traffic": captured_traffic("decode_append", MAIN_WORKLOAD),
            "traffic_source": "ncu dram__bytes_read.sum + dram__bytes_write.sum of one launch, "
                              "valid only for the kernel sources it was captured on",
            "algorithmic_bytes_per_launch": bytes_["step"],
            "avg_launch_ms": round(split_ms, 5),
            "kernel_ms": {n: round(v[0] / max(v[1], 1), 5) for n, v in kt.items()},
        },
        "e2e": {"value": round(world * bytes_["step"] / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                "ms_per_step": round(e2e_ms, 5), "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "output_matches_device": bool(e2e_ok),
                "how": "one packed pinned H2D copy + pkv_store_kvcache + pkv_decode_attention "
                       "+ pinned D2H of out, captured once as a CUDA graph and replayed",
                "eager_ms_per_step": round(e2e_eager_ms, 5),
                "eager_phases": phases},
        "gpu_launches": int(round(launches_per_step * args.steps)),
        "clocks": clk.summary(2032.0),
        "device_error": code,
    }
    if rank == 0 and world == 1:
        line["cpu_baseline"] = cpu_baseline(case, bytes_)
    if other:
        line["other_workloads"] = other
    if rank == 0:
        print(json.dumps(line), flush=True)


def other_workloads(pkv, args, rank, flush, peaks, only=None):
    res = {}
    steps = max(3, min(args.steps, 10))
    # Long-context and prefix-sharing decode.
    for name, make in (("long_decode_32k", W.long_decode), ("prefix_decode_b64", W.prefix_decode)):
        if only is not None and name != only:
            continue
        case = make(seed=replica_seed(1003 if name.startswith("long") else 1004, rank))
        b = decode_step_bytes(case)
        shared = case.shared_prefix_blocks if name.startswith("prefix") else 0
        bench = DecodeBench(case, pkv, shared_blocks=shared)
        for _ in range(3):
            bench.step()
        kt = kernel_times(pkv, bench.step, steps, flush, ["shared_prefix", "decode"])

        def attn():
            if shared:
                pkv.pkv_decode_attention_shared_prefix(bench.q, bench.kc, bench.vc, bench.bt,
                                                       bench.cl, case.scale, shared, bench.out)
            else:
                pkv.pkv_decode_attention(bench.q, bench.kc, bench.vc, bench.bt, bench.cl,
                                         case.scale, bench.out)

        # The step (store + attention) and the attention call alone, each
        # captured as a CUDA graph and replayed (no host launch time inside).
        per, _ = time_steps(capture_graph(bench.step), steps, flush)
        aper, _ = time_steps(capture_graph(attn), steps, flush)
        ms = sum(per) / len(per)
        dec_ms = sum(aper) / len(aper)
        entry = {"step_ms": round(ms, 5), "decode_ms": round(dec_ms, 5),
                 "timing": "graph replays, L2 flushed before each",
                 "kernel_ms_eager": {n: round(v[0] / max(v[1], 1), 5) for n, v in kt.items()
                                     if v[1]},
                 "kv_bytes": b["kv"], "kv_gbs": round(b["kv"] / (dec_ms * 1e-3) / 1e9, 2),
                 "frac_of_hbm_peak": round(b["kv"] / (dec_ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
                 "tokens_per_s_per_layer": round(case.num_seqs / (ms * 1e-3), 1)}
        if shared:
            def plain():
                pkv.pkv_decode_attention(bench.q, bench.kc, bench.vc, bench.bt, bench.cl,
                                         case.scale, bench.out)

            pper, _ = time_steps(capture_graph(plain), steps, flush)
            u = unique_kv_bytes(case)
            entry.update({
                "decode": f"pkv_decode_attention_shared_prefix ({shared} shared blocks): "
                          "shared-prefix tcgen05 kernel + split-K decode of the private parts",
                "unique_kv_bytes": u,
                "unique_kv_gbs": round(u / (dec_ms * 1e-3) / 1e9, 2),
                "unique_frac_of_hbm_peak": round(u / (dec_ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
                "plain_decode_ms": round(sum(pper) / len(pper), 5)})
        res[name] = entry
        del bench
        torch.cuda.empty_cache()
    if only is None or only == "qwen_decode_b128_int8":
        res["qwen_decode_b128_int8"] = int8_decode_workload(pkv, steps, flush, peaks, rank)
        torch.cuda.empty_cache()
    if only is None or only == "chunked_prefill_8x512_int8":
        res["chunked_prefill_8x512_int8"] = int8_prefill_workload(pkv, steps, flush, peaks, rank)
        torch.cuda.empty_cache()
    if only is None:
        res["host_block_manager"] = host_block_manager(pkv)
    if only is not None and only != "chunked_prefill_8x512":
        return res
    # Chunked prefill.
    case = W.chunked_prefill(seed=replica_seed(1005, rank))
    c = case.cache
    kc, vc, bt, cl = to_dev(c.k_cache), to_dev(c.v_cache), to_dev(c.block_tables), to_dev(c.context_lens)
    q, kn, vn, sm = to_dev(case.q), to_dev(case.k_new), to_dev(case.v_new), to_dev(case.slot_mapping)
    cu = to_dev(case.cu_seqlens_q)
    out = torch.empty_like(q)

    def pstep():
        pkv.pkv_store_kvcache(kn, vn, sm, kc, vc)
        pkv.pkv_prefill_attention(q, kc, vc, bt, cu, cl, case.scale, out)

    def pcall():
        pkv.pkv_prefill_attention(q, kc, vc, bt, cu, cl, case.scale, out)

    def scall():
        pkv.pkv_store_kvcache(kn, vn, sm, kc, vc)

    for _ in range(3):
        pstep()
    kt = kernel_times(pkv, pstep, steps, flush, ["store_kvcache", "prefill"])
    # Step, prefill call and store call each replayed from a CUDA graph.
    per, _ = time_steps(capture_graph(pstep), steps, flush)
    pper, _ = time_steps(capture_graph(pcall), steps, flush)
    sper, _ = time_steps(capture_graph(scall), steps, flush)
    flops = prefill_flops(case)
    pre_ms = sum(pper) / len(pper)
    st_ms = sum(sper) / len(sper)
    store_bytes = int((case.slot_mapping >= 0).sum()) * 8 * 128 * 2 * 2 * 2
    tf = flops / (pre_ms * 1e-3) / 1e12
    res["chunked_prefill_8x512"] = {
        "step_ms": round(sum(per) / len(per), 5), "prefill_ms": round(pre_ms, 5), "flops": flops,
        "timing": "graph replays, L2 flushed before each",
        "tflops": round(tf, 2), "frac_of_bf16_peak": round(tf / peaks["bf16_tflops"], 4),
        "frac_of_bf16_sustained": round(tf / peaks["bf16_tflops_sustained"], 4),
        "kernel_ms_eager": {n: round(v[0] / max(v[1], 1), 5) for n, v in kt.items()},
        "store_ms": round(st_ms, 5), "store_bytes": store_bytes,
        "store_gbs": round(store_bytes / (st_ms * 1e-3) / 1e9, 2)}
    return res


def int8_decode_workload(pkv, steps, flush, peaks, rank) -> dict:
    """The 128-sequence decode step over the INT8 cache: quantising store of
    the new rows, then the split-K decode over the codes.  The INT8 pool
    holds the same tokens as the bf16 pool."""
    case = W.qwen_decode(seed=replica_seed(1002, rank))
    c = case.cache
    nb, bs, hkv, d = (int(x) for x in c.k_cache.shape)
    kc, vc, ks, vs = int8_pool_of(c)
    q, kn, vn, sm = to_dev(case.q), to_dev(case.k_new), to_dev(case.v_new), to_dev(case.slot_mapping)
    bt, cl = to_dev(c.block_tables), to_dev(c.context_lens)
    out = torch.empty_like(q)

    def step():
        pkv.pkv_store_kvcache_int8(kn, vn, sm, kc, vc, ks, vs)
        pkv.pkv_decode_attention_int8(q, kc, vc, ks, vs, bt, cl, case.scale, out)

    def dcall():
        pkv.pkv_decode_attention_int8(q, kc, vc, ks, vs, bt, cl, case.scale, out)

    for _ in range(3):
        step()
    pkv.pkv_reserve_workspace(case.num_seqs, int(case.q.shape[1]), d, int(c.block_tables.shape[1]))
    kt = kernel_times(pkv, step, steps, flush, ["store_kvcache_int8", "decode_int8"])
    per, _ = time_steps(capture_graph(step), steps, flush)
    dper, _ = time_steps(capture_graph(dcall), steps, flush)
    ms = sum(per) / len(per)
    dec_ms = sum(dper) / len(dper)
    kv = int(c.context_lens.sum()) * hkv * (2 * d + 2 * 4)  # codes + one fp32 scale per row, K and V
    dec_bytes = kv + case.q.numel() * 2 * 2 + (c.block_tables.numel() + c.context_lens.numel()) * 4
    gbs = dec_bytes / (dec_ms * 1e-3) / 1e9
    return {"step_ms": round(ms, 5), "decode_ms": round(dec_ms, 5), "kv_bytes": kv,
            "decode_bytes": dec_bytes, "decode_gbs": round(gbs, 2),
            "frac_of_hbm_peak": round(gbs / peaks["hbm_gbs"], 4),
            "tokens_per_s_per_layer": round(case.num_seqs / (ms * 1e-3), 1),
            "kernels": "store_kvcache_int8; decode_int8 = the split-K decode kernel over codes"}


def int8_pool_of(c):
    """Device INT8 pool (codes [NB, Hkv, 256, D], scales [NB, Hkv, 256])
    holding the same tokens as the case's bf16 pool: the quantising store is
    run over every slot of it."""
    nb, bs, hkv, d = (int(x) for x in c.k_cache.shape)
    kc = torch.empty((nb, hkv, bs, d), dtype=torch.int8, device="cuda")
    vc = torch.empty_like(kc)
    ks = torch.empty((nb, hkv, bs), dtype=torch.float32, device="cuda")
    vs = torch.empty_like(ks)
    kb, vb = to_dev(c.k_cache).view(nb * bs, hkv, d), to_dev(c.v_cache).view(nb * bs, hkv, d)
    every = torch.arange(nb * bs, dtype=torch.int32, device="cuda")
    import paged_kv_cache_493_b300 as pkv
    pkv.pkv_store_kvcache_int8(kb, vb, every, kc, vc, ks, vs)
    torch.cuda.synchronize()
    return kc, vc, ks, vs


def int8_prefill_workload(pkv, steps, flush, peaks, rank) -> dict:
    """The 8 x 512 chunked-prefill step over the INT8 cache: quantising
    store of the chunk's rows, then the INT8 prefill (tiles dequantised to
    bf16 in shared memory, then the tcgen05 pipeline)."""
    case = W.chunked_prefill(seed=replica_seed(1005, rank))
    c = case.cache
    kc, vc, ks, vs = int8_pool_of(c)
    bt, cl, cu = to_dev(c.block_tables), to_dev(c.context_lens), to_dev(case.cu_seqlens_q)
    q, kn, vn, sm = to_dev(case.q), to_dev(case.k_new), to_dev(case.v_new), to_dev(case.slot_mapping)
    out = torch.empty_like(q)

    def step():
        pkv.pkv_store_kvcache_int8(kn, vn, sm, kc, vc, ks, vs)
        pkv.pkv_prefill_attention_int8(q, kc, vc, ks, vs, bt, cu, cl, case.scale, out)

    def pcall():
        pkv.pkv_prefill_attention_int8(q, kc, vc, ks, vs, bt, cu, cl, case.scale, out)

    for _ in range(3):
        step()
    kt = kernel_times(pkv, step, steps, flush, ["store_kvcache_int8", "prefill_int8"])
    per, _ = time_steps(capture_graph(step), steps, flush)
    pper, _ = time_steps(capture_graph(pcall), steps, flush)
    flops = prefill_flops(case)
    pre_ms = sum(pper) / len(pper)
    tf = flops / (pre_ms * 1e-3) / 1e12
    return {"step_ms": round(sum(per) / len(per), 5), "prefill_ms": round(pre_ms, 5),
            "flops": flops, "timing": "graph replays, L2 flushed before each",
            "tflops": round(tf, 2), "frac_of_bf16_peak": round(tf / peaks["bf16_tflops"], 4),
            "frac_of_bf16_sustained": round(tf / peaks["bf16_tflops_sustained"], 4),
            "kernel_ms_eager": {n: round(v[0] / max(v[1], 1), 5) for n, v in kt.items()},
            "kernels": "store_kvcache_int8; prefill_int8 = the tcgen05 prefill kernel with "
                       "producer warps dequantising INT8 tiles to bf16 in shared memory"}


def host_block_manager(pkv, steps: int = 2000) -> dict:
    """Host cost of producing the decode inputs: the block manager (C++, behind
    the C ABI) admitting 128 prompts of 4096 tokens that share a 2048-token
    prefix, then decode steps (one call each) that append one token to each of
    the 128 sequences and fill the slot mapping, the [128, max_blocks] block
    table and the context lengths."""
    prompts = W.shared_prefix_prompts()
    b = len(prompts)
    max_blocks = -(-(4096 + steps) // W.BLOCK_SIZE)
    bm = pkv.BlockManager(8 * 1024)
    t0 = time.perf_counter()
    cached = [bm.allocate(s, p) for s, p in enumerate(prompts)]
    alloc_s = time.perf_counter() - t0
    ids = torch.arange(b, dtype=torch.int64)
    tokens = torch.zeros(b, dtype=torch.int32)
    slots = torch.empty(b, dtype=torch.int32)
    tables = torch.empty(b, max_blocks, dtype=torch.int32)
    lens = torch.empty(b, dtype=torch.int32)
    t0 = time.perf_counter()
    for i in range(steps):
        tokens.fill_(i)
        bm.decode_step_into(ids, tokens, slots, tables, lens)
    step_s = (time.perf_counter() - t0) / steps
    ok = bool((lens == 4096 + steps).all()) and bm.num_free_blocks() == 8 * 1024 - (
        2048 // W.BLOCK_SIZE + b * (-(-(4096 + steps) // W.BLOCK_SIZE) - 2048 // W.BLOCK_SIZE))
    bm.close()
    return {"unit": "us (host, one thread)", "num_seqs": b,
            "allocate_us_per_prompt": round(alloc_s / b * 1e6, 2),
            "cached_tokens_first_prompt": cached[0], "cached_tokens_others": cached[1],
            "decode_step_us": round(step_s * 1e6, 3), "decode_steps": steps,
            "pool_accounting_ok": ok}


def run_single(args, rank, world, local):
    """One non-default workload alone: its warm-up and timed steps, one JSON line."""
    import paged_kv_cache_493_b300 as pkv
    from paged_kv_cache_493_b300 import _build
    _build.build()
    pkv.load_library()
    torch.cuda.set_device(local)
    peaks, _ = load_peaks()
    res = other_workloads(pkv, args, rank, Flusher(), peaks, only=args.workload)
    if rank == 0:
        print(json.dumps({"workload": args.workload, **res[args.workload]}), flush=True)


# ----------------------------------------------------------------------------- oracle arm
def oracle_step_sample(case, seqs):
    """store + decode of the listed sequences on the CPU oracle; returns KV bytes processed."""
    import oracle
    c = case.cache
    sel = torch.tensor(seqs, dtype=torch.long)
    kc, vc = oracle.store_kvcache(case.k_new[sel], case.v_new[sel], case.slot_mapping[sel],
                                  c.k_cache, c.v_cache)
    oracle.decode(case.q[sel], kc, vc, c.block_tables[sel], c.context_lens[sel], case.scale)
    hkv, d = int(c.k_cache.shape[2]), int(c.k_cache.shape[3])
    return int(c.context_lens[sel].sum()) * hkv * d * 4


def oracle_step_parallel(case, seqs, workers):
    """store + decode of the listed sequences on the CPU oracle over `workers`
    host threads (oracle.parallel: the same C functions, one task per
    sequence); returns KV bytes processed."""
    import oracle
    import oracle.parallel as op
    c = case.cache
    sel = torch.tensor(seqs, dtype=torch.long)
    kc, vc = oracle.store_kvcache(case.k_new[sel], case.v_new[sel], case.slot_mapping[sel],
                                  c.k_cache, c.v_cache)
    op.decode(case.q[sel], kc, vc, c.block_tables[sel], c.context_lens[sel], case.scale,
              workers=workers)
    hkv, d = int(c.k_cache.shape[2]), int(c.k_cache.shape[3])
    return int(c.context_lens[sel].sum()) * hkv * d * 4


def cpu_baseline(case, bytes_, budget_s: float = 12.0):
    """The oracle as it stands (fp64 C) on a bounded sample of the workload:
    single-threaded, and over every host core (one task per sequence)."""
    import oracle.parallel as op
    n = case.num_seqs
    cores = op.host_cores()

    def leg(workers, batch):
        t0 = time.perf_counter()
        kv, i = 0, 0
        while i < n and time.perf_counter() - t0 < budget_s:
            chunk = list(range(i, min(n, i + batch)))
            kv += (oracle_step_sample(case, chunk) if workers == 1
                   else oracle_step_parallel(case, chunk, workers))
            i += len(chunk)
        return kv / (time.perf_counter() - t0) / 1e9, i, time.perf_counter() - t0

    one, n1, t1 = leg(1, 16)
    many, nm, tm = leg(cores, max(cores, 16))
    return {"value": round(many, 6), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "host_cpu_count": os.cpu_count(),
            "sample": f"store + decode of {nm} of {n} sequences (all heads), {tm:.1f} s, fp64 C "
                      f"over {cores} threads (one sequence per task)",
            "single_core": {"value": round(one, 6), "cores": 1,
                            "sample": f"store + decode of {n1} of {n} sequences, {t1:.1f} s"}}


def run_reference(args, rank, world):
    if rank != 0:
        return
    import oracle.parallel as op
    case = W.qwen_decode(seed=1002)
    cores = op.host_cores()
    per_step = min(case.num_seqs, max(8, cores))  # sequences per step: a bounded sample
    n = case.num_seqs
    for i in range(args.warmup):
        oracle_step_parallel(case, [(i * per_step + j) % n for j in range(per_step)], cores)
    times, kv = [], 0
    for i in range(args.steps):
        seqs = [(i * per_step + j) % n for j in range(per_step)]
        t0 = time.perf_counter()
        kv += oracle_step_parallel(case, seqs, cores)
        times.append(time.perf_counter() - t0)
    total = sum(times)
    value = kv / total / 1e9
    line = {
        "impl": "reference",
        "metric": METRIC, "value": round(value, 6), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": MAIN_WORKLOAD, "num_seqs": n, "num_q_heads": 16, "num_kv_heads": 8,
                   "head_dim": 128, "block_size": 256, "num_blocks": case.cache.num_blocks,
                   "parallelism": "host cores"},
        "cpu_baseline": {"value": round(value, 6), "unit": "GB/s", "cores": cores,
                         "kind": "oracle", "host_cpu_count": os.cpu_count(),
                         "sample": f"each step: store + decode of {per_step} of {n} sequences, "
                                   f"fp64 C over {cores} threads (one sequence per task)"},
        "e2e": {"value": round(value, 6), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["pkv", "reference"], default="pkv")
    ap.add_argument("--only-main", action="store_true", help="skip the other workloads")
    ap.add_argument("--workload", default=MAIN_WORKLOAD,
                    choices=[MAIN_WORKLOAD, "long_decode_32k", "prefix_decode_b64",
                             "chunked_prefill_8x512", "qwen_decode_b128_int8",
                             "chunked_prefill_8x512_int8"],
                    help="run one non-default workload alone (for profiling) and print its entry")
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "pkv":
        args.warmup = 3
    if args.gpus > 1 and int(os.environ.get("WORLD_SIZE", "1")) == 1:
        # N replicas need one process per GPU: start them under torchrun.
        if args.impl == "pkv" and torch.cuda.device_count() < args.gpus:
            sys.exit(f"--gpus {args.gpus}: only {torch.cuda.device_count()} CUDA device(s) visible")
        import socket
        with socket.socket() as s:
            s.bind(("127.0.0.1", 0))
            port = s.getsockname()[1]
        cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
               f"--nproc-per-node={args.gpus}", "--master-addr=127.0.0.1",
               f"--master-port={port}", os.path.abspath(__file__)] + list(
                   argv if argv is not None else sys.argv[1:])
        sys.exit(subprocess.call(cmd))
    rank, world, local = dist_setup()
    if world != args.gpus:
        sys.exit(f"--gpus {args.gpus} but WORLD_SIZE={world}: launch one process per GPU")
    try:
        if args.impl == "reference":
            run_reference(args, rank, world)
        elif args.workload != MAIN_WORKLOAD:
            run_single(args, rank, world, local)
        else:
            run_gpu(args, rank, world, local)
    finally:
        if torch.distributed.is_available() and torch.distributed.is_initialized():
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
