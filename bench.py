"""Benchmark one continuous-batching paged-attention step through libcb's C ABI.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--config decode|mixed|long_decode|long_decode_window|tiny_mixed|trace]

A step is the whole hot path on one synthetic batch: scatter of the step's new
K/V through slot_mapping, then paged attention of every query row (decode and
prefill rows). The default workload is the pure-decode step: 64 requests,
q_len 1, seq_len ~ U{128..2048}, 32 Q / 8 KV heads, head_dim 128,
block_size 16, bf16.

Reported metric: achieved KV-read HBM bandwidth (algorithmic KV bytes of the
step, every attended position of every request counted once, over the step's
device time) and query tokens/s, with the roofline of the dominant kernel
against the measured HBM copy bandwidth. The step's KV is larger than L2
(129 MB); between timed steps a 512 MiB read evicts the previous step's lines
and leaves L2 clean (``--flush write`` writes 512 MiB instead, which leaves
dirty lines whose write-back then competes with the step's reads). With N > 1 (torchrun), every rank runs an independent
replica of the step (the path needs no exchange) and the job value is the sum
of the bytes over the slowest rank's time.

``--config trace`` replays the FIFO continuous-batching trace (512 requests,
lognormal prompts, geometric outputs, max_batch_tokens 4096, 65536 pages of 16
tokens) step by step: every step is scatter + attention of that step's batch,
timed on its own; the line reports the whole trace's KV GB/s and tokens/s with
per-step percentiles. ``--config trace_prefill_first`` replays the same request
stream under the prefill-first policy (safety margin 0). ``--config copy_blocks``
times the batched block copy behind swapping (8192 blocks of 32 KB for K and V
between disjoint pool blocks; bytes read + written).

``--impl reference`` times the CPU oracle (float64 NumPy, as it stands) on the
same workload instead, on the host cores.
"""
from __future__ import annotations

import os

# the oracle leg is timed single-threaded; set before numpy loads
for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import argparse
import hashlib
import datetime
import json
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

FLUSH_BYTES = 512 << 20
GRAPH_Q_INTERVAL = 64  # query padding interval of --graph (the decode step's 64 requests fit)
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
# the default line: the long-context decode step (the largest single-GPU workload), with the
# mixed continuous-batching step and the windowed long decode measured beside it
DEFAULT_CONFIG = "long_decode"
EXTRA_CONFIGS = ("mixed", "long_decode_window")


# ---------------------------------------------------------------- accounting


def kv_bytes(spec) -> int:
    """Algorithmic KV bytes: every attended position of every request once, K and V."""
    return spec.kv_tokens_attended() * 2 * spec.num_kv_heads * spec.head_dim * spec.elt_bytes()


def decode_kernel_bytes(spec) -> int:
    """Algorithmic bytes of the decode kernel: decode rows' KV + their q and out."""
    e = spec.elt_bytes()
    n = 0
    for r in range(spec.R):
        if int(spec.q_lens[r]) != 1:
            continue
        ctx = int(spec.ctx_lens[r])
        lo = 0 if spec.sliding_window <= 0 else max(0, ctx - spec.sliding_window + 1)
        n += (ctx - lo + 1) * 2 * spec.num_kv_heads * spec.head_dim * e
        n += 2 * spec.num_q_heads * spec.head_dim * e
    return n


def prefill_flops(spec) -> int:
    """Algorithmic FLOPs of the prefill rows (q_len > 1): 4 x Hq x D per attended
    (query, key) pair -- the causal (and windowed) pairs only, not the dense tiles."""
    pairs = 0
    for r in range(spec.R):
        ql = int(spec.q_lens[r])
        if ql <= 1:
            continue
        ctx = int(spec.ctx_lens[r])
        for i in range(ql):
            hi = ctx + i
            lo = 0 if spec.sliding_window <= 0 else max(0, hi - spec.sliding_window + 1)
            pairs += hi - lo + 1
    return 4 * spec.num_q_heads * spec.head_dim * pairs


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def bf16_peak():
    """Dense bf16 TFLOP/s for a kernel timed alone (burst), and where it comes from."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_BF16_TFLOPS, "fallback"


def kernel_source_sha(name: str) -> str:
    src = os.path.join(ROOT, "paged_kv_attention_cb_gb300", "csrc", name)
    try:
        with open(src, "rb") as f:
            return hashlib.sha256(f.read()).hexdigest()[:16]
    except OSError:
        return ""


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if the kernel source still matches."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)[kernel]
    except Exception:
        return None
    if rec.get("workload") != workload or rec.get("source_sha") != kernel_source_sha(rec["source"]):
        return None
    return rec.get("dram_bytes_per_launch")


# ---------------------------------------------------------------- clocks


class ClockSampler:
    """nvidia-smi samples of the SM clock and throttle reasons around a timed region.

    Sampling starts before the region (the `with` block) and runs until a sample after
    it has arrived; the summary takes the samples stamped inside the region, or, for a
    region shorter than the sampling period, the two samples that bracket it."""

    PERIOD_MS = 50

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.t0 = self.t1 = None
        # raw samples (the JSON line carries their summary); CB_BENCH_CLOCKS_DIR keeps them
        self.path = os.path.join(os.environ.get("CB_BENCH_CLOCKS_DIR", tempfile.gettempdir()),
                                 f"bench_clocks_{os.getpid()}.csv")

    def _lines(self):
        try:
            with open(self.path) as f:
                return f.read().splitlines()
        except OSError:
            return []

    def _wait_for(self, pred, timeout_s):
        end = time.time() + timeout_s
        while time.time() < end:
            if pred(self._rows()):
                return
            time.sleep(0.01)

    def __enter__(self):
        q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w", buffering=1)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={q}", "--format=csv,noheader",
                 "-lms", str(self.PERIOD_MS)], stdout=self.f, stderr=subprocess.DEVNULL)
            self._wait_for(lambda rows: len(rows) >= 1, 5.0)  # sampling is live
        except Exception:
            self.proc = None
        self.t0 = datetime.datetime.now()
        return self

    def __exit__(self, *exc):
        self.t1 = datetime.datetime.now()
        if self.proc is not None:
            self._wait_for(lambda rows: any(r[0] > self.t1 for r in rows), 2.0)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def _rows(self):
        rows = []
        for line in self._lines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f")
                rows.append((ts, float(parts[2].split()[0]), float(parts[3].split()[0]),
                             parts[6:10]))
            except ValueError:
                continue
        return rows

    def summary(self):
        if self.proc is None or self.t0 is None or self.t1 is None:
            return None
        rows = self._rows()
        inside = [r for r in rows if self.t0 <= r[0] <= self.t1]
        window = "inside"
        if not inside:
            before = [r for r in rows if r[0] < self.t0][-1:]
            after = [r for r in rows if r[0] > self.t1][:1]
            inside = before + after
            window = "bracketing (timed region shorter than the sampling period)"
        if not inside:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in inside:
            for n, v in zip(names, r[3]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(r[1] for r in inside),
                "sm_max_mhz": max(r[2] for r in inside), "samples": len(inside),
                "window": window, "reasons": sorted(reasons)}


class NvmlClockSampler:
    """SM clock and throttle reasons read through NVML every PERIOD_S on a background
    thread, from just before the timed region to just after it, so that even a
    region of a few milliseconds holds samples. Falls back to ClockSampler (nvidia-smi)
    where libnvidia-ml cannot be loaded."""

    PERIOD_S = 0.002
    # nvmlClocksEventReason bits
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown"}

    def __init__(self, index: int):
        import ctypes
        import threading

        self.index = index
        self.samples = []  # (time, sm_mhz, reasons)
        self.t0 = self.t1 = None
        self.max_mhz = None
        self._stop = threading.Event()
        self._thread = None
        self._fallback = None
        try:
            self.nvml = ctypes.CDLL("libnvidia-ml.so.1")
            if self.nvml.nvmlInit_v2() != 0:
                raise OSError("nvmlInit failed")
            self.handle = ctypes.c_void_p()
            found = False
            try:  # the CUDA device's own GPU (NVML numbers every GPU of the machine)
                import torch

                uuid = "GPU-" + str(torch.cuda.get_device_properties(index).uuid)
                found = self.nvml.nvmlDeviceGetHandleByUUID(uuid.encode(),
                                                            ctypes.byref(self.handle)) == 0
            except Exception:
                found = False
            if not found and self.nvml.nvmlDeviceGetHandleByIndex_v2(
                    index, ctypes.byref(self.handle)) != 0:
                raise OSError("no NVML handle")
            fn = getattr(self.nvml, "nvmlDeviceGetCurrentClocksEventReasons", None)
            self.reasons_fn = fn or self.nvml.nvmlDeviceGetCurrentClocksThrottleReasons
            mx = ctypes.c_uint()
            if self.nvml.nvmlDeviceGetMaxClockInfo(self.handle, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = float(mx.value)
        except (OSError, AttributeError):
            self.nvml = None
            self._fallback = ClockSampler(index)

    def _sample(self):
        import ctypes

        mhz = ctypes.c_uint()
        rs = ctypes.c_ulonglong()
        if self.nvml.nvmlDeviceGetClockInfo(self.handle, 1, ctypes.byref(mhz)) != 0:
            return
        if self.reasons_fn(self.handle, ctypes.byref(rs)) != 0:
            rs.value = 0
        self.samples.append((time.perf_counter(), float(mhz.value), int(rs.value)))

    def _run(self):
        while not self._stop.is_set():
            self._sample()
            time.sleep(self.PERIOD_S)

    def __enter__(self):
        import threading

        if self._fallback is not None:
            self._fallback.__enter__()
            return self
        self._sample()
        self._thread = threading.Thread(target=self._run, daemon=True)
        self._thread.start()
        self.t0 = time.perf_counter()
        return self

    def __exit__(self, *exc):
        if self._fallback is not None:
            return self._fallback.__exit__(*exc)
        self.t1 = time.perf_counter()
        time.sleep(2 * self.PERIOD_S)
        self._stop.set()
        self._thread.join(timeout=1.0)

    def summary(self):
        if self._fallback is not None:
            return self._fallback.summary()
        if self.t0 is None or self.t1 is None:
            return None
        inside = [x for x in self.samples if self.t0 <= x[0] <= self.t1]
        window = "inside"
        if not inside:
            before = [x for x in self.samples if x[0] < self.t0][-1:]
            after = [x for x in self.samples if x[0] > self.t1][:1]
            inside = before + after
            window = "bracketing (timed region shorter than the sampling period)"
        if not inside:
            return None
        reasons = sorted({name for x in inside for bit, name in self.REASONS.items() if x[2] & bit})
        return {"sm_mhz": statistics.median(x[1] for x in inside),
                "sm_max_mhz": self.max_mhz if self.max_mhz else max(x[1] for x in inside),
                "samples": len(inside), "window": window, "reasons": reasons,
                "source": f"NVML every {1e3 * self.PERIOD_S:.0f} ms"}


# ---------------------------------------------------------------- distributed


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("gloo", init_method="env://")
    return world, rank, local


def reduce_max(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


# ---------------------------------------------------------------- our arm


def run_ours(args, spec, world, rank, local):
    import torch

    import paged_kv_attention_cb_gb300 as cb

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    x = workloads.draw_tensors(spec, dev)
    md = workloads.metadata_tensors(spec, dev)
    ws = cb.alloc_workspace(spec.R, spec.T, spec.num_q_heads, spec.num_kv_heads, spec.head_dim,
                            dev)
    out = torch.empty_like(x["q"])
    flush_buf = torch.ones(FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
    graph = None
    if args.graph:
        # graphs need a created stream; the step's buffers are the persistent ones above
        graph = cb.GraphCache(q_interval=GRAPH_Q_INTERVAL)
        torch.cuda.set_stream(torch.cuda.Stream(dev))
    stream = torch.cuda.current_stream(dev)

    class Flush:
        def fill_(self, v):
            if args.flush == "write":
                flush_buf.fill_(v)
            else:
                flush_buf.max()  # reads every line; the result is discarded

    flush = Flush()

    def attention(*a, **k):
        if graph is None:
            return cb.paged_attention(*a, ring_blocks=spec.ring_blocks, **k)
        return cb.paged_attention_graphed(graph, *a, **k)

    def eager_step():
        cb.paged_attention(out, x["q"], x["k_cache"], x["v_cache"], md["query_start_loc"],
                           md["seq_lens"], md["block_table"], spec.query_start_loc,
                           spec.seq_lens, ws, scale=spec.scale,
                           sliding_window=spec.sliding_window, ring_blocks=spec.ring_blocks,
                           k_new=x["k_new"], v_new=x["v_new"], slot_mapping=md["slot_mapping"],
                           stream=stream)

    def step():
        if graph is None:
            return eager_step()
        attention(out, x["q"], x["k_cache"], x["v_cache"], md["query_start_loc"],
                  md["seq_lens"], md["block_table"], spec.query_start_loc, spec.seq_lens, ws,
                  scale=spec.scale, sliding_window=spec.sliding_window, k_new=x["k_new"],
                  v_new=x["v_new"], slot_mapping=md["slot_mapping"], stream=stream)

    for _ in range(args.warmup):
        flush.fill_(1)
        step()
    torch.cuda.synchronize()
    if cb.read_error_word(ws) != 0:
        raise RuntimeError("device bounds check fired during warm-up")

    # ---- timed region: per-step CUDA events on the launching stream, L2 flushed between steps
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    stops = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    launches0 = cb.launch_count()
    barrier(world)
    torch.cuda.synchronize()
    with NvmlClockSampler(local) as clocks:
        for i in range(args.steps):
            flush.fill_(i & 0xFF)
            starts[i].record(stream)
            step()
            stops[i].record(stream)
        torch.cuda.synchronize()
    barrier(world)
    launches = cb.launch_count() - launches0
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, stops)]
    local_ms = sum(step_ms)
    total_ms = reduce_max(local_ms, world)
    ms_per_step = total_ms / args.steps

    # ---- the same steps after a dirty (write) flush, for comparison
    alt_ms = None
    if args.flush == "read":
        a0 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        a1 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        for i in range(args.steps):
            flush_buf.fill_(i & 0xFF)
            a0[i].record(stream)
            step()
            a1[i].record(stream)
        torch.cuda.synchronize()
        alt_ms = reduce_max(sum(s.elapsed_time(e) for s, e in zip(a0, a1)), world) / args.steps

    # ---- per-kernel attribution pass (same steps, events around each launch; graph
    # replays are not timed per kernel, so this pass runs the same kernels eagerly)
    cb.kernel_timing(True)
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        eager_step()
    per_kernel = cb.kernel_timing_collect()
    cb.kernel_timing(False)

    # ---- end to end through the public API: pinned host inputs in, result out. The
    # step's inputs (q, k_new, v_new and the four metadata arrays) sit packed in one pinned
    # host buffer and go over in one copy; the output comes back in one copy.
    parts = [("q", x["q"]), ("k_new", x["k_new"]), ("v_new", x["v_new"])] + list(md.items())
    offs, total = {}, 0
    for k, v in parts:
        offs[k] = total
        total += (v.numel() * v.element_size() + 255) // 256 * 256
    host_buf = torch.empty(total, dtype=torch.uint8, pin_memory=True)
    dev_buf = torch.empty(total, dtype=torch.uint8, device=dev)

    def view(buf, k, like):
        n = like.numel() * like.element_size()
        return buf[offs[k]:offs[k] + n].view(like.dtype).view(like.shape)

    for k, v in parts:
        view(host_buf, k, v).copy_(v.cpu())
    dv = {k: view(dev_buf, k, v) for k, v in parts}
    host_out = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    h2d = sum(v.numel() * v.element_size() for _, v in parts)
    d2h = host_out.numel() * host_out.element_size()

    def e2e_step():
        dev_buf.copy_(host_buf, non_blocking=True)
        attention(out, dv["q"], x["k_cache"], x["v_cache"], dv["query_start_loc"],
                  dv["seq_lens"], dv["block_table"], spec.query_start_loc, spec.seq_lens, ws,
                  scale=spec.scale, sliding_window=spec.sliding_window, k_new=dv["k_new"],
                  v_new=dv["v_new"], slot_mapping=dv["slot_mapping"], stream=stream)
        host_out.copy_(out, non_blocking=True)

    for _ in range(max(1, args.warmup)):
        e2e_step()
    torch.cuda.synchronize()
    e_starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    e_stops = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier(world)
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        e_starts[i].record(stream)
        e2e_step()
        e_stops[i].record(stream)
    torch.cuda.synchronize()
    e2e_serial_ms = reduce_max(sum(s.elapsed_time(e) for s, e in zip(e_starts, e_stops)), world)
    barrier(world)

    # ---- the same end-to-end steps pipelined, as a serving loop runs them: every step
    # still copies its own inputs in (one packed copy) and its result out (one copy) inside
    # the timed region, but step i+1's copy-in (on an upload stream) and step i-1's
    # copy-out (on a download stream) overlap step i's kernels. Inputs and outputs are
    # double-buffered on the device; events order each buffer's reuse. Each cudaMemcpyAsync
    # costs ~11 us of latency on these boxes whatever its size, which the serial steps pay
    # twice per step.
    up, down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    dev_bufs = [dev_buf, torch.empty_like(dev_buf)]
    outs = [out, torch.empty_like(out)]
    host_outs = [host_out, torch.empty(out.shape, dtype=out.dtype, pin_memory=True)]
    dvs = [{k: view(b, k, v) for k, v in parts} for b in dev_bufs]

    def pipelined(n):
        ev_in = [torch.cuda.Event() for _ in range(n)]
        ev_done = [torch.cuda.Event() for _ in range(n)]
        ev_out = [torch.cuda.Event() for _ in range(n)]
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        prev = torch.cuda.current_stream()
        # copies run on the current stream; a `with torch.cuda.stream(...)` block around
        # each would cost ~10 us of host time per copy, more than the copy's own enqueue
        torch.cuda.set_stream(up)
        t0.record(up)
        for i in range(n):
            b = i & 1
            if i >= 2:
                up.wait_event(ev_done[i - 2])  # step i-2 no longer reads this input buffer
            dev_bufs[b].copy_(host_buf, non_blocking=True)
            ev_in[i].record(up)
            stream.wait_event(ev_in[i])
            if i >= 2:
                stream.wait_event(ev_out[i - 2])  # step i-2's result is copied out
            d = dvs[b]
            attention(outs[b], d["q"], x["k_cache"], x["v_cache"], d["query_start_loc"],
                      d["seq_lens"], d["block_table"], spec.query_start_loc, spec.seq_lens, ws,
                      scale=spec.scale, sliding_window=spec.sliding_window, k_new=d["k_new"],
                      v_new=d["v_new"], slot_mapping=d["slot_mapping"], stream=stream)
            ev_done[i].record(stream)
            down.wait_event(ev_done[i])
            torch.cuda.set_stream(down)
            host_outs[b].copy_(outs[b], non_blocking=True)
            torch.cuda.set_stream(up)
            ev_out[i].record(down)
        up.wait_event(ev_out[n - 1])
        t1.record(up)
        torch.cuda.set_stream(prev)
        torch.cuda.synchronize()
        return t0.elapsed_time(t1)

    pipelined(max(2, args.warmup))
    barrier(world)
    e2e_ms = reduce_max(pipelined(args.steps), world)
    barrier(world)
    # ---- host-bound regime: steps back to back (no flush, one sync at the end)
    def wall_us(fn, n=200):
        fn()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(n):
            fn()
        torch.cuda.synchronize()
        return 1e6 * (time.perf_counter() - t0) / n

    def host_us(fn, n=200):
        fn()
        torch.cuda.synchronize()
        t = 0.0
        for _ in range(n):
            t0 = time.perf_counter()
            fn()
            t += time.perf_counter() - t0
        torch.cuda.synchronize()
        return 1e6 * t / n

    graph_info = None
    if graph is not None:
        hq = np.ascontiguousarray(spec.query_start_loc, dtype=np.int32)
        hs = np.ascontiguousarray(spec.seq_lens, dtype=np.int32)
        prepared = cb.PreparedGraphStep(
            graph, out, x["q"], x["k_cache"], x["v_cache"], md["query_start_loc"],
            md["seq_lens"], md["block_table"], hq, hs, ws, scale=spec.scale,
            sliding_window=spec.sliding_window, k_new=x["k_new"], v_new=x["v_new"],
            slot_mapping=md["slot_mapping"], stream=stream)
        graph_info = {"q_interval": GRAPH_Q_INTERVAL,
                      "wall_us_per_step_graphed": wall_us(prepared),
                      "wall_us_per_step_eager": wall_us(eager_step),
                      "host_us_per_call_graphed_prepared": host_us(prepared),
                      "host_us_per_call_graphed": host_us(step),
                      "host_us_per_call_eager": host_us(eager_step)}
        graph_info.update(graph.stats())
        # a host-bound batch: 64 decodes over 16..128 positions (a few us on the device)
        small = workloads.decode_step(seed=11, lo=16, hi=128)
        xs = workloads.draw_tensors(small, dev)
        mds = workloads.metadata_tensors(small, dev)
        wss = cb.alloc_workspace(small.R, small.T, small.num_q_heads, small.num_kv_heads,
                                 small.head_dim, dev)
        outs = torch.empty_like(xs["q"])
        kw = dict(scale=small.scale, k_new=xs["k_new"], v_new=xs["v_new"],
                  slot_mapping=mds["slot_mapping"], stream=stream)
        args_s = (outs, xs["q"], xs["k_cache"], xs["v_cache"], mds["query_start_loc"],
                  mds["seq_lens"], mds["block_table"], small.query_start_loc, small.seq_lens, wss)
        g2 = cb.GraphCache(q_interval=GRAPH_Q_INTERVAL)
        prep_s = cb.PreparedGraphStep(
            g2, outs, xs["q"], xs["k_cache"], xs["v_cache"], mds["query_start_loc"],
            mds["seq_lens"], mds["block_table"],
            np.ascontiguousarray(small.query_start_loc, dtype=np.int32),
            np.ascontiguousarray(small.seq_lens, dtype=np.int32), wss, **kw)
        graph_info["small_decode"] = {
            "workload": small.name,
            "wall_us_per_step_graphed": wall_us(prep_s),
            "wall_us_per_step_eager": wall_us(lambda: cb.paged_attention(*args_s, **kw))}
        g2.close()
    return dict(ms_per_step=ms_per_step, step_ms=step_ms, launches=launches, alt_ms=alt_ms,
                per_kernel=per_kernel, e2e_ms_per_step=e2e_ms / args.steps, h2d=h2d, d2h=d2h,
                h2d_copies=1, e2e_serial_ms_per_step=e2e_serial_ms / args.steps,
                clocks=clocks.summary(), graph=graph_info)


# ---------------------------------------------------------------- oracle


def oracle_inputs(spec):
    """Host float64-ready copies of the step's seeded inputs (CPU torch generator)."""
    x = workloads.draw_tensors(spec, "cpu")
    f = lambda t: t.float().numpy()
    return {k: f(v) for k, v in x.items()}


def time_oracle(spec, budget_s: float, h=None, max_steps=None):
    """Run whole oracle steps (scatter + attention) until the time budget is spent."""
    import oracle

    if h is None:
        h = oracle_inputs(spec)
    done = 0
    t0 = time.perf_counter()
    while True:
        oracle.step(h["q"], h["k_cache"], h["v_cache"], h["k_new"], h["v_new"], spec.slot_mapping,
                    spec.query_start_loc, spec.seq_lens, spec.block_table, spec.block_size,
                    spec.scale, spec.sliding_window, ring_blocks=spec.ring_blocks)
        done += 1
        el = time.perf_counter() - t0
        if el >= budget_s or (max_steps is not None and done >= max_steps):
            return done, el


def oracle_all_cores(config, budget_s):
    """The same oracle timing in a child process whose BLAS may use every host core
    (this process pins it to one thread before NumPy loads)."""
    cores = os.cpu_count() or 1
    env = dict(os.environ)
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[v] = str(cores)
    code = ("import bench, workloads, json\n"
            f"spec = workloads.by_name({config!r})\n"
            f"sample, what = bench.oracle_sample_spec(spec, bench.oracle_sample_size({config!r}))\n"
            f"n, el = bench.time_oracle(sample, {float(budget_s)!r})\n"
            "print(json.dumps({'value': bench.kv_bytes(sample) * n / el / 1e9, 'steps': n, 'seconds': el}))\n")
    try:
        out = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True,
                             text=True, timeout=max(120.0, 6 * budget_s))
        r = json.loads(out.stdout.strip().splitlines()[-1])
        r["cores"] = cores
        return r
    except Exception as e:  # the figure is context; the bench line does not depend on it
        return {"error": str(e)[:200], "cores": cores}


def oracle_sample_spec(spec, max_requests=None):
    """A bounded sample of the workload for the oracle: the first requests of the step."""
    if max_requests is None or max_requests >= spec.R:
        return spec, "whole step"
    r = max_requests
    s = workloads.StepSpec(**{**spec.__dict__})
    s.q_lens = spec.q_lens[:r]
    s.ctx_lens = spec.ctx_lens[:r]
    s.query_start_loc = spec.query_start_loc[:r + 1]
    s.seq_lens = spec.seq_lens[:r]
    s.block_table = spec.block_table[:r]
    s.slot_mapping = spec.slot_mapping[:int(spec.query_start_loc[r])]
    return s, f"first {r} of {spec.R} requests"


def oracle_sample_size(config):
    # requests per oracle sample so that one sample takes a few seconds at most
    return {"decode": None, "tiny_mixed": None, "mixed": 24, "long_decode": 2,
            "long_decode_window": 8, "long_decode_ring": 8}.get(config)


# ---------------------------------------------------------------- trace (c5)


def compact_spec(spec):
    """The same step over a pool holding only its own pages (renumbered after the
    reserved ones), so that the oracle can be timed on it without the whole pool."""
    used = sorted({int(p) for r in range(spec.R)
                   for p in spec.block_table[r, :-(-int(spec.seq_lens[r]) // spec.block_size)]})
    remap = {p: workloads.RESERVED_PAGES + i for i, p in enumerate(used)}
    bt = np.zeros_like(spec.block_table)
    for r in range(spec.R):
        n = -(-int(spec.seq_lens[r]) // spec.block_size)
        bt[r, :n] = [remap[int(p)] for p in spec.block_table[r, :n]]
    slots = np.array([remap[int(s) // spec.block_size] * spec.block_size + int(s) % spec.block_size
                      for s in spec.slot_mapping], dtype=np.int64)
    return workloads.StepSpec(**{**spec.__dict__, "block_table": bt, "slot_mapping": slots,
                                 "num_blocks": workloads.RESERVED_PAGES + len(used)})


def trace_specs(n_steps=0, policy="fifo"):
    from workloads.fifo_trace import TraceConfig, fifo_trace, prefill_first_config

    cfg = TraceConfig() if policy == "fifo" else prefill_first_config()
    specs = [st.spec for st in fifo_trace(cfg, max_steps=n_steps or None)]
    return cfg, specs


def run_trace_ours(args, cfg, specs, world, rank, local):
    """Every trace step through the C ABI with the cache carried from step to step."""
    import torch

    import paged_kv_attention_cb_gb300 as cb

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    g = torch.Generator(device=dev)
    g.manual_seed(cfg.seed)
    shape = (cfg.num_pages, cfg.block_size, cfg.num_kv_heads, cfg.head_dim)
    k_cache = torch.randn(*shape, generator=g, device=dev).to(torch.bfloat16)
    v_cache = torch.randn(*shape, generator=g, device=dev).to(torch.bfloat16)
    max_r = max(sp.R for sp in specs)
    max_t = max(sp.T for sp in specs)
    ws = cb.alloc_workspace(max_r, max_t, cfg.num_q_heads, cfg.num_kv_heads, cfg.head_dim, dev)
    out_buf = torch.empty(max_t, cfg.num_q_heads, cfg.head_dim, dtype=torch.bfloat16, device=dev)
    flush_buf = torch.ones(FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
    # every step's inputs drawn once (seed = trace seed + step), resident in HBM
    steps = []
    for sp in specs:
        gs = torch.Generator(device=dev)
        gs.manual_seed(int(sp.seed))
        f = lambda *sh: torch.randn(*sh, generator=gs, device=dev).to(torch.bfloat16)
        q = f(sp.T, sp.num_q_heads, sp.head_dim)
        kn = f(sp.T, sp.num_kv_heads, sp.head_dim)
        vn = f(sp.T, sp.num_kv_heads, sp.head_dim)
        steps.append((sp, q, kn, vn, workloads.metadata_tensors(sp, dev)))
    torch.cuda.synchronize()

    def call(i, q=None, kn=None, vn=None, md=None):
        sp, q0, kn0, vn0, md0 = steps[i]
        md = md or md0
        cb.paged_attention(out_buf[:sp.T], q0 if q is None else q, k_cache, v_cache,
                           md["query_start_loc"], md["seq_lens"], md["block_table"],
                           sp.query_start_loc, sp.seq_lens, ws, scale=sp.scale,
                           k_new=kn0 if kn is None else kn, v_new=vn0 if vn is None else vn,
                           slot_mapping=md["slot_mapping"], stream=stream)

    n = len(steps)
    for i in range(min(args.warmup, n)):
        call(i)
    torch.cuda.synchronize()
    if cb.read_error_word(ws) != 0:
        raise RuntimeError("device bounds check fired during warm-up")

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(n)]
    launches0 = cb.launch_count()
    barrier(world)
    torch.cuda.synchronize()
    with NvmlClockSampler(local) as clocks:
        for i in range(n):
            flush_buf.max()  # evicts L2 (clean) between steps
            ev[i][0].record(stream)
            call(i)
            ev[i][1].record(stream)
        torch.cuda.synchronize()
    barrier(world)
    launches = cb.launch_count() - launches0
    if cb.read_error_word(ws) != 0:
        raise RuntimeError("device bounds check fired during the trace")
    step_ms = [a.elapsed_time(b) for a, b in ev]

    cb.kernel_timing(True)
    for i in range(n):
        flush_buf.max()
        call(i)
    per_kernel = cb.kernel_timing_collect()
    cb.kernel_timing(False)

    # end to end: each step's inputs and metadata packed in one pinned host buffer and
    # copied in one transfer; the output back in one transfer
    def packed(parts):
        offs, total = {}, 0
        for k, v in parts:
            offs[k] = total
            total += (v.numel() * v.element_size() + 255) // 256 * 256
        return offs, total

    sizes = [packed([("q", q), ("k", kn), ("v", vn)] + list(md.items()))[1]
             for _, q, kn, vn, md in steps[:n]]
    cap = max(sizes) if sizes else 256
    host_buf = torch.empty(cap, dtype=torch.uint8, pin_memory=True)
    dev_buf = torch.empty(cap, dtype=torch.uint8, device=dev)
    ho = torch.empty(max_t * cfg.num_q_heads * cfg.head_dim, dtype=torch.bfloat16,
                     pin_memory=True)
    e2e_ms = 0.0
    h2d = d2h = 0
    for i in range(n):
        sp, q, kn, vn, md = steps[i]
        parts = [("q", q), ("k", kn), ("v", vn)] + list(md.items())
        offs, total = packed(parts)

        def view(buf, k, like):
            nb = like.numel() * like.element_size()
            return buf[offs[k]:offs[k] + nb].view(like.dtype).view(like.shape)

        for k, v in parts:
            view(host_buf, k, v).copy_(v.cpu())
        dvs = {k: view(dev_buf, k, v) for k, v in parts}
        dmd = {k: dvs[k] for k in md}
        nq = q.numel()
        torch.cuda.synchronize()
        flush_buf.max()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        dev_buf[:total].copy_(host_buf[:total], non_blocking=True)
        call(i, dvs["q"], dvs["k"], dvs["v"], dmd)
        ho[:nq].copy_(out_buf[:sp.T].view(-1), non_blocking=True)
        b.record(stream)
        torch.cuda.synchronize()
        e2e_ms += a.elapsed_time(b)
        h2d += sum(v.numel() * v.element_size() for _, v in parts)
        d2h += 2 * nq
    return dict(step_ms=step_ms, launches=launches, per_kernel=per_kernel, e2e_ms=e2e_ms,
                h2d=h2d, d2h=d2h, clocks=clocks.summary())


def trace_oracle(specs, budget_s, max_requests=24):
    """The oracle (as it stands) on evenly spaced sampled steps, each over its own
    compacted pool and at most `max_requests` requests, until the budget is spent."""
    n = len(specs)
    # coarse to fine over the trace, then its first and last steps
    ks = [8, 4, 12, 2, 6, 10, 14, 1, 3, 5, 7, 9, 11, 13, 15]
    order = list(dict.fromkeys([int(k * n / 16) for k in ks] + [0, n - 1]))
    done_b = done_t = 0
    el = 0.0
    used = []
    for i in order:
        sample = compact_spec(oracle_sample_spec(specs[i], max_requests)[0])
        h = oracle_inputs(sample)
        _, t = time_oracle(sample, 0.0, h, max_steps=1)
        el += t
        done_b += kv_bytes(sample)
        done_t += sample.T
        used.append(i)
        if el >= budget_s:
            break
    return done_b, done_t, el, used


def trace_main(args, world, rank, local, metric):
    policy = "prefill_first" if args.config == "trace_prefill_first" else "fifo"
    cfg, specs = trace_specs(args.trace_steps, policy)
    kvb = [kv_bytes(sp) for sp in specs]
    tot_b, tot_t = sum(kvb), sum(sp.T for sp in specs)
    conf = {"workload": f"{policy}_trace_512req_bf16", "requests": cfg.num_requests,
            "policy": policy,
            "trace_steps": len(specs), "query_tokens": tot_t,
            "num_q_heads": cfg.num_q_heads, "num_kv_heads": cfg.num_kv_heads,
            "head_dim": cfg.head_dim, "block_size": cfg.block_size,
            "num_blocks": cfg.num_pages, "max_batch_tokens": cfg.max_batch_tokens,
            "max_requests_per_batch": cfg.max_requests_per_batch,
            "safety_margin": cfg.safety_margin, "kv_bytes_total": tot_b,
            "l2": "512 MiB read between timed steps (L2 evicted, clean)",
            "parallelism": f"replicas x{world}"}
    if args.impl == "reference":
        if rank != 0:
            return
        b, t, el, used = trace_oracle(specs, args.cpu_budget)
        val = b / el / 1e9
        line = {"impl": "reference", "metric": metric, "value": val, "unit": "GB/s",
                "n_gpus": args.gpus, "steps": len(used), "warmup": 0,
                "ms_per_step": 1e3 * el / len(used), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": conf, "tokens_per_s": t / el,
                "cpu_baseline": {"value": val, "unit": "GB/s", "cores": 1, "kind": "oracle",
                                 "sample": f"trace steps {used}, first 24 requests each"},
                "e2e": {"value": val, "unit": "GB/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return
    res = run_trace_ours(args, cfg, specs, world, rank, local)
    total_ms = reduce_max(sum(res["step_ms"]), world)
    if rank != 0:
        return
    n = len(specs)
    value = world * tot_b / (total_ms * 1e-3) / 1e9
    peak, peak_kind = peaks()
    pk = res["per_kernel"]
    dom = max(pk.items(), key=lambda kv: kv[1][0])[0] if pk else None
    dom_ms = pk[dom][0] if dom else None  # summed over all steps
    dom_bytes = sum(decode_kernel_bytes(sp) for sp in specs) if dom == "decode_split" else None
    achieved = dom_bytes / (dom_ms * 1e-3) / 1e9 if (dom_bytes and dom_ms) else None
    roofline = {"kernel": dom, "bound": "hbm", "achieved": achieved, "peak": peak,
                "unit": "GB/s", "frac": (achieved / peak) if achieved else None,
                "peak_source": f"{peak_kind} HBM copy bandwidth",
                "algorithmic_bytes_per_launch": (dom_bytes / pk[dom][1]) if dom_bytes else None,
                "avg_launch_ms": (dom_ms / pk[dom][1]) if dom else None, "traffic": None}
    step_gbs = [b / (ms * 1e-3) / 1e9 for b, ms in zip(kvb, res["step_ms"])]
    pct = lambda a, q: float(np.percentile(np.asarray(a), q))
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        b, t, el, used = trace_oracle(specs, args.cpu_budget)
        cpu = {"value": b / el / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
               "sample": f"trace steps {used} (first 24 requests each), {el:.1f} s"}
    line = {"metric": metric, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": n, "warmup": args.warmup, "ms_per_step": total_ms / n,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic", "config": conf,
            "tokens_per_s": world * tot_t / (total_ms * 1e-3),
            "step_ms_percentiles": {q: pct(res["step_ms"], q) for q in (10, 50, 90, 99)},
            "step_gbs_percentiles": {q: pct(step_gbs, q) for q in (10, 50, 90)},
            "e2e": {"value": world * tot_b / (res["e2e_ms"] * 1e-3) / 1e9, "unit": "GB/s",
                    "ms_per_step": res["e2e_ms"] / n, "h2d_bytes_per_step": res["h2d"] / n,
                    "d2h_bytes_per_step": res["d2h"] / n},
            "gpu_launches": res["launches"],
            "per_kernel_ms": {k: v[0] / v[1] for k, v in pk.items()},
            "roofline": roofline, "cpu_baseline": cpu, "clocks": res["clocks"]}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- block copy (swap data movement)


COPY_BLOCKS = 8192


def copy_main(args, world, rank, local):
    """Batched block copy: COPY_BLOCKS pairs of disjoint blocks of a 16-token, 8-head,
    head_dim-128 bf16 pool (K and V); value = bytes read + written / device time."""
    import torch

    import paged_kv_attention_cb_gb300 as cb

    metric = "batched KV block copy: HBM GB/s (bytes read + written); % of copy roofline"
    nb, bs, hkv, d = 3 * COPY_BLOCKS, 16, 8, 128
    block_bytes = bs * hkv * d * 2
    moved = 2 * 2 * COPY_BLOCKS * block_bytes  # K and V, read and written
    conf = {"workload": f"copy_{COPY_BLOCKS}_blocks_bf16", "blocks": COPY_BLOCKS,
            "block_size": bs, "num_kv_heads": hkv, "head_dim": d, "num_blocks": nb,
            "bytes_per_step": moved, "l2": "512 MiB read between timed steps (L2 evicted, clean)",
            "parallelism": f"replicas x{world}"}
    rng = np.random.default_rng(9)
    perm = rng.permutation(nb).astype(np.int32)
    src, dst = perm[:COPY_BLOCKS], perm[COPY_BLOCKS:2 * COPY_BLOCKS]
    if args.impl == "reference":
        if rank != 0:
            return
        import oracle

        n = 512  # bounded sample of the same copy
        hk = np.zeros((n * 3, bs, hkv, d), np.float32)
        hv = np.zeros_like(hk)
        per = []
        for _ in range(args.steps):
            t0 = time.perf_counter()
            oracle.copy_blocks(hk, hv, hk, hv, np.arange(n), np.arange(n, 2 * n))
            per.append(time.perf_counter() - t0)
        val = 2 * 2 * n * block_bytes * args.steps / sum(per) / 1e9
        line = {"impl": "reference", "metric": metric, "value": val, "unit": "GB/s",
                "n_gpus": args.gpus, "steps": args.steps, "warmup": 0,
                "ms_per_step": 1e3 * sum(per) / args.steps, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
                "config": conf,
                "cpu_baseline": {"value": val, "unit": "GB/s", "cores": 1, "kind": "oracle",
                                 "sample": f"{n} blocks per step (bf16 block bytes counted)"},
                "e2e": {"value": val, "unit": "GB/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    g = torch.Generator(device=dev)
    g.manual_seed(9)
    k = torch.randn(nb, bs, hkv, d, generator=g, device=dev).to(torch.bfloat16)
    v = torch.randn(nb, bs, hkv, d, generator=g, device=dev).to(torch.bfloat16)
    ds, dd = torch.from_numpy(src).to(dev), torch.from_numpy(dst).to(dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    flush_buf = torch.ones(FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
    for _ in range(args.warmup):
        cb.copy_blocks(k, v, k, v, ds, dd, error_word=err, stream=stream)
    torch.cuda.synchronize()
    if int(err.item()) != 0:
        raise RuntimeError("device bounds check fired")
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    launches0 = cb.launch_count()
    barrier(world)
    torch.cuda.synchronize()
    with NvmlClockSampler(local) as clocks:
        for a, b in ev:
            flush_buf.max()
            a.record(stream)
            cb.copy_blocks(k, v, k, v, ds, dd, error_word=err, stream=stream)
            b.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    launches = cb.launch_count() - launches0
    ms = reduce_max(sum(a.elapsed_time(b) for a, b in ev), world) / args.steps
    # end to end: swap-out of the same blocks = gather into staging + copy to pinned host
    stage_k = torch.empty(COPY_BLOCKS, bs, hkv, d, dtype=torch.bfloat16, device=dev)
    stage_v = torch.empty_like(stage_k)
    host_k = torch.empty(stage_k.shape, dtype=torch.bfloat16, pin_memory=True)
    host_v = torch.empty_like(host_k, pin_memory=True)
    ids = torch.arange(COPY_BLOCKS, dtype=torch.int32, device=dev)
    e2e_ms = 0.0
    for _ in range(args.steps):
        flush_buf.max()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        cb.copy_blocks(k, v, stage_k, stage_v, ds, ids, stream=stream)
        host_k.copy_(stage_k, non_blocking=True)
        host_v.copy_(stage_v, non_blocking=True)
        b.record(stream)
        torch.cuda.synchronize()
        e2e_ms += a.elapsed_time(b)
    e2e_ms = reduce_max(e2e_ms, world) / args.steps
    if rank != 0:
        return
    peak, peak_kind = peaks()
    value = world * moved / (ms * 1e-3) / 1e9
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        import oracle

        n = 512
        hk = np.zeros((n * 3, bs, hkv, d), np.float32)
        hv = np.zeros_like(hk)
        t0 = time.perf_counter()
        reps = 0
        while time.perf_counter() - t0 < min(args.cpu_budget, 5.0):
            oracle.copy_blocks(hk, hv, hk, hv, np.arange(n), np.arange(n, 2 * n))
            reps += 1
        el = time.perf_counter() - t0
        cpu = {"value": 2 * 2 * n * block_bytes * reps / el / 1e9, "unit": "GB/s", "cores": 1,
               "kind": "oracle", "sample": f"{reps} x {n} blocks (bf16 block bytes counted)"}
    swapped = 2 * COPY_BLOCKS * block_bytes
    line = {"metric": metric, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic", "config": conf,
            "e2e": {"value": world * swapped / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
                    "ms_per_step": e2e_ms, "what": "swap-out: gather + copy to pinned host, "
                    "bytes swapped out / time", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": swapped},
            "gpu_launches": launches,
            "roofline": {"kernel": "copy_blocks", "bound": "hbm", "achieved": value / world,
                         "peak": peak, "unit": "GB/s", "frac": value / world / peak,
                         "peak_source": f"{peak_kind} HBM copy bandwidth",
                         "algorithmic_bytes_per_launch": moved, "avg_launch_ms": ms,
                         "traffic": recorded_traffic("copy_blocks", conf["workload"])},
            "cpu_baseline": cpu, "clocks": clocks.summary()}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- main


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default: 1000 for the GPU arm, so that the timed "
                         "region spans several clock samples; 10 for the oracle arm)")
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default=DEFAULT_CONFIG,
                    choices=sorted(workloads.CONFIGS) + ["trace", "trace_prefill_first",
                                                         "copy_blocks"])
    ap.add_argument("--graph", action="store_true",
                    help="run the step through CUDA graphs cached per padded shape (decode)")
    ap.add_argument("--trace-steps", type=int, default=0,
                    help="--config trace: time only the first N steps of the trace (0: all)")
    ap.add_argument("--cpu-budget", type=float, default=10.0,
                    help="seconds of oracle work for the cpu_baseline figure")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--extras", dest="extras", action="store_true", default=None,
                    help="also measure the mixed step and the windowed long decode and report "
                         "them in the same line (default: on for the default workload)")
    ap.add_argument("--no-extras", dest="extras", action="store_false")
    ap.add_argument("--flush", choices=["read", "write"], default="read",
                    help="L2 eviction between timed steps: read (clean) or write (dirty) 512 MiB")
    args = ap.parse_args()
    if args.steps is None:
        args.steps = 1000 if args.impl == "ours" else 10
    if args.warmup < 3:
        args.warmup = 3
    if args.extras is None:
        args.extras = args.config == DEFAULT_CONFIG and args.impl == "ours" and not args.graph

    world, rank, local = dist_setup()
    metric = "paged-attn step: achieved KV-read HBM GB/s & query tokens/s; % of roofline"
    if args.config.startswith("trace"):
        trace_main(args, world, rank, local, metric)
        return
    if args.config == "copy_blocks":
        copy_main(args, world, rank, local)
        return
    spec = workloads.by_name(args.config)
    if args.graph and (spec.T % GRAPH_Q_INTERVAL or spec.R % GRAPH_Q_INTERVAL
                       or spec.dtype != "bf16"):
        raise SystemExit("--graph: the workload's R and T must be multiples of "
                         f"{GRAPH_Q_INTERVAL} (bf16)")
    kvb = kv_bytes(spec)
    cfg = {"workload": spec.name, "requests": spec.R, "query_tokens": spec.T,
           "num_q_heads": spec.num_q_heads, "num_kv_heads": spec.num_kv_heads,
           "head_dim": spec.head_dim, "block_size": spec.block_size,
           "num_blocks": spec.num_blocks, "sliding_window": spec.sliding_window,
           "kv_bytes_per_step": kvb,
           "l2": ("inputs larger than L2; 512 MiB read between timed steps (L2 evicted, clean)"
                  if args.flush == "read" else "flushed (512 MiB write) between timed steps"),
           "parallelism": f"replicas x{world}"}
    if args.graph:
        cfg["cuda_graphs"] = f"cached per padded shape, q_interval {GRAPH_Q_INTERVAL}"

    if args.impl == "reference":
        if rank != 0:
            return
        sample, what = oracle_sample_spec(spec, oracle_sample_size(args.config))
        h = oracle_inputs(sample)
        for _ in range(args.warmup):
            time_oracle(sample, 0.0, h, max_steps=1)
        per = []
        for _ in range(args.steps):
            n, el = time_oracle(sample, 0.0, h, max_steps=1)
            per.append(el)
        t = sum(per)
        sb = kv_bytes(sample) * args.steps
        val = sb / t / 1e9
        line = {"impl": "reference", "metric": metric, "value": val, "unit": "GB/s",
                "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": 1e3 * t / args.steps, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": cfg,
                "tokens_per_s": sample.T * args.steps / t,
                "cpu_baseline": {"value": val, "unit": "GB/s", "cores": 1, "kind": "oracle",
                                 "sample": f"{what}, one oracle step per timed step"},
                "e2e": {"value": val, "unit": "GB/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return

    res = run_ours(args, spec, world, rank, local)
    extras = {}
    if args.extras:
        for name in EXTRA_CONFIGS:
            xs = workloads.by_name(name)
            extras[name] = (xs, run_ours(args, xs, world, rank, local))
    if rank != 0:
        return
    line = workload_summary(spec, res, world)
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        sample, what = oracle_sample_spec(spec, oracle_sample_size(args.config))
        n, el = time_oracle(sample, args.cpu_budget)
        cpu = {"value": kv_bytes(sample) * n / el / 1e9, "unit": "GB/s", "cores": 1,
               "kind": "oracle", "sample": f"{what} x {n} oracle steps in {el:.1f} s",
               "all_cores": oracle_all_cores(args.config, min(args.cpu_budget, 10.0))}
    out = {"metric": metric, "value": line.pop("value"), "unit": "GB/s", "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": line.pop("ms_per_step"),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
           "dtype": "bf16" if spec.dtype == "bf16" else "f32", "data": "synthetic",
           "config": cfg}
    out.update(line)
    out["cpu_baseline"] = cpu
    if extras:
        out["extra_workloads"] = {}
        for name, (xs, xr) in extras.items():
            xl = workload_summary(xs, xr, world)
            xl["workload"] = xs.name
            out["extra_workloads"][name] = xl
            if name == "mixed" and xl.get("roofline_prefill"):
                # the tensor-core roofline of the prefill tile kernel, on the mixed step
                out["roofline_prefill"] = dict(xl["roofline_prefill"], workload=xs.name)
    if res.get("graph"):
        out["graph"] = res["graph"]
    print(json.dumps(out), flush=True)


def workload_summary(spec, res, world):
    """Throughput, end-to-end figure and rooflines of one workload's run_ours result."""
    kvb = kv_bytes(spec)
    ms = res["ms_per_step"]
    peak, peak_kind = peaks()
    pk = res["per_kernel"]
    # dominant kernel: most device time in the attribution pass
    dom = max(pk.items(), key=lambda kv: kv[1][0])[0] if pk else None
    dom_ms = pk[dom][0] / pk[dom][1] if dom else None
    if dom == "decode_split":
        dom_bytes = decode_kernel_bytes(spec)
    elif dom == "portable_attention":
        dom_bytes = kvb + 2 * spec.T * spec.num_q_heads * spec.head_dim * spec.elt_bytes()
    else:
        dom_bytes = kvb
    line = {"value": world * kvb / (ms * 1e-3) / 1e9, "ms_per_step": ms,
            "tokens_per_s": world * spec.T / (ms * 1e-3),
            "step_ms_median": statistics.median(res["step_ms"]),
            "value_after_write_flush": (world * kvb / (res["alt_ms"] * 1e-3) / 1e9
                                        if res["alt_ms"] else None)}
    e2e_ms = res["e2e_ms_per_step"]
    e2e_serial = res["e2e_serial_ms_per_step"]
    line["e2e"] = {"value": world * kvb / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
                   "ms_per_step": e2e_ms, "h2d_bytes_per_step": res["h2d"],
                   "d2h_bytes_per_step": res["d2h"], "h2d_copies_per_step": res["h2d_copies"],
                   "mode": "pipelined: step i+1's copy-in and step i-1's copy-out overlap step i",
                   "serial": {"value": world * kvb / (e2e_serial * 1e-3) / 1e9,
                              "ms_per_step": e2e_serial,
                              "mode": "copy in, step, copy out, one step at a time"}}
    line["gpu_launches"] = res["launches"]
    line["per_kernel_ms"] = {k: v[0] / v[1] for k, v in pk.items()}
    achieved = dom_bytes / (dom_ms * 1e-3) / 1e9 if dom_ms else None
    line["roofline"] = {"kernel": dom, "bound": "hbm", "achieved": achieved, "peak": peak,
                        "unit": "GB/s", "frac": (achieved / peak) if achieved else None,
                        "peak_source": f"{peak_kind} HBM copy bandwidth",
                        "algorithmic_bytes_per_launch": dom_bytes, "avg_launch_ms": dom_ms,
                        "traffic": recorded_traffic(dom, spec.name) if dom else None}
    if dom != "decode_split" and "decode_split" in pk:
        dms = pk["decode_split"][0] / pk["decode_split"][1]
        db = decode_kernel_bytes(spec)
        line["roofline_decode"] = {"kernel": "decode_split", "bound": "hbm",
                                   "achieved": db / (dms * 1e-3) / 1e9, "peak": peak,
                                   "unit": "GB/s", "frac": db / (dms * 1e-3) / 1e9 / peak,
                                   "algorithmic_bytes_per_launch": db, "avg_launch_ms": dms}
    if "prefill_tc" in pk:
        fl = prefill_flops(spec)
        pms = pk["prefill_tc"][0] / pk["prefill_tc"][1]
        tpk, tkind = bf16_peak()
        ach = fl / (pms * 1e-3) / 1e12
        line["roofline_prefill"] = {
            "kernel": "prefill_tile", "bound": "tensor", "achieved": ach, "peak": tpk,
            "unit": "TFLOP/s", "frac": ach / tpk,
            "peak_source": f"{tkind} dense bf16 (burst: the kernel is timed alone)",
            "algorithmic_flops_per_launch": fl, "avg_launch_ms": pms,
            "traffic": recorded_traffic("prefill_tc", spec.name)}
        if "decode_split" in pk:
            # the whole step's bound with the two parts one after the other at their peaks:
            # every byte at the measured HBM bandwidth plus every FLOP at the bf16 peak
            t_star = (kvb / (peak * 1e9) + fl / (tpk * 1e12)) * 1e3
            line["step_bound"] = {"t_star_ms": t_star, "step_ms": ms, "t_star_over_step": t_star / ms,
                                  "what": "algorithmic KV bytes / measured HBM + prefill FLOPs / "
                                          "measured bf16 peak (the kernels run side by side, "
                                          "so the step can beat it)"}
    line["clocks"] = res["clocks"]
    return line


if __name__ == "__main__":
    main()
