"""Benchmark of the paged-attention hot path on one GB300 (or N replicas).

A step is one pass of the decode hot path over one batch of synthetic input:
the write of each sequence's new token into the paged cache and split-KV
decode attention over the block-paged cache, in one launch
(pa_decode_append; segments split across CTAs are merged inside it).  With
``--separate-write`` the step is the two calls pa_cache_write and pa_decode.
The workload is the Qwen3-8B-shaped decode step: 32 sequences with context
lengths ~ U[512, 4096], 32 query / 8 kv heads, head_dim 128, block size 16,
bf16 KV ~ N(0, 1), random non-contiguous block tables from a pool of 1.25x
the blocks needed (seed 1002).

Printed: one JSON line.  ``value`` is the effective KV-read bandwidth, the
algorithmic KV bytes of the step (every valid K and V element of every
(sequence, kv head) once) divided by the device time of the step, with the
inputs resident in HBM.  The step's KV (304 MB) is larger than the 129 MB L2
and read in the same order every step, so no L2 flush is needed between steps
(smaller working sets are flushed between steps: a write of a buffer of twice
the L2 size, then a read of another one, so that no dirty line of the flush is
written back inside the timed region).

``--impl reference`` times the fp64 CPU oracle instead (the only reference
implementation of this method), on a bounded sample of the same workload.

For N > 1 (torchrun) every rank runs an independent replica on its own GPU
(the path needs no exchange between GPUs); value = all ranks' bytes / the
slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "paged decode attention: effective KV-read GB/s and % of GB300 HBM peak; us/step"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
WORKLOAD = 2
FP8_FORMATS = {"e4m3": "fp8_e4m3", "e5m2": "fp8_e5m2"}  # -> workloads.KV_FP8 / KV_FP8_E5M2


FALLBACK_BF16_TFLOPS = 1900.0
# the timed K-step measurement is repeated until the timed region lasts about
# this long, so that the clock sampler sees it
MIN_TIMED_S = 0.5

# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) per launch of
# each hot kernel, averaged over the launches of one ncu launch-list capture
# of this bench's own command (see the summaries in profiles/).  A figure is reported only while the kernel's
# source files hash to what they were when it was captured.
CSRC = os.path.join(ROOT, "paged_kv_attention_14_gb300", "csrc")
NCU_TRAFFIC = {
    # the decode kernel as the bench launches it, with the step's cache write
    # fused in (pa_decode_append; split segments are merged inside it):
    # dram__bytes_read.sum 305,605,120 + dram__bytes_write.sum 3,228,928
    # (the timed pa_decode launch writes no appended rows: 131 KB, 0.04%, less)
    "decode": {"workload": 2, "bytes": 308_834_048,
               "sha256": "f60f4519bc7b6121e76327083a7effb5ab28087124dca02a19359265384d06a9",
               "sources": ["pa_device.cuh", "pa_decode_kernels.cuh", "pa_decode_mma_bf16.cu", "pa_decode.cu"]},
    # the tcgen05 prefill kernel launched alone (default variant, fp16 P.V):
    # dram__bytes_read.sum 48,910,592 + dram__bytes_write.sum 1,990,400
    "prefill": {"workload": 5, "bytes": 50_900_992,
                "sha256": "3fc16caf0e868c39f32eb5ea3d348925bcbd55ad4fbd0ede2d14bd4eabdae64f",
                "sources": ["pa_device.cuh", "pa_prefill_tc.cuh", "pa_prefill_tc.cu"]},
}


def _src_sha256(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(CSRC, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def _traffic(kernel: str, workload: int, local: bool = False):
    t = NCU_TRAFFIC[kernel]
    if local or t["bytes"] is None or t["workload"] != workload or _src_sha256(t["sources"]) != t["sha256"]:
        return None
    return t["bytes"]


def _peaks():
    """(HBM GB/s, bf16 dense TFLOP/s burst, 'measured' | 'fallback')."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


def _max_over_ranks(vals, dev):
    """Element-wise maximum over the ranks of per-rank values (times: the
    slowest rank's), through the default process group."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in vals], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t]


def _job_throughput(world_size: int, units_per_rank: float, seconds: float) -> float:
    """Whole-job rate of independent replicas: all ranks' units over the
    slowest rank's time."""
    return world_size * units_per_rank / seconds


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


class ClockSampler:
    """nvidia-smi clocks and throttle reasons of one GPU, sampled while running.

    A reader thread stamps every sample with the host clock; ``stop()`` keeps
    the samples taken between ``mark_start()`` and ``mark_end()`` (the timed
    region), or all of them if that region was shorter than the sampling
    period.  The GPU is named by its UUID, which nvidia-smi and CUDA agree on
    whatever the device numbering."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    PERIOD_MS = 50

    def __init__(self, gpu_index: int, out_path: str | None = None):
        self.gpu = gpu_index
        self.proc = None
        self.out_path = out_path
        self.lines = []
        self.thread = None
        self.t0 = self.t1 = None
        self.stopping = False
        self.target = None

    def _target(self) -> str:
        """The GPU as nvidia-smi names it: its nvidia-smi index, found by
        CUDA's UUID in nvidia-smi's list; where nvidia-smi hides UUIDs, the
        only GPU it lists, else the CUDA_VISIBLE_DEVICES entry of the device.
        nvidia-smi sometimes answers "No devices were found" while NVML is
        busy, so the list is asked for a few times."""
        uuid = None
        try:
            import torch
            u = str(torch.cuda.get_device_properties(self.gpu).uuid)
            uuid = u if u.startswith("GPU-") else "GPU-" + u
        except Exception:
            pass
        listed = []
        for _ in range(10):
            try:
                r = subprocess.run(["nvidia-smi", "--query-gpu=index,uuid", "--format=csv,noheader"],
                                   capture_output=True, text=True, timeout=20)
            except (OSError, subprocess.TimeoutExpired):
                break
            listed = [[x.strip() for x in line.split(",")] for line in r.stdout.splitlines() if "," in line]
            listed = [x for x in listed if x[0].isdigit()]
            if r.returncode == 0 and listed:
                break
            time.sleep(0.2)
        for idx, u in listed:
            if uuid is not None and u == uuid:
                return idx
        if len(listed) == 1:
            return listed[0][0]
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        ids = [x.strip() for x in vis.split(",") if x.strip()]
        if len(ids) > self.gpu and ids[self.gpu].isdigit():
            return ids[self.gpu]
        return str(self.gpu)

    def _spawn(self):
        if self.target is None:
            self.target = self._target()
        return subprocess.Popen(["nvidia-smi", "-i", self.target, f"--query-gpu={self.FIELDS}",
                                 "--format=csv,noheader,nounits", "-lms", str(self.PERIOD_MS)],
                                stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)

    def _read(self):
        # nvidia-smi sometimes exits at once with "No devices were found" (NVML
        # busy); it is started again until stop() is called
        while True:
            for line in self.proc.stdout:
                self.lines.append((time.perf_counter(), line))
            self.proc.wait()
            if self.stopping:
                return
            if self.lines and "No devices were found" in self.lines[-1][1]:
                self.target = None  # named again at the next start
            time.sleep(self.PERIOD_MS / 1000)
            try:
                self.proc = self._spawn()
            except OSError:
                return

    def start(self):
        import threading
        self.stopping = False
        try:
            self.proc = self._spawn()
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.3)

    def mark_start(self):
        self.t0 = time.perf_counter()

    def mark_end(self):
        self.t1 = time.perf_counter()

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
        self.stopping = True
        for _ in range(3):  # the reader may have just started a new nvidia-smi
            p = self.proc
            p.terminate()
            try:
                p.wait(timeout=10)
            except subprocess.TimeoutExpired:
                p.kill()
            self.thread.join(timeout=1)
            if not self.thread.is_alive():
                break
        if self.out_path:
            with open(self.out_path, "w") as f:
                f.write("".join(f"{t:.4f},{line}" for t, line in self.lines))
        parsed = []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for t, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                parsed.append((t, float(parts[1]), float(parts[2]),
                               {n for n, v in zip(names, parts[5:9]) if v.lower() == "active"}))
            except ValueError:
                continue
        if not parsed:
            first = self.lines[0][1].strip() if self.lines else ""
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples" + (f": {first}" if first else "")]}
        inside = [p for p in parsed if self.t0 is not None and self.t1 is not None and self.t0 <= p[0] <= self.t1]
        use = inside or parsed
        return {"sm_mhz": statistics.median(p[1] for p in use), "sm_max_mhz": max(p[2] for p in use),
                "reasons": sorted(set().union(*(p[3] for p in use))), "samples": len(use),
                "samples_in_timed_region": len(inside)}


def _first_key(pos: int, window: int, chunk: int) -> int:
    """First key a query at ``pos`` sees: sliding window of ``window`` keys,
    chunked-local attention with chunks of ``chunk`` positions (0: off)."""
    lo = 0
    if window:
        lo = max(lo, pos - window + 1)
    if chunk:
        lo = max(lo, (pos // chunk) * chunk)
    return lo


def _local_config(args) -> dict:
    """Non-default settings of the run (fp16 cache, local attention), for the
    JSON line's config (none when off)."""
    d = {}
    if args.fp16:
        d["kv_cache"] = "fp16"
    if args.fp8_cache:
        d["kv_cache"] = args.fp8_format
    if args.per_head_scales:
        d["fp8_scales"] = "per kv head"
    if args.workload == 5:
        d["mixed_step"] = {"fused": ("cache write, then decode and prefill in one persistent launch" if args.separate_write
                                     else "cache write, decode and prefill in one persistent launch"),
                           "streams": "cache write, then the decode on a second stream beside the prefill",
                           "serial": "cache write, decode, prefill in order on one stream"}[args.mixed_mode]
    if args.prefill_impl:
        d["prefill_impl"] = {1: "mma.sync", 2: "tcgen05, fp16 P.V", 3: "tcgen05, P as a hi + lo pair"}[args.prefill_impl]
    if args.sliding_window:
        d["sliding_window"] = args.sliding_window
    if args.attention_chunk:
        d["attention_chunk"] = args.attention_chunk
    return d


class _L2Flush:
    """Evicts the L2 between timed steps: a write of one buffer of ``nbytes``
    and a read (a sum) of another."""

    def __init__(self, nbytes: int, dev):
        import torch
        self.w = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        self.r = torch.zeros(nbytes // 8, dtype=torch.int64, device=dev)
        self.acc = torch.zeros((), dtype=torch.int64, device=dev)

    def __call__(self):
        import torch
        self.w.zero_()
        torch.sum(self.r, dim=0, out=self.acc)


def _decode_kv_bytes(b, window: int, chunk: int) -> int:
    """Algorithmic KV bytes of the decode part: every K and V element the
    queries may see, of every (sequence, kv head), read once."""
    lens = b.context_lens_decode.cpu().tolist()
    tokens = sum(L - _first_key(L - 1, window, chunk) for L in lens if L > 0)
    return tokens * b.num_kv_heads * b.head_dim * 2 * b.kv_elem_bytes


def _prefill_flops(b, window: int = 0, chunk: int = 0) -> int:
    """Algorithmic flops of the causal prefill chunks: per query row and head,
    4 * head_dim flops (QK^T and PV multiply-adds) per key it may see (at or
    before it, and within its window / chunk)."""
    qsl = b.query_start_loc.cpu().tolist()
    lens = b.context_lens_prefill.cpu().tolist()
    keys = 0
    for s, L in enumerate(lens):
        n = qsl[s + 1] - qsl[s]
        if not window and not chunk:
            # query i sits at L - n + i and sees L - n + i + 1 keys
            keys += n * (L - n) + n * (n + 1) // 2
        else:
            keys += sum(p + 1 - _first_key(p, window, chunk) for p in range(L - n, L))
    return keys * 4 * b.head_dim * b.num_q_heads


def run_ours(args):
    import torch
    import torch.distributed as dist

    from paged_kv_attention_14_gb300 import build as pa_build
    from paged_kv_attention_14_gb300 import binding as B
    from paged_kv_attention_14_gb300 import workloads as W
    from paged_kv_attention_14_gb300.step import GraphedStep, MixedStep

    ws, rank, local = _dist()
    if ws > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    B.load(pa_build.build())

    b = W.workload(args.workload, device=dev, poison=False, fp8_format=FP8_FORMATS[args.fp8_format],
                   fp16=args.fp16, per_head_scales=args.per_head_scales, fp8_cache=args.fp8_cache)
    kv = {W.KV_BF16: B.PA_KV_BF16, W.KV_F16: B.PA_KV_F16, W.KV_FP8: B.PA_KV_FP8_E4M3,
          W.KV_FP8_E5M2: B.PA_KV_FP8_E5M2}[b.kv_dtype]
    kv8 = kv in (B.PA_KV_FP8_E4M3, B.PA_KV_FP8_E5M2)
    desc = B.make_desc(b.num_blocks, b.num_kv_heads, b.num_q_heads, b.head_dim, kv,
                       b.k_scale if kv8 else 0.0, b.v_scale if kv8 else 0.0, decode_impl=args.decode_impl,
                       prefill_impl=args.prefill_impl,
                       sliding_window=args.sliding_window, attention_chunk=args.attention_chunk,
                       k_scales=b.k_scales, v_scales=b.v_scales)
    if not kv8:
        kc, vc = b.k_pool, b.v_pool
    else:
        kc = torch.empty(tuple(b.k_pool.shape), dtype=torch.uint8, device=dev)
        vc = torch.empty_like(kc)
        k_rows, v_rows, slots = b.pool_tokens_as_rows()
        B.pa_cache_write(desc, k_rows, v_rows, kc, vc, slots)
        del k_rows, v_rows, slots
        b.k_pool = b.v_pool = None
    S = b.context_lens_decode.shape[0]
    maxL = b.max_context_len_decode()
    # the single-launch mixed step's workspace (it also serves pa_decode)
    wsp = B.mixed_workspace(desc, S, maxL, dev)
    out = torch.empty(S, b.num_q_heads, b.head_dim, device=dev)
    kv_bytes = _decode_kv_bytes(b, args.sliding_window, args.attention_chunk)
    # the captured traffic figures are for the default settings only
    local = bool(args.sliding_window or args.attention_chunk or args.fp16 or args.per_head_scales or args.prefill_impl
                 or args.fp8_cache)
    mixed = b.q_prefill is not None
    if mixed:
        pf_out = torch.empty(b.q_prefill.shape, dtype=torch.float32, device=dev)
        qsl = b.query_start_loc
        pf_maxq = int((qsl[1:] - qsl[:-1]).max())
        pf_maxL = int(b.context_lens_prefill.max())
        pf_flops = _prefill_flops(b, args.sliding_window, args.attention_chunk)
    # cache write + decode (+ prefill)
    # cache write + decode (+ prefill); a fused mixed step launches one
    # kernel for decode and prefill together
    launches_per_step = 2 + (1 if mixed else 0)
    l2_bytes = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = None
    if kv_bytes < 2 * l2_bytes:
        # small working set: flush L2 by writing a buffer larger than it, then
        # reading another one, which evicts the written (dirty) lines before
        # the timed kernels start instead of during them
        flush = _L2Flush(2 * l2_bytes, dev)

    # mixed step: decode and prefill in one persistent launch, the cache
    # write inside it (--mixed-mode fused), the decode on a second stream
    # beside the prefill (streams) or one after the other (serial), these
    # two after a cache write of their own
    pf_ws = None
    if mixed and args.prefill_entry == "balanced":
        pf_ws = B.prefill_workspace(desc, int(b.context_lens_prefill.shape[0]), pf_maxq, dev)
    pf_entry = "pa_prefill_chunk_balanced" if pf_ws is not None else "pa_prefill_chunk"
    # a decode-only step whose new rows are one token per sequence (every
    # decode workload) appends them in the decode launch (pa_decode_append)
    # where the library takes it, unless --separate-write
    append = not mixed and not args.separate_write
    # a mixed step's fused mode writes the step's rows in its launch too
    # (pa_mixed_attention_append; the workload's chunks start at block
    # boundaries), unless --separate-write
    ms = MixedStep(desc, kc, vc, b.scale, decode_out=out, workspace=wsp, max_context_len_decode=maxL,
                   prefill_out=pf_out if mixed else None, max_q_len=pf_maxq if mixed else 0,
                   max_context_len_prefill=pf_maxL if mixed else 0, mode=args.mixed_mode,
                   prefill_workspace=pf_ws, decode_append=append,
                   write_in_step=mixed and not args.separate_write)
    decode, prefill, attend = ms.decode, ms.prefill, ms.attend
    if ms.mode == "fused":
        launches_per_step = 2
    args.mixed_mode = ms.mode  # the mode that runs (fused falls back to streams where it does not apply)

    def step():
        ms(b.k_new, b.v_new, b.slot_mapping, (b.q_decode, b.block_tables_decode, b.context_lens_decode),
           (b.q_prefill, b.query_start_loc, b.block_tables_prefill, b.context_lens_prefill) if mixed else None)

    for _ in range(args.warmup):
        if flush is not None:
            flush()
        step()
    torch.cuda.synchronize()
    fused_write = (mixed and ms.write_in_step and ms.mode == "fused" and
                   not ms.prefill_balanced((b.q_prefill, b.query_start_loc, b.block_tables_prefill,
                                            b.context_lens_prefill)))
    if ms.decode_append or fused_write:
        launches_per_step = 1  # the write and the attention in one launch
    step_how = ("pa_decode_append (the step's cache write and decode in one launch)" if ms.decode_append else
                "pa_mixed_attention_append (the step's cache write, decode and prefill in one launch)" if fused_write
                else "pa_cache_write, then " + ("pa_mixed_attention" if ms.mode == "fused" and mixed else
                                                "pa_decode" + (" and the prefill" if mixed else "")))

    K = args.steps
    # A repeat times exactly K steps.  The K-step measurement is repeated
    # until the timed region lasts about MIN_TIMED_S, so that nvidia-smi
    # clock samples fall inside it; the reported time per step is the
    # median repeat's.
    t_est = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_est[0].record()
    for _ in range(3):
        if flush is not None:
            flush()
        step()
    t_est[1].record()
    torch.cuda.synchronize()
    est_s = max(t_est[0].elapsed_time(t_est[1]) * 1e-3 / 3, 1e-6)
    R = max(1, min(2000, int(math.ceil(MIN_TIMED_S / (K * est_s)))))
    K2 = max(10, K // 2)
    R2 = max(1, min(2000, int(math.ceil(MIN_TIMED_S / 2 / (K2 * est_s)))))
    if args.repeats:  # a fixed count (profiling runs, where launches are slow)
        R = R2 = args.repeats
    # the raw nvidia-smi samples go to the file PA_BENCH_CLOCKS_CSV names, if any
    sampler = ClockSampler(local, os.environ.get("PA_BENCH_CLOCKS_CSV") or None)
    sampler.start()
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sampler.mark_start()
    # timed region 1: whole steps, CUDA events only at step boundaries (an
    # event between two kernels would cut the programmatic-dependent overlap
    # of the decode launch with the cache write); with an L2 flush between
    # steps, events around each step leave the flush out
    # Without a flush (inputs larger than L2) one event pair brackets the K
    # back-to-back steps of a repeat; with one, events bracket each step so
    # that the flush stays outside the timed region.  (An event pair alone
    # measures a few microseconds on these boxes: per-step events would add
    # that to every step.)
    def ev_pair():
        return torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    rep_ms = []
    for _ in range(R):
        if flush is None:
            ev = [ev_pair()]
            ev[0][0].record()
            for i in range(K):
                step()
            ev[0][1].record()
        else:
            ev = [ev_pair() for _ in range(K)]
            for i in range(K):
                flush()
                ev[i][0].record()
                step()
                ev[i][1].record()
        rep_ms.append(ev)
    # timed region 2: the kernels of each entry point alone (decode; prefill),
    # K2 back-to-back calls under one event pair, or events around each call
    # after a flush
    rep_d, rep_p = [], []
    for _ in range(R2):
        if flush is None:
            ev_d, ev_p = [ev_pair()], [ev_pair()]
            ev_d[0][0].record()
            for i in range(K2):
                decode(b.q_decode, b.block_tables_decode, b.context_lens_decode)
            ev_d[0][1].record()
            if mixed:
                ev_p[0][0].record()
                for i in range(K2):
                    prefill(b.q_prefill, b.query_start_loc, b.block_tables_prefill, b.context_lens_prefill)
                ev_p[0][1].record()
        else:
            ev_d = [ev_pair() for _ in range(K2)]
            ev_p = [ev_pair() for _ in range(K2)]
            for i in range(K2):
                flush()
                ev_d[i][0].record()
                decode(b.q_decode, b.block_tables_decode, b.context_lens_decode)
                ev_d[i][1].record()
                if mixed:
                    ev_p[i][0].record()
                    prefill(b.q_prefill, b.query_start_loc, b.block_tables_prefill, b.context_lens_prefill)
                    ev_p[i][1].record()
        rep_d.append(ev_d)
        rep_p.append(ev_p)
    torch.cuda.synchronize()
    sampler.mark_end()
    if ws > 1:
        dist.barrier()
    clocks = sampler.stop()

    def per_step(reps, n):
        return statistics.median(sum(a.elapsed_time(c) for a, c in ev) / n for ev in reps)

    step_ms = per_step(rep_ms, K)
    dec_ms = per_step(rep_d, K2)
    pf_ms = per_step(rep_p, K2) if mixed else 0.0
    if ws > 1:
        step_ms, dec_ms, pf_ms = _max_over_ranks([step_ms, dec_ms, pf_ms], dev)
    assert int(wsp[:4].view(torch.int32)[0]) == 0, "decode kernel reported a wait timeout"

    # End to end through the public API: every step copies its inputs from one
    # pinned host buffer into one device buffer (one H2D copy; the tensors the
    # library gets are views into it) and reads the step's result back.
    names = ["q_decode", "k_new", "v_new", "slot_mapping", "block_tables_decode", "context_lens_decode"]
    if mixed:
        names += ["q_prefill", "query_start_loc", "block_tables_prefill", "context_lens_prefill"]
    srcs = [getattr(b, n).contiguous() for n in names]
    offs, total = [], 0
    for t in srcs:
        offs.append(total)
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    host_buf = torch.empty(total, dtype=torch.uint8).pin_memory()
    dev_buf = torch.empty(total, dtype=torch.uint8, device=dev)
    views = {}
    for n, t, o in zip(names, srcs, offs):
        nb = t.numel() * t.element_size()
        host_buf[o:o + nb].copy_(t.reshape(-1).view(torch.uint8).cpu())
        views[n] = dev_buf[o:o + nb].view(t.dtype).view(t.shape)
    out_host = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    pf_host = torch.empty(pf_out.shape, dtype=pf_out.dtype).pin_memory() if mixed else None
    h2d = total
    d2h = out_host.numel() * out_host.element_size() + (pf_host.numel() * pf_host.element_size() if mixed else 0)
    # a decode-only step's kernel stores its output straight into the pinned
    # host buffer (the decode entry points take host-resident out / lse), so
    # the result reaches the host without a copy after the kernel;
    # --e2e-out device keeps the output on the device and copies it back
    out_to_host = not mixed and args.e2e_out == "host"
    ms_e2e = ms
    if out_to_host:
        ms_e2e = MixedStep(desc, kc, vc, b.scale, decode_out=out_host, workspace=wsp, max_context_len_decode=maxL,
                           mode=args.mixed_mode, decode_append=append)

    def e2e_issue():
        dev_buf.copy_(host_buf, non_blocking=True)
        ms_e2e(views["k_new"], views["v_new"], views["slot_mapping"],
               (views["q_decode"], views["block_tables_decode"], views["context_lens_decode"]),
               (views["q_prefill"], views["query_start_loc"], views["block_tables_prefill"],
                views["context_lens_prefill"]) if mixed else None)
        if mixed:
            pf_host.copy_(pf_out, non_blocking=True)
        if not out_to_host:
            out_host.copy_(out, non_blocking=True)

    # the public API's step as a user drives it: one CUDA-graph replay of the
    # copies in, the step and the copies out, then a wait for the result
    graphed = GraphedStep(e2e_issue)

    def e2e_step():
        graphed()

    for _ in range(max(3, args.warmup)):
        if flush is not None:
            flush()
        e2e_step()
    ke = max(10, min(K, 200))
    tot = 0.0
    for _ in range(ke):
        if flush is not None:
            flush()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        e2e_step()
        tot += time.perf_counter() - t0
    e2e_s = tot / ke
    if ws > 1:
        (e2e_s,) = _max_over_ranks([e2e_s], dev)
    if out_to_host:
        # the same step with the same inputs: the result in host memory equals
        # the device-resident one bit for bit
        assert torch.equal(out_host, out.cpu()), "the output stored into host memory differs"

    if rank == 0:
        peak, tc_peak, peak_kind = _peaks()
        gbs = _job_throughput(ws, kv_bytes, step_ms * 1e-3) / 1e9
        dec_gbs = kv_bytes / (dec_ms * 1e-3) / 1e9
        alone_how = ("timed alone: back-to-back calls under one event pair" if flush is None
                     else "timed alone: events around each call after an L2 flush")
        line = {
            "metric": METRIC,
            "value": round(gbs, 1),
            "unit": "GB/s",
            "n_gpus": ws,
            "steps": K,
            "warmup": args.warmup,
            "ms_per_step": round(step_ms, 5),
            "us_per_step": round(step_ms * 1e3, 2),
            "pct_hbm_peak": {f"of {peak_kind} {peak:.1f} GB/s": round(100 * gbs / ws / peak, 1),
                             f"of nominal {NOMINAL_HBM_GBS:.0f} GB/s": round(100 * gbs / ws / NOMINAL_HBM_GBS, 1)},
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": b.kv_dtype,
            "data": "synthetic",
            "config": {"workload": b.name, "num_seqs": S, "kv_tokens": int(b.context_lens_decode.sum()),
                       "kv_bytes_per_step": kv_bytes,
                       "l2": ("flushed before every step (write of 2x L2, then read of 2x L2)" if flush is not None else
                              f"inputs larger than L2 ({kv_bytes >> 20} MiB KV vs {l2_bytes >> 20} MiB L2), no flush"),
                       "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU", **_local_config(args)},
            "roofline": {"bound": "hbm",
                         "kernel": "pa_decode (one decode kernel launch), " + alone_how,
                         "achieved": round(dec_gbs, 1), "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                         "frac": round(dec_gbs / peak, 4), "kernel_us": round(dec_ms * 1e3, 2),
                         "traffic": _traffic("decode", args.workload, local)},
            "e2e": {"value": round(_job_throughput(ws, kv_bytes, e2e_s) / 1e9, 1), "unit": "GB/s", "us_per_step": round(e2e_s * 1e6, 1),
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "how": "step.GraphedStep: one CUDA-graph replay per step of the pinned-host-to-device copy of the "
                           "inputs, the cache write and attention, and " +
                           ("the kernel's stores of the output straight into pinned host memory" if out_to_host else
                            "the copy of the outputs to pinned host memory") + ", then a wait; host wall clock"},
            # timed region 2 calls each entry point alone: decode (and prefill)
            "step_calls": step_how,
            "gpu_launches": launches_per_step * K * R + (2 if mixed else 1) * K2 * R2,
            "timed_repeats": {"steps": R, "kernels_alone": R2,
                              "note": f"each repeat times exactly {K} steps ({K2} calls of each entry point alone); "
                                      "ms_per_step is the median repeat",
                              "events": ("one event pair around the repeat's back-to-back steps (calls)"
                                         if flush is None else "an event pair around each step (call), "
                                         "after its L2 flush")},
            "clocks": clocks,
        }
        if clocks.get("sm_mhz"):
            line["cycles_per_step"] = round(step_ms * 1e-3 * clocks["sm_mhz"] * 1e6)
        if mixed:
            pf_tf = pf_flops / (pf_ms * 1e-3) / 1e12
            line["prefill"] = {"kernel": pf_entry, "us": round(pf_ms * 1e3, 2), "flops": pf_flops,
                               "tflops": round(pf_tf, 1)}
            if pf_ms > dec_ms:
                # the prefill dominates the step: the roofline is its tensor-core bound
                # (algorithmic flops; the bf16 hi/lo split of P adds half again to PV)
                line["roofline_decode"] = line["roofline"]
                line["roofline"] = {"bound": "tensor", "kernel": pf_entry + ", " + alone_how,
                                    "achieved": round(pf_tf, 1), "peak": tc_peak,
                                    "peak_kind": f"{peak_kind} bf16 dense (burst)", "unit": "TFLOP/s",
                                    "frac": round(pf_tf / tc_peak, 4), "kernel_us": round(pf_ms * 1e3, 2),
                                    "traffic": _traffic("prefill", args.workload, local or pf_ws is not None)}
        if not args.no_cpu_baseline:
            if b.kv_dtype in (W.KV_BF16, W.KV_F16):
                line["cpu_baseline"] = cpu_baseline(args.workload, budget_s=args.cpu_budget,
                                                    window=args.sliding_window, chunk=args.attention_chunk,
                                                    fp16=args.fp16)
            else:
                # the oracle's 8-bit encoder (a search over every code) would
                # need minutes to encode this pool before the first timed call
                line["cpu_baseline"] = {"value": None, "unit": "GB/s", "kind": "oracle",
                                        "unavailable": "timed on the 16-bit workloads only"}
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()


def _oracle_sample(n_workload: int, budget_s: float, window: int = 0, chunk: int = 0, fp16: bool = False):
    """Run the fp64 oracle over whole sequences of the workload (all heads)
    until ``budget_s`` of CPU time is used; returns (kv_bytes, seconds, n_seqs)."""
    import oracle
    from paged_kv_attention_14_gb300 import workloads as W

    b = W.workload(n_workload, device="cpu", poison=False, fp16=fp16)
    if b.kv_dtype not in (W.KV_BF16, W.KV_F16):
        raise RuntimeError("the CPU baseline covers the 16-bit workloads")
    code = oracle.KV_F16 if fp16 else oracle.KV_BF16
    kc, vc = b.k_pool, b.v_pool
    S = b.context_lens_decode.shape[0]
    done_bytes, t_used, n = 0, 0.0, 0
    order = list(range(S))
    while t_used < budget_s and n < 10 * S:
        s = order[n % S]
        pairs = [(s, h) for h in range(b.num_q_heads)]
        t0 = time.perf_counter()
        oracle.decode(code, 16, b.num_kv_heads, b.num_q_heads, b.head_dim, b.q_decode, kc, vc,
                      b.block_tables_decode, b.context_lens_decode, b.scale, pairs=pairs, window=window, chunk=chunk)
        t_used += time.perf_counter() - t0
        L = int(b.context_lens_decode[s])
        done_bytes += (L - _first_key(L - 1, window, chunk)) * b.num_kv_heads * b.head_dim * 2 * 2
        n += 1
    return done_bytes, t_used, n, b.name


def _oracle_worker(rank, nproc, n_workload, phases, barrier, results, window=0, chunk=0, fp16=False):
    """One process of the all-cores oracle run: builds the (seeded) workload,
    then for each phase of ``phases`` seconds runs the oracle over (sequence,
    kv head) units rank, rank + nproc, ... (the g query heads of one kv head,
    which read that head's K and V once: its algorithmic bytes) and reports
    (bytes, seconds, units)."""
    import torch

    torch.set_num_threads(1)
    import oracle
    from paged_kv_attention_14_gb300 import workloads as W

    b = W.workload(n_workload, device="cpu", poison=False, fp16=fp16)
    code = oracle.KV_F16 if fp16 else oracle.KV_BF16
    S, Hkv = b.context_lens_decode.shape[0], b.num_kv_heads
    g = b.num_q_heads // Hkv
    u = rank % (S * Hkv)
    for phase_s in phases:
        barrier.wait()
        t0 = time.perf_counter()
        done, n = 0, 0
        while time.perf_counter() - t0 < phase_s:
            s, kvh = divmod(u, Hkv)
            pairs = [(s, kvh * g + i) for i in range(g)]
            oracle.decode(code, 16, Hkv, b.num_q_heads, b.head_dim, b.q_decode, b.k_pool, b.v_pool,
                          b.block_tables_decode, b.context_lens_decode, b.scale, pairs=pairs, window=window,
                          chunk=chunk)
            L = int(b.context_lens_decode[s])
            done += (L - _first_key(L - 1, window, chunk)) * b.head_dim * 2 * 2
            n += 1
            u = (u + nproc) % (S * Hkv)
        results.put((rank, done, time.perf_counter() - t0, n))


def _oracle_all_cores(n_workload: int, phases, nproc: int | None = None, window: int = 0, chunk: int = 0,
                      fp16: bool = False):
    """The oracle on every host core: ``nproc`` spawned processes (the GPU is
    already in use in this process, so no fork), one thread each.  Returns per
    phase (kv_bytes, wall seconds, sequences), the workload name and nproc."""
    import multiprocessing as mp

    nproc = nproc or len(os.sched_getaffinity(0))
    ctx = mp.get_context("spawn")
    barrier = ctx.Barrier(nproc)
    results = ctx.Queue()
    procs = [ctx.Process(target=_oracle_worker, args=(r, nproc, n_workload, list(phases), barrier, results, window, chunk, fp16))
             for r in range(nproc)]
    for p in procs:
        p.start()
    out = []
    for _ in phases:
        got = [results.get(timeout=600) for _ in range(nproc)]
        out.append((sum(g[1] for g in got), max(g[2] for g in got), sum(g[3] for g in got)))
    for p in procs:
        p.join(timeout=60)
    return out, nproc


def cpu_baseline(n_workload: int, budget_s: float = 10.0, window: int = 0, chunk: int = 0, fp16: bool = False):
    """The oracle on all host cores for about ``budget_s`` seconds (the
    reported baseline), plus one thread for ``budget_s / 2``."""
    nbytes1, secs1, n1, name = _oracle_sample(n_workload, budget_s / 2, window, chunk, fp16)
    (res,), nproc = _oracle_all_cores(n_workload, [budget_s], window=window, chunk=chunk, fp16=fp16)
    nbytes, secs, n = res
    return {"value": round(nbytes / secs / 1e9, 4), "unit": "GB/s", "cores": nproc, "kind": "oracle",
            "sample": f"{n} (sequence, kv head) units (their g query heads each) of '{name}', fp64 C oracle, "
                      f"{nproc} processes x 1 thread, {secs:.1f} s wall",
            "single_thread": {"value": round(nbytes1 / secs1 / 1e9, 4), "unit": "GB/s", "cores": 1,
                              "sample": f"{n1} whole sequences, {secs1:.1f} s"}}


def run_reference(args):
    ws, rank, local = _dist()
    if rank != 0:
        return
    import oracle  # noqa: F401  (built on first use)
    from paged_kv_attention_14_gb300 import workloads as W

    if args.workload == 4:
        print(json.dumps({"impl": "reference", "unavailable": "the oracle arm samples the 16-bit workloads; "
                          "encoding workload 4's 8-bit pool with the oracle takes minutes"}), flush=True)
        return
    # each step: one bounded sample of the workload through the oracle on all
    # host cores, sized so that the whole run takes about two minutes
    per_step = max(0.01, min(5.0, 120.0 / max(1, args.steps + args.warmup)))
    phases, nproc = _oracle_all_cores(args.workload, [per_step] * (args.warmup + args.steps),
                                      window=args.sliding_window, chunk=args.attention_chunk, fp16=args.fp16)
    timed = phases[args.warmup:]
    nbytes = sum(p[0] for p in timed)
    secs = sum(p[1] for p in timed)
    value = nbytes / secs / 1e9
    name = W.WORKLOAD_NAMES[args.workload] + (" (fp16 variant)" if args.fp16 else "")
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * secs / args.steps, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": name, **_local_config(args)},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": nproc, "kind": "oracle",
                             "sample": f"(sequence, kv head) units of '{name}' per step on {nproc} processes x 1 "
                                       f"thread, about {per_step:.3f} s each"},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", type=int, default=WORKLOAD, choices=[1, 2, 3, 4, 5])
    ap.add_argument("--decode-impl", type=int, default=0, help="0 auto, 1 CUDA-core, 2 tensor-core")
    ap.add_argument("--prefill-impl", type=int, default=0,
                    help="0 auto, 1 mma.sync, 2 tcgen05 (fp16 P.V), 3 tcgen05 (P as a hi + lo pair)")
    ap.add_argument("--fp8-format", choices=sorted(FP8_FORMATS), default="e4m3",
                    help="8-bit cache format of workload 4 (same shapes)")
    ap.add_argument("--prefill-entry", choices=["chunk", "balanced"], default="chunk",
                    help="prefill entry point: pa_prefill_chunk (a CTA per query tile and kv head) or "
                         "pa_prefill_chunk_balanced (the library's choice of that grid or the balanced kernel)")
    ap.add_argument("--e2e-out", choices=("host", "device"), default="host",
                    help="decode-only workloads' e2e step: the kernel stores the output into pinned host memory "
                         "(host) or on the device, copied back after the kernel (device)")
    ap.add_argument("--separate-write", action="store_true",
                    help="pa_cache_write as its own launch: then pa_decode instead of pa_decode_append, or "
                         "pa_mixed_attention instead of pa_mixed_attention_append")
    ap.add_argument("--mixed-mode", choices=["fused", "streams", "serial"], default="fused",
                    help="mixed step (workload 5): one persistent launch, two streams, or one after the other")
    ap.add_argument("--per-head-scales", action="store_true",
                    help="workload 4 with one FP8 scale per kv head (heads of different magnitudes)")
    ap.add_argument("--fp8-cache", action="store_true",
                    help="workload 5 with an 8-bit cache (format --fp8-format; the same draws quantised)")
    ap.add_argument("--fp16", action="store_true",
                    help="fp16 variant of a bf16 workload (fp16 cache, q and new rows)")
    ap.add_argument("--sliding-window", type=int, default=0, help="sliding-window attention of W keys (0: off)")
    ap.add_argument("--attention-chunk", type=int, default=0, help="chunked-local attention over chunks of C (0: off)")
    ap.add_argument("--cpu-budget", type=float, default=10.0, help="seconds of oracle time for cpu_baseline")
    ap.add_argument("--repeats", type=int, default=0,
                    help="repeats of the timed K steps (0: as many as fill about half a second)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.fp16 and args.workload == 4:
        ap.error("--fp16 applies to the bf16 workloads (1, 2, 3, 5)")
    if args.per_head_scales and args.workload != 4:
        ap.error("--per-head-scales applies to the FP8 workload (4)")
    if args.fp8_cache and (args.workload != 5 or args.fp16):
        ap.error("--fp8-cache applies to workload 5")
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
