"""Decode-attention benchmark: µs per decode step, KV-read GB/s and the HBM
roofline fraction on the 100K-token long-context batch.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--partition-size P]

Prints ONE JSON line.  The default workload is the long-context decode step
(1 sequence x 100000 tokens, 24 query / 4 KV heads, head_dim 256, bf16 KV
cache, 16-token blocks, PARTITION_SIZE 512).  A step is one full pa_decode
call (V2: one launch, or the partition kernel and the log-sum-exp reduce)
over inputs already resident in HBM.  The KV cache (409.6 MB) is larger than
the 129 MB L2, so the timed steps run back to back, as a decode loop runs
them; each step is also timed alone after a 256 MiB read sweep that evicts
L2 (reads, so that no dirty lines are left to be written back while the
step runs).  Workloads whose inputs fit in L2 get that sweep before every
timed step.

`--impl reference` times the float64 CPU oracle on the host cores instead
(the reference arm): each step is the whole batch when the run fits its
budget (--ref-budget-s), else an even spread of rows scaled to a full step.

Multi-GPU (`torchrun --nproc-per-node N bench.py --gpus N`): every rank runs
its own replica of the batch on its own GPU (the decode step has no
cross-GPU exchange), timing is max over ranks, and kv_read_gbs is the sum of
all ranks' bytes over that time.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import glob
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import paged_attention_decode_v2_gb300 as pa  # noqa: E402
from paged_attention_decode_v2_gb300 import workloads as wl  # noqa: E402

METRIC = "decode-attention µs/step and KV-read GB/s (% of HBM peak) at 100K context"
UNIT = "us/step"
FALLBACK_HBM_GBS = 6800.0
L2_FLUSH_BYTES = 256 << 20
L2_BYTES = 129 << 20

# DRAM bytes (read + write) per launch of the dominant kernel, from one ncu
# capture, keyed by a hash of the code (comments and layout left out) of the
# sources that kernel is built from.  A change to any of them makes the
# figure stale, and the bench then reports null.
KERNEL_SOURCES = {
    "pa_tc_kernel": ("pa_tc.cuh", "pa_tc_host.cu", "pa_tc_bf16.cu", "pa_sm100.cuh",
                     "pa_device.cuh", "pa_internal.h", "pa_grid_reduce.cuh"),
    "pa_generic_kernel": ("pa_generic.cuh", "pa_generic_bf16.cu", "pa_generic_f32.cu",
                          "pa_device.cuh", "pa_internal.h"),
    "pa_prefill_kernel": ("pa_prefill.cuh", "pa_prefill_host.cu", "pa_prefill_bf16.cu",
                          "pa_sm100.cuh", "pa_device.cuh", "pa_internal.h"),
    "pa_sx_kernel": ("pa_sx.cuh", "pa_tc_host.cu", "pa_sx_bf16.cu", "pa_sm100.cuh",
                     "pa_device.cuh", "pa_internal.h", "pa_grid_reduce.cuh"),
}
NCU_TRAFFIC = {
    # (kernel, source hash, workload, partition size, path): bytes per launch
    # the one-launch V2 kernel (pass 1 and the in-grid reduce)
    ("pa_tc_kernel", "c6cec55e5b4e9c57", "long_100k", 512, "v2"): 409_757_440 + 3_322_880,
    # the split-x kernel in one launch (its own pass 1 and the same in-grid reduce)
    ("pa_sx_kernel", "b9d31cdbf8604998", "long_100k", 512, "v2"): 409_761_280 + 4_934_400,
    ("pa_prefill_kernel", "fb27f3351a287baf", "prefill_32k", 0, "prefill"):
        1_358_718_464 + 194_669_824,
}


def _code_only(text: str) -> str:
    """C / C++ source without its comments and with whitespace runs folded
    to one space (string literals kept as they are), so that an edit of a
    comment or of the layout does not count as a change of the kernel."""
    out, i, n = [], 0, len(text)
    while i < n:
        ch = text[i]
        if ch == '"':  # string literal, escapes included
            j = i + 1
            while j < n and text[j] != '"':
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(ch)
            i += 1
    return " ".join("".join(out).split())


def kernel_source_hash(kernel: str) -> str:
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "paged_attention_decode_v2_gb300", "csrc", name),
                  encoding="utf-8") as fh:
            h.update(name.encode())
            h.update(_code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str, workload: str, P: int, path: str):
    if kernel not in KERNEL_SOURCES:
        return None
    return NCU_TRAFFIC.get((kernel, kernel_source_hash(kernel), workload, P, path))


def max_over_ranks(values, world, device=None):
    """Element-wise max of `values` over all ranks (identity when world == 1).
    The tensor lives on `device` for NCCL and on the CPU for gloo."""
    if world <= 1:
        return list(values)
    dist = torch.distributed
    on_cpu = dist.get_backend() == "gloo" or device is None
    t = torch.tensor(values, dtype=torch.float64, device="cpu" if on_cpu else device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def measured_hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.marks = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.gpu), "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, name):
        self.marks.append((name, time.time()))

    def wait_first(self, timeout=5.0):
        """Wait (bounded) until nvidia-smi has printed its first sample, so
        the GPU loops that follow are covered from their start."""
        t0 = time.time()
        while self.proc and not self.lines and time.time() - t0 < timeout:
            time.sleep(0.01)

    def count(self, t0, t1):
        return sum(1 for ts, _ in self.lines if t0 <= ts <= t1)

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ts, line in self.lines:
            if not (t0 <= ts <= t1):
                continue
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def hold_until_sampled(sampler, t0, step_fn, device, min_samples=5, max_s=3.0):
    """Repeat ``step_fn`` (untimed) until the clock sampler holds at least
    ``min_samples`` samples since ``t0`` or ``max_s`` seconds have passed, so
    the clock record covers the GPU under this load even when the timed
    loops last only milliseconds.  Returns the number of extra steps run."""
    if sampler.proc is None:
        return 0
    n, t_hold = 0, time.time()
    while sampler.count(t0, time.time()) < min_samples and time.time() - t_hold < max_s:
        for _ in range(20):
            step_fn()
        torch.cuda.synchronize(device)
        n += 20
    return n


def gpu_id_for_smi(device) -> str:
    """nvidia-smi's id for this device (its UUID when torch knows it)."""
    try:
        u = str(torch.cuda.get_device_properties(device).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return str(device.index or 0)


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def run_ours(args, rank, world, device):
    w = wl.WORKLOADS[args.workload]
    P = args.partition_size or w.partition_sizes[0]
    batch = wl.make(w, device=device)
    sx = {}
    if args.split_x:
        # the caches rewritten (on the device, before timing) into the pages'
        # V1 layout: keys [blocks, kv_heads, head_dim / 8, block_size, 8],
        # values [blocks, kv_heads, head_dim, block_size]
        nb, hkv, bsz, dh = batch.k_cache.shape
        xg = 16 // batch.k_cache.element_size()
        k5 = batch.k_cache.view(nb, hkv, bsz, dh // xg, xg).permute(0, 1, 3, 2, 4).contiguous()
        v4 = batch.v_cache.permute(0, 1, 3, 2).contiguous()
        batch = dataclasses.replace(batch, k_cache=k5, v_cache=v4)
        sx = dict(split_x=True)
    params = pa.make_params(batch.q, batch.k_cache, batch.block_tables,
                            max_seq_len=batch.max_seq_len, scale=batch.scale, partition_size=P,
                            out_dtype=torch.float32, **sx)
    path = pa.decode_path(params) if args.path == "decode" else (1 if args.path == "v1" else 2)
    family = pa.decode_kernel(params)
    # kernel launches of the step on this path (V2: one when pass 1 merges its
    # own partials, two with the dependent reduce kernel)
    launches_per_step = pa.decode_launches(pa.make_params(
        batch.q, batch.k_cache, batch.block_tables, max_seq_len=batch.max_seq_len,
        scale=batch.scale, partition_size=P, out_dtype=torch.float32,
        v1_max_seq_len=max(batch.max_seq_len, 1) if path == 1 else 1, **sx))
    one_launch_v2 = path == 2 and launches_per_step == 1
    kname = ("pa_sx_kernel" if family == 2 and args.split_x else
             "pa_tc_kernel" if family == 2 else "pa_generic_kernel") + \
        (" (V2 in one launch: pass 1 + merge)" if one_launch_v2 else
         " (V2 pass 1)" if path == 2 else " (V1)")
    ws = pa.alloc_workspace(params, device=device)
    out = torch.empty(tuple(batch.q.shape), dtype=torch.float32, device=device)
    flush_buf = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=device)
    flush_sink = torch.empty((), dtype=torch.int32, device=device)

    class _Flush:
        def zero_(self):
            # a read sweep larger than L2: evicts it without leaving dirty lines
            torch.amax(flush_buf, dim=0, out=flush_sink)
            # then keep the GPU busy for ~100 us so the host has enqueued the
            # step (and its events) before the GPU reaches the start event:
            # the event window then holds device time only
            torch.cuda._sleep(200_000)

    flush = _Flush()
    stream = torch.cuda.current_stream(device)
    kw = dict(max_seq_len=batch.max_seq_len, scale=batch.scale, partition_size=P, **sx)

    def step():
        if args.path == "decode":
            pa.decode(batch.q, batch.k_cache, batch.v_cache, batch.block_tables, batch.seq_lens,
                      out, ws, **kw)
        elif args.path == "v1":
            pa.decode_v1(batch.q, batch.k_cache, batch.v_cache, batch.block_tables,
                         batch.seq_lens, out, max_seq_len=batch.max_seq_len, scale=batch.scale,
                         **sx)
        else:
            pa.decode_v2(batch.q, batch.k_cache, batch.v_cache, batch.block_tables,
                         batch.seq_lens, out, ws, **kw)

    kv_bytes = batch.kv_bytes()
    alg_bytes = kv_bytes + batch.q_bytes()

    sampler = ClockSampler(gpu_id_for_smi(device))
    if rank == 0:
        sampler.start()
        sampler.wait_first()
    t_gpu0 = time.time()
    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize(device)

    # ---- timed region: K full steps, events around each step ----------------
    # Inputs larger than L2 (2x its 129 MB): the K steps run back to back, as
    # a decode loop runs them, between one pair of events (the L2 is evicted
    # once before; each step streams more than L2 holds).  Smaller inputs: an
    # L2-evicting read sweep before every step, each step between its own
    # events.  The per-step-after-sweep time is reported for every workload.
    back_to_back = kv_bytes > 2 * L2_BYTES
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(device)
    t_start = time.time()
    loop_ms = None
    if back_to_back:
        e_loop = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
        flush.zero_()
        torch.cuda._sleep(2_000_000)  # ~1 ms: the host queues the steps ahead of the GPU
        e_loop[0].record(stream)
        for i in range(args.steps):
            step()
        e_loop[1].record(stream)
        torch.cuda.synchronize(device)
        loop_ms = e_loop[0].elapsed_time(e_loop[1]) / args.steps
    for i in range(args.steps):
        flush.zero_()
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize(device)
    if world > 1:
        torch.distributed.barrier()
    t_end = time.time()
    flushed_ms = [a.elapsed_time(b) for a, b in ev]
    step_ms = [loop_ms] if back_to_back else flushed_ms
    out_step = out.clone()   # the step's result (the two-call form below rewrites out)

    # ---- the dominant kernel: the step itself when it is one launch; with two
    # launches, V2 pass 1 alone.  The two-call form (pass 1, then the reduce)
    # is timed for V2 either way, as context.
    dom_ms, red_ms, p1_ms = [], [], []
    if path == 2:
        evp = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
        for i in range(args.steps):
            flush.zero_()
            evp[i][0].record(stream)
            pa.decode_v2_partitions(batch.q, batch.k_cache, batch.v_cache, batch.block_tables,
                                    batch.seq_lens, ws, out_dtype=torch.float32, **kw)
            evp[i][1].record(stream)
            pa.decode_v2_reduce(params, batch.seq_lens, ws, out)
            evp[i][2].record(stream)
        torch.cuda.synchronize(device)
        p1_ms = [e[0].elapsed_time(e[1]) for e in evp]
        red_ms = [e[1].elapsed_time(e[2]) for e in evp]
    dom_ms = p1_ms if (path == 2 and not one_launch_v2) else step_ms
    if path == 2 and not one_launch_v2 and back_to_back:
        # pass 1 alone, back to back like the steps
        e_p = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
        flush.zero_()
        torch.cuda._sleep(2_000_000)
        e_p[0].record(stream)
        for i in range(args.steps):
            pa.decode_v2_partitions(batch.q, batch.k_cache, batch.v_cache, batch.block_tables,
                                    batch.seq_lens, ws, out_dtype=torch.float32, **kw)
        e_p[1].record(stream)
        torch.cuda.synchronize(device)
        dom_ms = [e_p[0].elapsed_time(e_p[1]) / args.steps]
    t_dom_end = time.time()

    # ---- end to end through the C ABI with host buffers ---------------------
    # pa_decode_host: q, block table and lengths copied in from pinned host
    # memory, the step, the result copied back, and the wait -- all inside
    # the timed region; the caches and the workspace stay resident.
    # the same path as the device-timed step (pa_decode's threshold, or V1 / V2
    # forced through it)
    v1max = {"v1": max(batch.max_seq_len, 1), "v2": 1}.get(args.path, pa.DEFAULT_V1_MAX_SEQ_LEN)
    hparams = pa.make_params(batch.q, batch.k_cache, batch.block_tables,
                             max_seq_len=batch.max_seq_len, scale=batch.scale, partition_size=P,
                             out_dtype=out.dtype, v1_max_seq_len=v1max, **sx)
    # the host inputs live in a pinned mirror of the staging layout, so the
    # call moves them in one copy
    mbuf, q_h, bt_h, sl_h = pa.alloc_host_mirror(hparams, batch.q.dtype, *batch.q.shape,
                                                 batch.block_tables.shape[1])
    q_h.copy_(batch.q.cpu())
    bt_h.copy_(batch.block_tables.cpu())
    sl_h.copy_(batch.seq_lens.cpu())
    out_h = torch.empty(tuple(out.shape), dtype=out.dtype).pin_memory()
    staging = pa.alloc_host_staging(hparams, device=device)
    ws_host = ws if pa.decode_path(hparams) == 2 else None
    e2e_s = []
    for i in range(args.warmup + args.steps):
        flush.zero_()
        torch.cuda.synchronize(device)
        t0 = time.perf_counter()
        pa.decode_host(q_h, batch.k_cache, batch.v_cache, bt_h, sl_h, out_h, ws_host, staging,
                       params=hparams, stream=stream)
        if i >= args.warmup:
            e2e_s.append(time.perf_counter() - t0)
    assert torch.equal(out_h, out_step.cpu()), "host-buffer step differs from the device step"
    h2d = q_h.numel() * q_h.element_size() + bt_h.numel() * 4 + sl_h.numel() * 4
    d2h = out_h.numel() * out_h.element_size()

    # ---- the end-to-end step taken apart ----------------------------------
    # The operations pa_decode_host enqueues (one copy of the mirrored inputs
    # into the staging buffer, the decode on the staged inputs, the copy of
    # the result back), issued one by one with stream events between them
    # while the GPU is still busy with a ~0.5 ms spin, so that every part is
    # queued before the first starts and the events hold device time only.
    # The rest of the end-to-end time (e2e minus the three parts) is host
    # time: issuing the copies and the launch, and the wait's wake-up.
    offs = pa.host_staging_offsets(hparams)
    n_in = offs[2] + sl_h.numel() * 4
    mirror_u8 = mbuf[:n_in]
    q_d = staging[:offs[1]].view(batch.q.dtype)[:batch.q.numel()].view(tuple(batch.q.shape))
    bt_d = staging[offs[1]:offs[2]].view(torch.int32)[:bt_h.numel()].view(tuple(bt_h.shape))
    sl_d = staging[offs[2]:offs[3]].view(torch.int32)[:sl_h.numel()]
    out_d = staging[offs[3]:].view(out.dtype)[:out.numel()].view(tuple(out.shape))
    parts = {"h2d": [], "step": [], "d2h": []}
    for i in range(args.warmup + args.steps):
        flush.zero_()
        torch.cuda._sleep(1_000_000)
        e = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        e[0].record(stream)
        staging[:n_in].copy_(mirror_u8, non_blocking=True)
        e[1].record(stream)
        pa.decode(q_d, batch.k_cache, batch.v_cache, bt_d, sl_d, out_d, ws_host,
                  max_seq_len=batch.max_seq_len, scale=batch.scale, partition_size=P,
                  v1_max_seq_len=v1max, **sx)
        e[2].record(stream)
        out_h.copy_(out_d, non_blocking=True)
        e[3].record(stream)
        torch.cuda.synchronize(device)
        if i >= args.warmup:
            parts["h2d"].append(e[0].elapsed_time(e[1]))
            parts["step"].append(e[1].elapsed_time(e[2]))
            parts["d2h"].append(e[2].elapsed_time(e[3]))
    assert torch.equal(out_h, out_step.cpu()), "the step taken apart differs from the device step"
    hold = hold_until_sampled(sampler, t_gpu0, step, device) if rank == 0 else 0
    t_gpu1 = time.time()
    if rank == 0:
        sampler.stop()

    assert pa.read_device_status(ws) == pa.PA_OK, "device status not OK after the bench"
    assert torch.isfinite(out_step).all().item(), "non-finite output"

    # reduce over ranks: max of times
    t_step, t_dom, t_e2e = max_over_ranks(
        [statistics.mean(step_ms), statistics.mean(dom_ms), statistics.mean(e2e_s) * 1e3], world,
        device)

    peak, peak_kind = measured_hbm_peak()
    achieved = alg_bytes / (t_dom * 1e-3) / 1e9
    traffic = ncu_traffic(kname.split(" ")[0], args.workload, P, "v2" if path == 2 else "v1")
    result = {
        "metric": METRIC,
        "value": round(t_step * 1e3, 3),
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(t_step, 6),
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if w.dtype == torch.bfloat16 else str(w.dtype).replace("torch.", ""),
        "data": "synthetic (seeded N(0,1) q/k/v, 0.1% of keys x30, random block table)",
        "config": {
            "workload": f"{w.name}: {w.num_seqs} seq x {batch.max_seq_len} tokens, "
                        f"{w.num_heads} q / {w.num_kv_heads} kv heads, head_dim {w.head_dim}, "
                        f"{str(w.dtype).replace('torch.', '')} KV, block {w.block_size}",
            "partition_size": P,
            "cache_layout": ("split-x (keys [blocks, kv_heads, head_dim/8, block, 8], values "
                             "[blocks, kv_heads, head_dim, block])" if args.split_x else
                             "[blocks, kv_heads, block, head_dim]"),
            "path": ("V2 in one launch (partition kernel merging its own partials)"
                     if one_launch_v2 else
                     "V2 (partition kernel + LSE reduce)" if path == 2 else "V1 single pass") +
                    (" via pa_decode" if args.path == "decode" else " forced"),
            "accumulate": "f32",
            "l2": (f"inputs larger than L2 (KV {kv_bytes / 1e6:.1f} MB > 2 x 129 MB): the timed "
                   "steps run back to back between one pair of CUDA events, after one 256 MiB "
                   "read sweep; step_after_flush_us times each step alone after its own sweep"
                   if back_to_back else
                   f"KV {kv_bytes / 1e6:.1f} MB fits in L2, so a 256 MiB read sweep evicts L2 "
                   "before every timed step"),
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
        },
        "step_after_flush_us": round(statistics.mean(flushed_ms) * 1e3, 3),
        "kv_read_gbs": round(world * alg_bytes / (t_step * 1e-3) / 1e9, 1),
        "hbm_frac_of_step": round(alg_bytes / (t_step * 1e-3) / 1e9 / peak, 4),
        "roofline": {
            "bound": "hbm",
            "kernel": kname,
            "achieved": round(achieved, 1),
            "peak": peak,
            "peak_source": f"{peak_kind} hbm_gbs (copy)",
            "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "traffic": traffic,
            "algorithmic_bytes_per_launch": alg_bytes,
            "launch_us": round(t_dom * 1e3, 3),
        },
        "two_call_form_us": ({"pass1": round(statistics.mean(p1_ms) * 1e3, 3),
                              "reduce": round(statistics.mean(red_ms) * 1e3, 3)}
                             if red_ms else None),
        "e2e": {"value": round(t_e2e * 1e3, 3), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "parts_us": dict(
                    {k: round(statistics.mean(v) * 1e3, 3) for k, v in parts.items()},
                    host=round(t_e2e * 1e3 - sum(statistics.mean(v) * 1e3
                                                 for v in parts.values()), 3)),
                "parts_how": "device time of the operations of pa_decode_host queued one by one "
                             "behind a GPU spin with stream events between them: h2d = one copy "
                             "of the pinned mirrored inputs, step = pa_decode on the staged "
                             "inputs, d2h = the result back; host = e2e minus the three "
                             "(issuing the copies and launch, the wait's wake-up)"},
        "gpu_launches": launches_per_step * args.steps,
    }
    if rank == 0:
        result["clocks"] = sampler.summary(t_gpu0, t_gpu1)
        result["clocks"]["window"] = (
            "whole GPU run: warm-up, timed steps, kernels timed apart, end-to-end loops"
            + (f", plus {hold} untimed steps until 5 samples" if hold else ""))
        result["clocks"]["timed_region_samples"] = sampler.count(t_start, t_end)
        if world == 1 and not args.no_cpu_baseline:
            result["cpu_baseline"] = cpu_baseline(batch, args.cpu_rows, args.cpu_seconds)
    return result


# ---------------------------------------------------------------------------
# prefill workloads (pa_prefill): TFLOP/s of the causal attention work
# ---------------------------------------------------------------------------
PREFILL_METRIC = "paged prefix-prefill attention TFLOP/s (causal FLOPs, tensor-core roofline)"
PREFILL_UNIT = "TFLOP/s"


def prefill_flops(pb) -> int:
    """Algorithmic FLOPs of one prefill step: 4 * D per (query head, query,
    visible key) -- 2 D for q . k and 2 D for p * v -- where query i of
    sequence b sees its C_b context tokens and chunk tokens 0..i."""
    w = pb.workload
    total = 0
    for b in range(w.num_seqs):
        n = int(pb.query_start[b + 1]) - int(pb.query_start[b])
        C = int(pb.ctx_lens[b])
        total += n * C + n * (n + 1) // 2
    return 4 * w.head_dim * w.num_heads * total


def measured_tensor_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return 1900.0, "fallback"


def run_prefill(args, rank, world, device):
    w = wl.PREFILL_WORKLOADS[args.workload]
    pb = wl.make_prefill(w, device=device)
    out = torch.empty(tuple(pb.q.shape), dtype=torch.float32, device=device)
    flush_buf = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=device)
    flush_sink = torch.empty((), dtype=torch.int32, device=device)
    stream = torch.cuda.current_stream(device)
    kw = dict(max_query_len=pb.max_query_len, max_ctx_len=pb.max_ctx_len, scale=pb.scale)

    def flush():
        torch.amax(flush_buf, dim=0, out=flush_sink)
        torch.cuda._sleep(200_000)

    def step(q, k, v, qs, cl, bt, o):
        pa.prefill(q, k, v, pb.k_cache, pb.v_cache, bt, qs, cl, o, **kw)

    flops = prefill_flops(pb)
    sampler = ClockSampler(gpu_id_for_smi(device))
    if rank == 0:
        sampler.start()
        sampler.wait_first()
    t_gpu0 = time.time()
    for _ in range(args.warmup):
        flush()
        step(pb.q, pb.k, pb.v, pb.query_start, pb.ctx_lens, pb.block_tables, out)
    torch.cuda.synchronize(device)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(device)
    t_start = time.time()
    for i in range(args.steps):
        flush()
        ev[i][0].record(stream)
        step(pb.q, pb.k, pb.v, pb.query_start, pb.ctx_lens, pb.block_tables, out)
        ev[i][1].record(stream)
    torch.cuda.synchronize(device)
    if world > 1:
        torch.distributed.barrier()
    t_end = time.time()
    step_ms = [a.elapsed_time(b) for a, b in ev]

    # end to end: the chunk's q / k / v, block table and lengths copied in
    # from pinned host memory, the call, the output copied back and waited for
    host = {n: getattr(pb, n).cpu().pin_memory()
            for n in ("q", "k", "v", "query_start", "ctx_lens", "block_tables")}
    dev = {n: torch.empty_like(getattr(pb, n)) for n in host}
    out_h = torch.empty(tuple(out.shape), dtype=out.dtype).pin_memory()
    e2e_s = []
    for i in range(args.warmup + args.steps):
        flush()
        torch.cuda.synchronize(device)
        t0 = time.perf_counter()
        for n in host:
            dev[n].copy_(host[n], non_blocking=True)
        step(dev["q"], dev["k"], dev["v"], dev["query_start"], dev["ctx_lens"],
             dev["block_tables"], out)
        out_h.copy_(out, non_blocking=True)
        torch.cuda.synchronize(device)
        if i >= args.warmup:
            e2e_s.append(time.perf_counter() - t0)
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = out_h.numel() * out_h.element_size()
    hold = 0
    if rank == 0:
        hold = hold_until_sampled(sampler, t_gpu0, lambda: step(
            pb.q, pb.k, pb.v, pb.query_start, pb.ctx_lens, pb.block_tables, out), device)
    t_gpu1 = time.time()
    if rank == 0:
        sampler.stop()
    assert torch.isfinite(out).all().item(), "non-finite output"

    t_step, t_e2e = max_over_ranks([statistics.mean(step_ms), statistics.mean(e2e_s) * 1e3],
                                   world, device)
    tflops = world * flops / (t_step * 1e-3) / 1e12
    peak, peak_kind = measured_tensor_peak()
    result = {
        "metric": PREFILL_METRIC,
        "value": round(tflops, 2),
        "unit": PREFILL_UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(t_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) q / k / v and cached context, random block table)",
        "config": {
            "workload": f"{w.name}: {w.num_seqs} seq(s), chunk(s) of "
                        f"{[int(pb.query_start[b + 1] - pb.query_start[b]) for b in range(w.num_seqs)]}"
                        f" tokens after {[int(x) for x in pb.ctx_lens]} cached, {w.num_heads} q / "
                        f"{w.num_kv_heads} kv heads, head_dim {w.head_dim}, "
                        f"{str(w.dtype).replace('torch.', '')}, block {w.block_size}",
            "accumulate": "f32",
            "l2": "a 256 MiB read sweep evicts L2 before every timed step",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
        },
        "roofline": {
            "bound": "tensor",
            "kernel": "pa_prefill_kernel",
            "achieved": round(flops / (t_step * 1e-3) / 1e12, 2),
            "peak": peak,
            "peak_source": f"{peak_kind} bf16_tflops (cuBLAS burst)",
            "unit": "TFLOP/s",
            "frac": round(flops / (t_step * 1e-3) / 1e12 / peak, 4),
            "traffic": ncu_traffic("pa_prefill_kernel", w.name, 0, "prefill"),
            "algorithmic_flops_per_launch": flops,
            "launch_ms": round(t_step, 4),
        },
        "e2e": {"value": round(world * flops / (t_e2e * 1e-3) / 1e12, 2), "unit": PREFILL_UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": args.steps,
    }
    if rank == 0:
        result["clocks"] = sampler.summary(t_gpu0, t_gpu1)
        result["clocks"]["window"] = (
            "whole GPU run: warm-up, timed steps, end-to-end loop"
            + (f", plus {hold} untimed steps until 5 samples" if hold else ""))
        result["clocks"]["timed_region_samples"] = sampler.count(t_start, t_end)
        if world == 1 and not args.no_cpu_baseline:
            result["cpu_baseline"] = cpu_baseline_prefill(pb, args.cpu_rows, args.cpu_seconds)
    return result


def _prefill_row_work(pb, rows):
    """Visible keys summed over the given flat (token * Hq + head) rows."""
    w = pb.workload
    qs = [int(x) for x in pb.query_start]
    work = 0
    for r in rows:
        t = r // w.num_heads
        b = max(i for i in range(w.num_seqs) if qs[i] <= t)
        work += int(pb.ctx_lens[b]) + (t - qs[b]) + 1
    return work


def cpu_baseline_prefill(pb, nrows, seconds, threads=None):
    """The prefill oracle timed on the host cores on a spread sample of rows,
    repeated for ``seconds``, scaled to the step's full (row x visible key)
    work."""
    import oracle
    pc = pb.to("cpu")
    w = pc.workload
    T = pc.q.shape[0]
    total_rows = T * w.num_heads
    rows = [int(i * (total_rows - 1) / max(1, nrows - 1)) for i in range(nrows)]
    total = sum(int(pc.ctx_lens[b]) * (int(pc.query_start[b + 1]) - int(pc.query_start[b]))
                for b in range(w.num_seqs))
    total += sum(n * (n + 1) // 2 for n in
                 (int(pc.query_start[b + 1]) - int(pc.query_start[b]) for b in range(w.num_seqs)))
    total *= w.num_heads
    work = _prefill_row_work(pc, rows)
    spent, reps = 0.0, 0
    while reps == 0 or spent < seconds:
        t0 = time.perf_counter()
        oracle.prefill(pc.q, pc.k, pc.v, pc.k_cache, pc.v_cache, pc.block_tables,
                       pc.query_start, pc.ctx_lens, pc.scale, rows=rows)
        spent += time.perf_counter() - t0
        reps += 1
    step_s = spent / reps * total / work
    flops = prefill_flops(pc)
    return {"value": round(flops / step_s / 1e12, 6), "unit": PREFILL_UNIT,
            "cores": oracle.max_threads(), "kind": "oracle",
            "sample": f"{len(rows)} of {total_rows} query-head rows spread over the chunk, "
                      f"{reps} repetitions ({spent:.1f} s), scaled by visible-key work to the "
                      f"full step ({step_s * 1e3:.0f} ms)"}


# ---------------------------------------------------------------------------
# the oracle on the host cores (cpu_baseline leg and the reference arm)
# ---------------------------------------------------------------------------
def _oracle_rows(batch_cpu, rows):
    import oracle
    t0 = time.perf_counter()
    oracle.decode(batch_cpu.q, batch_cpu.k_cache, batch_cpu.v_cache, batch_cpu.block_tables,
                  batch_cpu.seq_lens, batch_cpu.scale, rows=rows)
    return time.perf_counter() - t0


def cpu_baseline(batch, nrows, seconds):
    """The oracle timed on the host cores: the first ``nrows`` query-head rows
    of the step, repeated until ``seconds`` of CPU work have run, scaled to
    one full step."""
    import oracle
    bc = batch.to("cpu")
    w = bc.workload
    total_rows = w.num_seqs * w.num_heads
    rows = list(range(min(nrows, total_rows)))
    spent, reps = 0.0, 0
    while reps == 0 or spent < seconds:
        spent += _oracle_rows(bc, rows)
        reps += 1
    per_step_us = spent / reps * 1e6 * total_rows / len(rows)
    cores = oracle.max_threads()
    one_core = None  # the same sample once more on one core
    if cores > 1:
        oracle.set_threads(1)
        try:
            one_core = round(_oracle_rows(bc, rows) * 1e6 * total_rows / len(rows), 1)
        finally:
            oracle.set_threads(cores)
    return {"value": round(per_step_us, 1), "unit": UNIT, "cores": cores, "kind": "oracle",
            "one_core_value": one_core,
            "sample": f"{len(rows)} of {total_rows} query-head rows of one step, "
                      f"{reps} repetitions ({spent:.1f} s) on {cores} cores and one more on "
                      f"one core, scaled to the full step"}


def run_reference(args, rank, world):
    """The reference arm: the float64 oracle, as it stands, on all host
    cores.  A decode step is the whole batch (every query-head row) when
    the run fits --ref-budget-s, else an even spread of rows scaled to the
    step's work; a prefill step computes 8 spread rows scaled by
    visible-key work (a whole prefill step takes minutes on the host)."""
    if rank != 0:
        return None
    import oracle
    if args.workload in wl.PREFILL_WORKLOADS:
        pb = wl.make_prefill(wl.PREFILL_WORKLOADS[args.workload])
        base = cpu_baseline_prefill(pb, 8, 0.0)
        times = []
        for i in range(args.warmup + args.steps):
            b = cpu_baseline_prefill(pb, 8, 0.0)
            if i >= args.warmup:
                times.append(b["value"])
        v = round(statistics.mean(times), 6)
        return {
            "impl": "reference",
            "metric": PREFILL_METRIC, "value": v, "unit": PREFILL_UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": args.workload},
            "cpu_baseline": {"value": v, "unit": PREFILL_UNIT, "cores": base["cores"],
                             "kind": "oracle", "sample": base["sample"]},
            "e2e": {"value": v, "unit": PREFILL_UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
        }
    w = wl.WORKLOADS[args.workload]
    P = args.partition_size or w.partition_sizes[0]
    bc = wl.make(w, device="cpu")
    total_rows = w.num_seqs * w.num_heads
    # Whole steps (every query-head row of the batch) when the run fits the
    # budget; otherwise each step computes an even spread of rows, as many as
    # fit, and its time is scaled by the step's row x token work.
    t_full = _oracle_rows(bc, None)
    n_all = args.warmup + args.steps
    lens = bc.seq_lens.tolist()
    if t_full * n_all <= args.ref_budget_s:
        rows, scale_f = None, 1.0
        how = f"whole steps: all {total_rows} query-head rows of the batch"
    else:
        k = max(1, int(total_rows * args.ref_budget_s / (t_full * n_all)))
        rows = [int(i * total_rows / k) for i in range(k)]
        work = sum(lens[r // w.num_heads] for r in rows)
        scale_f = sum(lens) * w.num_heads / max(1, work)
        how = (f"{k} of {total_rows} query-head rows per step (evenly spread), scaled by the "
               f"step's row x token work")
    times = []
    for i in range(n_all):
        dt = _oracle_rows(bc, rows)
        if i >= args.warmup:
            times.append(dt * scale_f)
    t = statistics.mean(times)
    v = round(t * 1e6, 1)
    cores = oracle.max_threads()
    return {
        "impl": "reference",
        "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(t * 1e3, 3), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "partition_size": P},
        "cpu_baseline": {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": how},
        "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default="long_100k",
                    choices=sorted(wl.WORKLOADS) + sorted(wl.PREFILL_WORKLOADS))
    ap.add_argument("--partition-size", type=int, default=0)
    ap.add_argument("--split-x", action="store_true",
                    help="caches in the pages' V1 split-x layout (read directly)")
    ap.add_argument("--path", choices=("decode", "v1", "v2"), default="decode",
                    help="pa_decode (threshold dispatch), or force V1 / V2")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="host time the oracle baseline runs for (whole repetitions)")
    ap.add_argument("--cpu-rows", type=int, default=24,
                    help="query-head rows the CPU baseline computes")
    ap.add_argument("--ref-budget-s", type=float, default=150.0,
                    help="host seconds the reference arm may spend in all its steps")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world != args.gpus:
        if world == 1 and args.gpus > 1:
            ap.error("--gpus N > 1 needs torchrun --nproc-per-node N")
    if args.impl == "reference":
        if world > 1:
            torch.distributed.init_process_group("gloo")
        res = run_reference(args, rank, world)
        if res is not None:
            print(json.dumps(res), flush=True)
        if world > 1:
            torch.distributed.destroy_process_group()
        return

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    from paged_attention_decode_v2_gb300 import build
    if rank == 0 or world == 1:
        build.build()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=device)
        torch.distributed.barrier()
        if rank != 0:
            build.build()
    if args.workload in wl.PREFILL_WORKLOADS:
        res = run_prefill(args, rank, world, device)
    else:
        res = run_ours(args, rank, world, device)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
