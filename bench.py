#!/usr/bin/env python
"""Benchmark: sparse shared-KV MLA attention, CSA decode, one GB300 per rank.

A step is one pass of the whole hot path over one batch: the device planner
(sfm_metadata) and the attention + split combine (sfm_forward) for B = 32
decode query rows of q_n = 64 heads, each attending a 128-row window of its
paged ori cache plus 512 top-k compressed rows (cmp_ratio 4).  Inputs are
synthetic (seeded), resident in HBM, and rotate over enough independent input
sets that the attended bytes of consecutive steps never sit in L2.

Metric: attended KV rows per second (each attended row counted once per query
row, not per head), reported with TFLOP/s and the roofline of the dominant
kernel.  ``e2e`` repeats the measurement through the public two-call API with
the step's inputs copied from pinned host memory and O / LSE read back.

``--impl reference`` times the CPU oracle (fp64, all host cores) on the same
workload instead; it is a deliberately slow correctness reference, not a
competitor.

Multi-GPU: the path has no exchange step, so N ranks run N independent
replicas (weak scaling); the time is the max over ranks.
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
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

NOMINAL_HBM_GBS = 7900.0      # HBM3e, nominal (the measured copy rate is the stricter denominator)
WORKLOADS = ("csa_decode", "hca_decode", "packed_decode", "packed_fp8_decode", "csa_prefill")
S_KV_FORMAT_CODES = {"plain": 0, "int8_packed": 1, "fp8_packed": 2}     # sfm_params.kv_format


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", choices=WORKLOADS, default="csa_decode")
    ap.add_argument("--sets", type=int, default=0,
                    help="rotating input sets (0: enough that their attended bytes exceed 3x L2, at most 16)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-second", action="store_true",
                    help="skip the HCA decode block that follows the CSA decode headline")
    ap.add_argument("--compact-pool", action="store_true",
                    help="HCA decode: store only the paged blocks the window reads (same attended rows and bytes; "
                         "a small device footprint for profiler captures)")
    ap.add_argument("--batch", type=int, default=None,
                    help="override the workload's batch size (small-batch measurements; not the headline)")
    ap.add_argument("--split-policy", choices=("invariant", "occupancy"), default="invariant",
                    help="sfm_params.split_policy: batch-invariant splits (the default) or occupancy splits")
    ap.add_argument("--no-small-batch", action="store_true",
                    help="skip the small-batch block (CSA / HCA decode at B = 4, 8, 16 under both split policies)")
    ap.add_argument("--streams", type=int, default=8,
                    help="streams that the concurrent-step and end-to-end legs spread independent input sets over")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    return ap.parse_args()


# ---------------------------------------------------------------------------
# distributed plumbing (replicas only)
# ---------------------------------------------------------------------------
def dist_init(backend):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group(backend=backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class _NvmlClocks:
    """SM clock and clock-event reasons read through the driver's NVML
    library (read-only queries, microseconds each), for sampling far more
    often than nvidia-smi's loop delivers lines."""
    CLOCK_SM = 1                       # NVML_CLOCK_SM
    # clock-event reason bits of NVML's public header
    BITS = ((0x8, "hw_slowdown"), (0x40, "hw_thermal_slowdown"), (0x20, "sw_thermal_slowdown"),
            (0x4, "sw_power_cap"))

    def __init__(self, uuid: str):
        import ctypes
        self.ct = ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit_v2 failed")
        self.lib = lib
        self.h = ctypes.c_void_p()
        if lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(self.h)) != 0:
            raise OSError("no NVML handle for " + uuid)
        try:
            self.reasons_fn = lib.nvmlDeviceGetCurrentClocksEventReasons
        except AttributeError:
            self.reasons_fn = lib.nvmlDeviceGetCurrentClocksThrottleReasons
        mx = ctypes.c_uint()
        if lib.nvmlDeviceGetMaxClockInfo(self.h, self.CLOCK_SM, ctypes.byref(mx)) != 0:
            raise OSError("nvmlDeviceGetMaxClockInfo failed")
        self.max_mhz = float(mx.value)

    def read(self):
        sm, bits = self.ct.c_uint(), self.ct.c_ulonglong()
        if self.lib.nvmlDeviceGetClockInfo(self.h, self.CLOCK_SM, self.ct.byref(sm)) != 0:
            return None
        if self.reasons_fn(self.h, self.ct.byref(bits)) != 0:
            return None
        return float(sm.value), [n for b, n in self.BITS if bits.value & b]


class ClockSampler:
    """Clocks and throttle reasons while the bench runs: nvidia-smi's query
    loop and, where the driver's NVML library loads, a 2 ms NVML poll (the
    timed steps of a decode workload last milliseconds, shorter than
    nvidia-smi's line interval on these hosts)."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []
        self.t = None
        self.nvml = None
        self.nv_rows = []
        self.done = threading.Event()
        self.poller = None

    def start(self):
        try:
            self.nvml = _NvmlClocks(self.gpu_id)
        except (OSError, AttributeError):
            self.nvml = None
        if self.nvml is not None:
            self.poller = threading.Thread(target=self._poll, daemon=True)
            self.poller.start()
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def _poll(self):
        while not self.done.is_set():
            v = self.nvml.read()
            if v is not None:
                self.nv_rows.append((time.time(), v[0], self.nvml.max_mhz, v[1]))
            time.sleep(0.002)

    def mark(self):
        return time.time()

    def stop(self):
        self.done.set()
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def _smi_rows(self):
        rows = []
        for ts, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                active = [n for n, f in zip(self.NAMES, parts[4:8]) if f.lower() == "active"]
                rows.append((ts, float(parts[0]), float(parts[1]), active))
            except ValueError:
                continue
        return rows

    def summary(self, t0=None, t1=None, t1_legs=None, t0_warm=None):
        rows, source = list(self.nv_rows), "NVML, 2 ms poll"
        if not rows:
            rows, source = self._smi_rows(), "nvidia-smi"
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no clock samples"], "samples": 0}
        inside = [r for r in rows if (t0 is None or r[0] >= t0) and (t1 is None or r[0] <= t1)]
        window = "timed region"
        if len(inside) < 5 and t1_legs is not None:
            # a timed region of a few ms holds few samples: take every timed
            # leg of the workload (they follow the steps back to back), then
            # the whole run of the workload from its first warm-up step
            legs = [r for r in rows if (t0 is None or r[0] >= t0) and r[0] <= t1_legs]
            if len(legs) > len(inside):
                inside, window = legs, "timed steps and the timed legs after them"
            if len(inside) < 5 and t0_warm is not None:
                busy = [r for r in rows if t0_warm <= r[0] <= t1_legs]
                if len(busy) > len(inside):
                    inside, window = busy, "warm-up, timed steps and the timed legs after them"
        if not inside:
            inside, window = rows, "warm-up + timed region"
        reasons = sorted({n for r in inside for n in r[3]})
        return {"sm_mhz": statistics.median(r[1] for r in inside), "sm_max_mhz": max(r[2] for r in inside),
                "reasons": reasons, "samples": len(inside), "window": window, "source": source}


# ---------------------------------------------------------------------------
# workload accounting (algorithmic bytes / FLOPs)
# ---------------------------------------------------------------------------
def make_problem(workload, device, seed, batch=None, compact_pool=False):
    import sfm_inputs as S
    kw = {} if batch is None or workload in ("swa_decode_tiny", "csa_prefill") else {"batch": batch}
    if compact_pool and workload == "hca_decode":
        kw["compact_pool"] = True
    return S.WORKLOADS[workload](device=device, seed=seed, **kw)


def accounting(prob, sfm):
    """Attended rows, algorithmic HBM bytes and FLOPs of one pass over the
    batch, from the KV rows the attention kernel's resolver actually hands to
    its copy warps (sfm_debug_attended: the forward with its row dump on)."""
    params = sfm.make_params(**prob.attrs())
    tens = sfm.make_tensors(prob.t["q"], prob.t["ori_kv"], **prob.tensor_kwargs())
    cap = ((prob.ori_topk * prob.sparse_block_size) or (prob.ori_win_left + prob.ori_win_right + 1)) + \
        (prob.cmp_topk or prob.max_seqlen_cmp_kv)
    dev = prob.t["q"].device
    md = torch.empty(sfm.sfm_metadata_size(params), dtype=torch.int32, device=dev)
    nb = sfm.sfm_workspace_size(params)
    ws = torch.empty(nb, dtype=torch.uint8, device=dev) if nb else None
    out = torch.empty(prob.t["q"].shape[:-1] + (512,), dtype=prob.torch_dtype, device=dev)
    lse = torch.empty(prob.num_tokens * prob.num_heads_q, dtype=torch.float32, device=dev) \
        if params.return_lse else None
    unwritten = -2
    rows = torch.full((prob.num_tokens, cap), unwritten, dtype=torch.int32, device=dev)
    counts = torch.zeros(prob.num_tokens, dtype=torch.int32, device=dev)
    sfm.sfm_metadata(params, tens, md)
    sfm.sfm_debug_attended(params, tens, md, prob.softmax_scale, out, lse, ws, rows, cap, counts)
    torch.cuda.synchronize()
    valid = (rows != -1) & (rows != unwritten)
    attended = int(valid.sum().item())
    # distinct KV rows read by the batch: (pool, row) pairs (entries name
    # rows of the cache buffers, bit 31 marks the compressed pool); query rows
    # of one sequence share most of their rows in prefill
    distinct = int(torch.unique(rows[valid]).numel())
    # block-table entries touched: distinct (query row, pool, block) triples
    bt_entries = 0
    if prob.layout_kv == "PAGED":
        cmp_pool = rows < 0
        r = rows.to(torch.int64) & 0x7FFFFFFF
        for is_cmp, bs in ((False, prob.ori_block_size), (True, prob.cmp_block_size)):
            if bs <= 0:
                continue
            m = valid & (cmp_pool == is_cmp)
            blk = torch.where(m, r // bs, torch.full_like(r, -1))
            srt, _ = torch.sort(blk, dim=1)
            new = (srt[:, 1:] != srt[:, :-1]) & (srt[:, 1:] >= 0)
            bt_entries += int(new.sum().item() + (srt[:, :1] >= 0).sum().item())
    T, qn = prob.num_tokens, prob.num_heads_q
    row_bytes = prob.kv_row_bytes()
    idx_entries = T * (prob.ori_topk + prob.cmp_topk)
    bytes_ = (distinct * row_bytes + T * qn * prob.d_qk * 2 + T * qn * 512 * 2 + T * qn * 4 + idx_entries * 4
              + bt_entries * 4 + prob.batch_size * 4 * 3)
    flops = attended * qn * (2 * prob.d_qk + 2 * 512)
    return {"attended_rows": attended, "distinct_rows": distinct, "bytes": bytes_, "flops": flops,
            "bt_entries": bt_entries}


# the sources the tensor-core attention kernel (the dominant launch of every
# workload) is compiled from; its traffic figure stays valid while they do
ATTN_SOURCES = ("sfm_attn_tc.cu", "sfm_tc.cuh", "sfm_internal.cuh")


def kernel_source_hash():
    h = hashlib.sha256()
    for f in ATTN_SOURCES:
        h.update(open(os.path.join(ROOT, "sparse_shared_kv_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def load_traffic(workload):
    """DRAM bytes per launch of the dominant kernel from a committed ncu summary,
    only while the kernel sources still hash to the captured version."""
    path = os.path.join(ROOT, "profiles", f"traffic_{workload}.json")
    try:
        d = json.load(open(path))
    except (OSError, ValueError):
        return None
    if d.get("source_hash") != kernel_source_hash():
        return None
    return d.get("dram_bytes_per_launch")


def measured_peaks():
    try:
        d = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d["bf16_tflops_sustained"]), "of measured"
    except (OSError, ValueError, KeyError):
        return 6800.0, 1900.0, 1700.0, "of fallback"


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def make_sets(args, workload, sfm, dev, rank, nsets):
    """Seeded input sets of a workload (enough that their attended bytes
    exceed 3x L2 when nsets is 0), their accounting and per-set buffers."""
    sets = [make_problem(workload, dev, 1000 + 97 * rank, args.batch, args.compact_pool)]
    acc = [accounting(sets[0], sfm)]
    if nsets <= 0:
        l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        nsets = max(2, min(16, -(-3 * l2 // max(1, acc[0]["bytes"]))))
    for i in range(1, nsets):
        sets.append(make_problem(workload, dev, 1000 + 97 * rank + i, args.batch, args.compact_pool))
        acc.append(accounting(sets[-1], sfm))
    runners = []
    policy = sfm.SPLIT_OCCUPANCY if args.split_policy == "occupancy" else sfm.SPLIT_BATCH_INVARIANT
    for p in sets:
        params = sfm.make_params(**p.attrs(), split_policy=policy)
        tens = sfm.make_tensors(p.t["q"], p.t["ori_kv"], **p.tensor_kwargs())
        md = torch.empty(sfm.sfm_metadata_size(params), dtype=torch.int32, device=dev)
        nb = sfm.sfm_workspace_size(params)
        ws = torch.empty(nb, dtype=torch.uint8, device=dev) if nb else None
        out = torch.empty(p.t["q"].shape[:-1] + (512,), dtype=p.torch_dtype, device=dev)
        lse = torch.empty(p.num_tokens * p.num_heads_q, dtype=torch.float32, device=dev)
        runners.append((p, params, tens, md, ws, out, lse))
    return sets, acc, runners


def measure(args, workload, sfm, dev, rank, world, sampler, nsets):
    """Device-timed steps (planner + forward) of one workload, the attention
    kernel's own time in a second leg of steps, and sfm_forward alone on plans
    made beforehand.  Returns the numbers and the sets (for the e2e leg)."""
    sets, acc, runners = make_sets(args, workload, sfm, dev, rank, nsets)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()

    def step(k):
        p, params, tens, md, ws, out, lse = runners[k % len(runners)]
        sfm.sfm_metadata(params, tens, md, stream)
        sfm.sfm_forward(params, tens, md, p.softmax_scale, out, lse, ws, status, stream)

    W = max(args.warmup, 3)
    t_warm = sampler.mark()
    for k in range(W):
        step(k)
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError(f"{workload}: device status {int(status.item()):#x} during warm-up")
    # work units of the first set's plan: splits (header word 6) x head groups
    units = int(runners[0][3][6].item()) * ((sets[0].num_heads_q + 63) // 64)

    # kernels per step: the planner, the attention kernel and, when a row can
    # have more than one split (a split-KV workspace is needed), the combine
    launches_per_step = 3 if sfm.sfm_workspace_size(runners[0][1]) > 0 else 2
    K = args.steps
    # the headline steps run exactly as a caller's would, with no events
    # between the kernels
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    t_in = sampler.mark()
    e0.record(stream)
    for k in range(K):
        step(k)
    e1.record(stream)
    torch.cuda.synchronize()
    t_out = sampler.mark()
    barrier(world)
    ms_total = e0.elapsed_time(e1)

    # the attention kernel's own time: a second leg of the same steps with the
    # kernel of every other step bracketed by events on its stream.  An event
    # record between two kernels ends their programmatic overlap, so these
    # steps run slower (their time is reported beside the headline, not as it)
    prof_every = 2
    prof_steps = list(range(0, K, prof_every))
    kb = {k: torch.cuda.Event(enable_timing=True) for k in prof_steps}
    ke = {k: torch.cuda.Event(enable_timing=True) for k in prof_steps}
    p0_, p1_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    p0_.record(stream)
    for k in range(K):
        if k in kb:
            sfm.sfm_set_profile_events(kb[k], ke[k])
            step(k)
            sfm.sfm_set_profile_events(None, None)
        else:
            step(k)
    p1_.record(stream)
    torch.cuda.synchronize()
    prof_leg_ms = max_over_ranks(p0_.elapsed_time(p1_), world, dev)
    kernel_ms = [kb[k].elapsed_time(ke[k]) for k in prof_steps]

    # the plan depends on the lengths only, so a model reuses one plan across
    # its layers: time sfm_forward alone on the plans of the sets as well
    # (reported beside the step, not in place of it)
    for k in range(len(runners)):
        p, params, tens, md, ws, out, lse = runners[k]
        sfm.sfm_metadata(params, tens, md, stream)
    for k in range(W):
        p, params, tens, md, ws, out, lse = runners[k % len(runners)]
        sfm.sfm_forward(params, tens, md, p.softmax_scale, out, lse, ws, status, stream)
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    f0.record(stream)
    for k in range(K):
        p, params, tens, md, ws, out, lse = runners[k % len(runners)]
        sfm.sfm_forward(params, tens, md, p.softmax_scale, out, lse, ws, status, stream)
    f1.record(stream)
    torch.cuda.synchronize()
    fwd_ms = max_over_ranks(f0.elapsed_time(f1), world, dev)

    # the same forwards captured as one CUDA graph of back-to-back calls
    # (rotating over the sets), replayed: launch cost off the host
    KG = min(K, 100)
    graph = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream(device=dev)
    cap.wait_stream(stream)
    with torch.cuda.stream(cap):
        with torch.cuda.graph(graph, stream=cap):
            cs = torch.cuda.current_stream()
            for k in range(KG):
                p, params, tens, md, ws, out, lse = runners[k % len(runners)]
                sfm.sfm_forward(params, tens, md, p.softmax_scale, out, lse, ws, status, cs)
    stream.wait_stream(cap)
    graph.replay()
    torch.cuda.synchronize()
    reps = max(1, K // KG)
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    g0.record(stream)
    for _ in range(reps):
        graph.replay()
    g1.record(stream)
    torch.cuda.synchronize()
    graph_ms = max_over_ranks(g0.elapsed_time(g1), world, dev) / (reps * KG)
    del graph

    # L2-warm, labelled: one input set's forward repeated (its KV stays in L2)
    p, params, tens, md, ws, out, lse = runners[0]
    for _ in range(W):
        sfm.sfm_forward(params, tens, md, p.softmax_scale, out, lse, ws, status, stream)
    torch.cuda.synchronize()
    w0, w1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    w0.record(stream)
    for _ in range(K):
        sfm.sfm_forward(params, tens, md, p.softmax_scale, out, lse, ws, status, stream)
    w1.record(stream)
    torch.cuda.synchronize()
    warm_ms = max_over_ranks(w0.elapsed_time(w1), world, dev) / K

    # the planner alone (sfm_metadata back to back over the sets)
    m0, m1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    m0.record(stream)
    for k in range(K):
        p, params, tens, md, ws, out, lse = runners[k % len(runners)]
        sfm.sfm_metadata(params, tens, md, stream)
    m1.record(stream)
    torch.cuda.synchronize()
    plan_ms = max_over_ranks(m0.elapsed_time(m1), world, dev) / K

    # independent steps (different input sets: their own plans, workspaces and
    # outputs) dealt round robin over several streams: the kernels of
    # different steps run concurrently and fill each other's latency gaps, as
    # independent batches served side by side would; a set's next step waits
    # for its previous one (an event), whichever stream that ran on
    ns = max(1, min(args.streams, len(runners)))
    cstreams = [torch.cuda.Stream(device=dev) for _ in range(ns)]
    # one event per set, re-recorded each step (a wait takes the event as it
    # stands when the wait is enqueued)
    done = [torch.cuda.Event() for _ in runners]
    used = [False] * len(runners)

    def cstep(k):
        i = k % len(runners)
        p, params, tens, md, ws, out, lse = runners[i]
        cs = cstreams[k % ns]
        if used[i]:
            cs.wait_event(done[i])
        sfm.sfm_metadata(params, tens, md, cs)
        sfm.sfm_forward(params, tens, md, p.softmax_scale, out, lse, ws, status, cs)
        done[i].record(cs)
        used[i] = True

    for s_ in cstreams:
        s_.wait_stream(stream)
    for k in range(W):
        cstep(k)
    for s_ in cstreams:
        stream.wait_stream(s_)
    torch.cuda.synchronize()
    c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    c0.record(stream)
    for s_ in cstreams:
        s_.wait_stream(stream)
    for k in range(K):
        cstep(k)
    for s_ in cstreams:
        stream.wait_stream(s_)
    c1.record(stream)
    torch.cuda.synchronize()
    t_legs = sampler.mark()
    conc_ms = max_over_ranks(c0.elapsed_time(c1), world, dev)
    if int(status.item()) != 0:
        raise RuntimeError(f"{workload}: device status {int(status.item()):#x} during the timed steps")

    ms_max = max_over_ranks(ms_total, world, dev)
    rows_total = sum_over_ranks(sum(acc[k % len(acc)]["attended_rows"] for k in range(K)), world, dev)
    flops_total = sum_over_ranks(sum(acc[k % len(acc)]["flops"] for k in range(K)), world, dev)

    hbm_peak, tc_peak, tc_peak_sustained, peak_note = measured_peaks()
    bytes_launch = statistics.mean(acc[k % len(acc)]["bytes"] for k in prof_steps)
    flops_launch = statistics.mean(acc[k % len(acc)]["flops"] for k in prof_steps)
    kavg = statistics.mean(kernel_ms)
    achieved_gbs = bytes_launch / (kavg * 1e-3) / 1e9
    achieved_tf = flops_launch / (kavg * 1e-3) / 1e12
    traffic = load_traffic(workload) if args.batch is None else None
    # the bound is whichever roofline time is longer for this workload: HBM
    # bytes at the measured copy bandwidth or FLOPs at the measured dense
    # 16-bit tensor rate (burst for a short step, sustained for a long one);
    # fp16 and bf16 products run at the same rate
    tc_ref = tc_peak if ms_max / K < 1.0 else tc_peak_sustained
    if flops_launch / (tc_ref * 1e12) > bytes_launch / (hbm_peak * 1e9):
        roof = {"bound": "tensor", "achieved": achieved_tf, "peak": tc_ref, "unit": "TFLOP/s",
                "frac": achieved_tf / tc_ref}
    else:
        roof = {"bound": "hbm", "achieved": achieved_gbs, "peak": hbm_peak, "unit": "GB/s",
                "frac": achieved_gbs / hbm_peak}
    roof.update({
        "traffic": traffic, "peak_note": peak_note,
        "kernel": "sfm_attn_tc_kernel (main attention kernel)", "kernel_ms_avg": kavg,
        "kernel_timed_steps": len(prof_steps),
        "kernel_timing": f"CUDA events on the launching stream around the attention kernel of every other "
                         f"step of a second leg of {K} steps (the headline steps carry no events)",
        "profiled_leg_ms_per_step": prof_leg_ms / K,
        "algorithmic_bytes_per_launch": bytes_launch, "algorithmic_flops_per_launch": flops_launch,
        "tensor_tflops": achieved_tf, "tensor_frac_of_bf16_peak": achieved_tf / tc_peak,
        "hbm_gbs": achieved_gbs, "hbm_frac": achieved_gbs / hbm_peak,
    })
    if traffic:
        roof["traffic_over_algorithmic"] = traffic / bytes_launch
    if roof["bound"] == "hbm":
        # the stricter of the two denominators is the measured copy rate; the
        # nominal HBM3e rate, for reference
        roof["frac_of_nominal"] = achieved_gbs / NOMINAL_HBM_GBS
        roof["nominal_peak"] = NOMINAL_HBM_GBS
    p0 = sets[0]
    config = {
        "workload": workload, "batch": p0.batch_size, "q_n": p0.num_heads_q, "d": 512,
        "d_qk": p0.d_qk, "cmp_topk": p0.cmp_topk, "ori_topk": p0.ori_topk, "cmp_ratio": p0.cmp_ratio,
        "window": p0.ori_win_left + p0.ori_win_right + 1 if p0.ori_topk == 0 else 0,
        "layout": f"{p0.layout_q}/{p0.layout_kv}",
        "attended_rows_per_step": statistics.mean(a["attended_rows"] for a in acc),
        "l2": f"inputs larger than L2: {len(sets)} rotating input sets "
              f"({len(sets) * bytes_launch / 1e6:.0f} MB of attended bytes)",
        "step": "sfm_metadata (device planner) + sfm_forward (attention"
                + (" + split combine)" if launches_per_step == 3 else "; one split per row, no combine)"),
        "parallelism": f"replicas x{world}",
        "split_policy": args.split_policy, "work_units": units,
    }
    fwd_launches = launches_per_step - 1
    res = {
        "workload": workload, "K": K, "W": W, "ms_max": ms_max, "rows_total": rows_total,
        "flops_total": flops_total, "fwd_ms": fwd_ms, "roofline": roof, "config": config,
        "graph_fwd_ms": graph_ms, "l2_warm_fwd_ms": warm_ms, "planner_ms": plan_ms,
        "concurrent_ms": conc_ms, "concurrent_streams": ns,
        "rows_per_step": rows_total / K,
        # every launch of every timed leg: steps, forwards, graph replays, L2-warm forwards, planner calls,
        # concurrent steps
        "timed_launches": 2 * launches_per_step * K + fwd_launches * K + fwd_launches * KG * reps
                          + fwd_launches * K + K + launches_per_step * K,
        "launches_per_step": launches_per_step, "clocks": sampler.summary(t_in, t_out, t_legs, t_warm),
        "dtype": {"int8_packed": "fp16 (int8 KV dequantized)", "fp8_packed": "fp16 (fp8 e4m3 KV dequantized)"}
                 .get(p0.kv_format, "bf16"),
    }
    return res, sets, acc


def run_ours(args):
    rank, world, local = dist_init("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import sparse_shared_kv_gb300 as sfm
    sfm.build()
    sfm.lib()

    gpu_uuid = str(torch.cuda.get_device_properties(dev).uuid)
    sampler = ClockSampler(gpu_uuid if gpu_uuid.startswith("GPU-") else f"GPU-{gpu_uuid}")
    sampler.start()
    head, sets, acc = measure(args, args.workload, sfm, dev, rank, world, sampler, args.sets)
    K = head["K"]
    stream = torch.cuda.current_stream()
    # end to end through the public two-call API, inputs from pinned host memory
    e2e = run_e2e(args, sfm, sets, acc, dev, stream)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(args, sets[0], acc[0])
    del sets, acc
    torch.cuda.empty_cache()
    # the second configuration the >= 70 % roofline target names (HCA decode),
    # measured in the same run when the headline is CSA decode
    second = None
    if args.workload == "csa_decode" and not args.no_second:
        second, s2, _ = measure(args, "hca_decode", sfm, dev, rank, world, sampler, 0)
        del s2
        torch.cuda.empty_cache()
    # small decode batches under both split policies (compact pools: the same
    # attended rows, a small footprint)
    small = None
    if args.workload == "csa_decode" and args.batch is None and not args.no_small_batch:
        small = {}
        for wl in ("csa_decode", "hca_decode"):
            for B in (4, 8, 16):
                for pol in ("invariant", "occupancy"):
                    a = argparse.Namespace(**vars(args))
                    a.batch, a.compact_pool, a.split_policy, a.sets = B, True, pol, 0
                    a.steps, a.warmup = min(args.steps, 100), max(3, min(args.warmup, 10))
                    r, s3, _ = measure(a, wl, sfm, dev, rank, world, sampler, 0)
                    del s3
                    small.setdefault(wl, {}).setdefault(str(B), {})[pol] = {
                        "ms_per_step": r["ms_max"] / r["K"], "kernel_ms": r["roofline"]["kernel_ms_avg"],
                        "forward_only_ms_per_step": r["fwd_ms"] / r["K"], "work_units": r["config"]["work_units"],
                        "value": r["rows_total"] / (r["ms_max"] * 1e-3), "steps": r["K"],
                        "launches": r["timed_launches"], "clocks_sm_mhz": r["clocks"].get("sm_mhz"),
                    }
        torch.cuda.empty_cache()
    sampler.stop()

    ms_max = head["ms_max"]
    value = head["rows_total"] / (ms_max * 1e-3)
    e2e_ms = max_over_ranks(e2e["ms_total"], world, dev)
    e2e_rows = sum_over_ranks(e2e["rows"], world, dev)
    fwd_ms = head["fwd_ms"]

    if rank == 0:
        line = {
            "metric": f"attended KV tokens/s ({args.workload.replace('_', ' ')}, 1 GB300 per rank)",
            "value": value,
            "unit": "tokens/s",
            "n_gpus": world,
            "steps": K,
            "warmup": head["W"],
            "ms_per_step": ms_max / K,
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": head["dtype"],
            "data": "synthetic (seeded generators, shapes and distributions of the pages' workloads)",
            "config": head["config"],
            "tflops": head["flops_total"] / (ms_max * 1e-3) / 1e12,
            "roofline": head["roofline"],
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_rows / (e2e_ms * 1e-3), "unit": "tokens/s",
                    "h2d_bytes_per_step": e2e["h2d"], "d2h_bytes_per_step": e2e["d2h"],
                    "ms_per_step": e2e_ms / e2e["steps"], "mode": e2e["mode"]},
            "forward_only": {"value": head["rows_total"] / (fwd_ms * 1e-3), "unit": "tokens/s",
                             "ms_per_step": fwd_ms / K,
                             "note": "sfm_forward alone (attention and, when rows have several splits, the "
                                     "combine) on plans made beforehand, "
                                     "as a model reuses one plan across its layers",
                             "cuda_graph": {"value": head["rows_per_step"] / (head["graph_fwd_ms"] * 1e-3),
                                            "unit": "tokens/s", "ms_per_forward": head["graph_fwd_ms"],
                                            "note": "the same forwards captured as one CUDA graph of back-to-back "
                                                    "calls over the rotating sets, replayed"},
                             "l2_warm": {"value": head["rows_per_step"] / (head["l2_warm_fwd_ms"] * 1e-3),
                                         "unit": "tokens/s", "ms_per_forward": head["l2_warm_fwd_ms"],
                                         "note": "L2-warm: one input set's forward repeated, its KV rows left in "
                                                 "L2 (not the headline)"}},
            "planner_only": {"ms_per_call": head["planner_ms"],
                             "note": "sfm_metadata (the device planner) alone, back to back over the sets"},
            "concurrent_steps": {"value": head["rows_total"] / (head["concurrent_ms"] * 1e-3), "unit": "tokens/s",
                                 "ms_per_step": head["concurrent_ms"] / K, "streams": head["concurrent_streams"],
                                 "note": "the same steps (planner + forward, inputs resident) with consecutive "
                                         "independent input sets spread over several streams, so kernels of "
                                         "different steps run concurrently; the headline value runs them back to "
                                         "back on one stream"},
            "gpu_launches": head["timed_launches"] + head["launches_per_step"] * e2e["steps"]
                            + (second["timed_launches"] if second else 0)
                            + (sum(v["launches"] for w in small.values() for b in w.values() for v in b.values())
                               if small else 0),
            "gpu_launches_note": "launches of this library's kernels in every timed leg of this line (steps, "
                                 "kernel-profiled steps, forward-only, graph replays, L2-warm forwards, planner "
                                 "calls, concurrent steps, end-to-end steps; HCA and small-batch blocks included)",
            "clocks": head["clocks"],
        }
        if second:
            line["hca_decode"] = {
                "value": second["rows_total"] / (second["ms_max"] * 1e-3), "unit": "tokens/s",
                "ms_per_step": second["ms_max"] / second["K"], "steps": second["K"],
                "tflops": second["flops_total"] / (second["ms_max"] * 1e-3) / 1e12,
                "forward_only_ms_per_step": second["fwd_ms"] / second["K"],
                "graph_ms_per_forward": second["graph_fwd_ms"], "l2_warm_ms_per_forward": second["l2_warm_fwd_ms"],
                "planner_ms_per_call": second["planner_ms"],
                "concurrent_ms_per_step": second["concurrent_ms"] / second["K"],
                "concurrent_streams": second["concurrent_streams"],
                "roofline": second["roofline"], "config": second["config"], "clocks": second["clocks"],
                "note": "the second configuration of the >= 70 % roofline target, timed in the same run "
                        "after the headline (its launches are counted in gpu_launches)",
            }
        if small:
            line["small_batch"] = {
                **small,
                "unit": "tokens/s", "n_gpus_per_rank": 1,
                "note": "decode batches of 4, 8 and 16 rows, timed like the headline (planner + forward per "
                        "step) under the batch-invariant split policy (the default) and the occupancy policy; "
                        "launches counted in gpu_launches",
            }
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_e2e(args, sfm, sets, acc, dev, stream):
    """Public API end to end, every step: one host->device copy of the step's
    inputs (all of them packed in one pinned buffer), sparse_flash_mla_metadata,
    sparse_flash_mla, one device->host copy of O and LSE.  Each input set's step
    is captured once as a CUDA graph of exactly those calls (as a decode loop
    would), and consecutive steps (independent batches) are replayed on several
    streams (--streams), so one step's copies overlap other steps' kernels and
    kernels of different steps run concurrently."""
    names = ("q", "cmp_sparse_indices", "ori_sparse_indices", "ori_block_table", "cmp_block_table",
             "seqused_ori_kv", "seqused_cmp_kv", "cmp_residual_kv", "sinks")

    def api_step(p, T, out, lse, st):
        md = sfm.sparse_flash_mla_metadata(
            p.num_heads_q, 1, 512, cu_seqlens_q=T["cu_seqlens_q"], cu_seqlens_ori_kv=T["cu_seqlens_ori_kv"],
            cu_seqlens_cmp_kv=T["cu_seqlens_cmp_kv"], seqused_ori_kv=T["seqused_ori_kv"],
            seqused_cmp_kv=T["seqused_cmp_kv"], cmp_residual_kv=T["cmp_residual_kv"], batch_size=p.batch_size,
            max_seqlen_q=p.max_seqlen_q, total_q=p.total_q, max_seqlen_ori_kv=p.max_seqlen_ori_kv,
            max_seqlen_cmp_kv=p.max_seqlen_cmp_kv, ori_topk=p.ori_topk, cmp_topk=p.cmp_topk,
            cmp_ratio=p.cmp_ratio, ori_mask_mode=p.ori_mask_mode, cmp_mask_mode=p.cmp_mask_mode,
            ori_win_left=p.ori_win_left, ori_win_right=p.ori_win_right, layout_q=p.layout_q,
            layout_kv=p.layout_kv, has_cmp_kv=p.has_cmp_kv, dtype=p.torch_dtype,
            kv_format=S_KV_FORMAT_CODES[p.kv_format], rope_head_dim=p.rope_head_dim,
            ori_block_size=p.ori_block_size, cmp_block_size=p.cmp_block_size, return_softmax_lse=True,
            batch_invariant=args.split_policy == "invariant", device=dev, stream=st)
        sfm.sparse_flash_mla(
            T["q"], metadata=md, ori_kv=T["ori_kv"], cmp_kv=T["cmp_kv"], ori_sparse_indices=T["ori_sparse_indices"],
            cmp_sparse_indices=T["cmp_sparse_indices"], ori_block_table=T["ori_block_table"],
            cmp_block_table=T["cmp_block_table"], cu_seqlens_q=T["cu_seqlens_q"],
            cu_seqlens_ori_kv=T["cu_seqlens_ori_kv"], cu_seqlens_cmp_kv=T["cu_seqlens_cmp_kv"],
            seqused_ori_kv=T["seqused_ori_kv"], seqused_cmp_kv=T["seqused_cmp_kv"],
            cmp_residual_kv=T["cmp_residual_kv"], sinks=T["sinks"], softmax_scale=p.softmax_scale,
            ori_row_stride=p.ori_row_stride, cmp_row_stride=p.cmp_row_stride or None, out=out, lse=lse,
            stream=st)

    legs, keep = [], []          # the graphs, and every buffer their nodes point at
    h2d = d2h = 0
    for i, p in enumerate(sets):
        parts = [(n, p.t[n]) for n in names if p.t[n] is not None]
        off, lay = 0, []
        for n, x in parts:
            nb = x.numel() * x.element_size()
            lay.append((n, off, nb, x))
            off += (nb + 255) // 256 * 256
        hbuf = torch.empty(off, dtype=torch.uint8).pin_memory()
        dbuf = torch.empty(off, dtype=torch.uint8, device=dev)
        T = dict(p.t)
        for n, o, nb, x in lay:
            hbuf[o:o + nb].copy_(x.reshape(-1).view(torch.uint8).cpu())
            T[n] = dbuf[o:o + nb].view(x.dtype).view(x.shape)
        on = p.num_tokens * p.num_heads_q * 512 * p.t["q"].element_size()
        ln = p.num_tokens * p.num_heads_q * 4
        obuf = torch.empty(on + ln, dtype=torch.uint8, device=dev)
        ohost = torch.empty(on + ln, dtype=torch.uint8).pin_memory()
        out = obuf[:on].view(p.torch_dtype).view(p.t["q"].shape[:-1] + (512,))
        lse = obuf[on:].view(torch.float32)
        if i == 0:
            h2d = sum(nb for _, _, nb, _ in lay)
            d2h = on + ln
        side = torch.cuda.Stream(device=dev)
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for _ in range(2):                      # allocator warm-up before capture
                dbuf.copy_(hbuf, non_blocking=True)
                api_step(p, T, out, lse, side)
                ohost.copy_(obuf, non_blocking=True)
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            st = torch.cuda.current_stream()
            dbuf.copy_(hbuf, non_blocking=True)
            api_step(p, T, out, lse, st)
            ohost.copy_(obuf, non_blocking=True)
        legs.append(g)
        keep.append((hbuf, dbuf, obuf, ohost, T, out, lse))
    torch.cuda.synchronize()
    ns = max(1, min(args.streams, len(legs)))
    streams = [torch.cuda.Stream(device=dev) for _ in range(ns)]
    done = [torch.cuda.Event() for _ in legs]       # one per set, re-recorded each step
    used = [False] * len(legs)

    def step(k):
        # steps dealt round robin over the streams; a set's graph replays only
        # after its previous replay (its buffers are reused), on whichever stream
        i = k % len(legs)
        st = streams[k % ns]
        if used[i]:
            st.wait_event(done[i])
        with torch.cuda.stream(st):
            legs[i].replay()
        done[i].record(st)
        used[i] = True

    for k in range(max(3, 2 * len(legs))):
        step(k)
    torch.cuda.synchronize()
    K = max(1, min(args.steps, 200))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    cur = torch.cuda.current_stream()
    e0.record(cur)
    for s_ in streams:
        s_.wait_stream(cur)
    for k in range(K):
        step(k)
    for s_ in streams:
        cur.wait_stream(s_)
    e1.record(cur)
    torch.cuda.synchronize()
    rows = sum(acc[k % len(acc)]["attended_rows"] for k in range(K))
    return {"ms_total": e0.elapsed_time(e1), "steps": K, "rows": rows, "h2d": h2d, "d2h": d2h,
            "mode": "per step: one H2D copy of all inputs from pinned memory, the public two-call API, one D2H "
                    "copy of O and LSE; each input set's step captured once as a CUDA graph, consecutive "
                    "(independent) steps replayed on %d streams" % ns}


# ---------------------------------------------------------------------------
# CPU oracle legs
# ---------------------------------------------------------------------------
def _oracle_rate(prob, host, bound, threads, seconds, chunk):
    """Attended rows per second of the oracle on `threads` host threads over
    consecutive chunks of query rows (wrapping around) for about `seconds`."""
    import oracle
    T = host.num_tokens
    t0 = time.time()
    rows = done = 0
    while True:
        toks = [(done + j) % T for j in range(chunk)]
        oracle.forward(host, toks, nthreads=threads)
        rows += sum(len(oracle.attended(host, t, bound)[0]) for t in toks)
        done += chunk
        if time.time() - t0 >= seconds:
            break
    dt = time.time() - t0
    return rows / dt, done, dt


def cpu_baseline(args, prob, acc, seconds=None):
    """The oracle on the host cores over a bounded sample of the workload:
    consecutive chunks of query rows until the time budget is spent, on all
    cores, then on one core; throughput = attended rows of the rows done /
    time."""
    import oracle
    host = prob.to("cpu")
    cores = os.cpu_count() or 1
    seconds = args.cpu_seconds if seconds is None else seconds
    b = oracle._Bound(host)
    T = host.num_tokens
    chunk = max(1, min(T, 4 * cores))
    v_all, done, dt = _oracle_rate(prob, host, b, cores, seconds, chunk)
    v_one, done1, dt1 = _oracle_rate(prob, host, b, 1, seconds / 2, 1)
    return {"value": v_all, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{done} query rows ({done / T:.2f} passes over the {T} rows of one input set, in chunks "
                      f"of {chunk}), {dt:.1f} s, fp64 C oracle with OpenMP",
            "single_core": {"value": v_one, "unit": "tokens/s", "cores": 1,
                            "sample": f"{done1} query rows, {dt1:.1f} s, one thread"}}


def run_reference(args):
    rank, world, local = dist_init("gloo")
    if rank != 0:
        return
    import oracle
    import sfm_inputs as S
    oracle.build()
    prob = S.WORKLOADS[args.workload](device="cpu", seed=1000)
    cores = os.cpu_count() or 1
    # attended rows per query row, from the oracle's own attended sets
    b = oracle._Bound(prob)
    counts = [len(oracle.attended(prob, t, b)[0]) for t in range(prob.num_tokens)]
    per_step = 2                                   # query rows per step: keeps the run to minutes
    W = max(args.warmup, 3)
    K = args.steps

    def step(k):
        toks = [(k * per_step + j) % prob.num_tokens for j in range(per_step)]
        oracle.forward(prob, toks, nthreads=cores)
        return sum(counts[t] for t in toks)

    for k in range(W):
        step(k)
    t0 = time.perf_counter()
    rows = 0
    for k in range(K):
        rows += step(k)
    dt = time.perf_counter() - t0
    value = rows / dt
    line = {
        "impl": "reference",
        "metric": f"attended KV tokens/s ({args.workload.replace('_', ' ')}, 1 GB300 per rank)",
        "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": dt * 1e3 / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic (seeded generators, shapes and distributions of the pages' workloads)",
        "config": {"workload": args.workload, "batch": prob.batch_size, "q_n": prob.num_heads_q,
                   "sample_per_step": f"{per_step} query rows of the batch"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"{per_step} query rows per step (of {prob.num_tokens}), {K} steps"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
        return
    run_ours(args)


if __name__ == "__main__":
    main()
