"""Benchmark of the paged-decode hot path on GB300.

One step = one decode step of the Llama-3-8B-shaped batch-64 workload (h_q 32,
h_kv 8, D 128, bf16, contexts log-uniform in [512, 8192]): append every
sequence's new K/V through the slot mapping, then paged decode attention
(split-K + log-sum-exp combine).  Step t of the timed loop uses the inputs of
workload step t mod 32, so contexts grow by one token per step as in decoding.

Printed JSON (rank 0): value = effective HBM GB/s of the whole step
(algorithmic bytes of append + attention / device time), with the attention
call's own roofline, an end-to-end figure through the public API with host
buffers, the CPU oracle as a baseline, and SM clocks sampled while the GPU
was busy.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged decode attn: effective HBM GB/s (% of GB300 peak), decode tokens/s"
WORKLOAD = "llama3_8b_decode"
WORKLOAD_DESC = ("Llama-3-8B-shaped paged decode: batch 64, h_q 32, h_kv 8, d_head 128, bf16, block 16, "
                 "contexts log-uniform in [512, 8192], randomly permuted pool (1.25x need), 32 decode steps "
                 "each appending one token per sequence")
FALLBACK_HBM_GBS = 6800.0
KERNEL_SOURCES = ["paged_kv_decode_27_gb300/csrc/decode_tc.cu", "paged_kv_decode_27_gb300/csrc/decode_merge.cuh",
                  "paged_kv_decode_27_gb300/csrc/pa_common.cuh"]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "decode_traffic.json")


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=64)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--partition", type=int, default=0)
    p.add_argument("--workload", default=WORKLOAD,
                   help="llama3_8b_decode (the headline line) or one of tiny_fp32, llama32_1b_decode, "
                        "prefix_shared_8k, mixed_mistral7b, llama32_1b_decode_int8, llama3_8b_decode_int8, "
                        "llama3_8b_verify, llama3_8b_verify_int8, llama3_8b_decode_rope (per-call figures for that "
                        "workload), or "
                        "llama3_8b_prefix_serving (decode steps driven by the block manager)")
    p.add_argument("--quick", action="store_true",
                   help="no CPU baseline, no 1 s pre-warm, no end-to-end pass (for profiler runs)")
    return p.parse_args()


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------

def max_over_ranks(x: float, device, world: int) -> float:
    """The largest value of x over all ranks: the slowest replica's time."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_gbs(bytes_per_rank: float, seconds: float, world: int) -> float:
    """Whole-job GB/s of `world` weak-scaling replicas: every rank moves the
    same bytes, and the job ends with the slowest one."""
    return world * bytes_per_rank / seconds / 1e9


def peak_hbm():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_sha() -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def measured_traffic(units_ratio: float):
    """DRAM bytes per attention call from the committed ncu summary, scaled
    from its captured case to this one by the K/V bytes processed; None when
    the kernel sources changed since the capture."""
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f)
    except Exception:
        return None
    if rec.get("kernel_sha") != kernel_sha():
        return None
    return float(rec["dram_bytes_per_call"]) * units_ratio if rec.get("scale_with_kv") else \
        float(rec["dram_bytes_per_call"])


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(self.gpu)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=2)

    def summary(self, t0, t1):
        win = [p for t, p in self.samples if t0 <= t <= t1] or [p for _, p in self.samples]
        if not win:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        sm = [float(p[1]) for p in win if p[1].replace(".", "").isdigit()]
        mx = [float(p[2]) for p in win if p[2].replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for p in win:
            for name, v in zip(names, p[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(win)}


def cpu_baseline(max_seconds: float = 10.0):
    """Time the float64 CPU oracle on a bounded sample of the workload: whole
    decode steps (all 64 sequences, all heads) in order, each after its append,
    until max_seconds of decode time; in a fresh 1-thread process."""
    code = r"""
import json, os, sys, time
sys.path.insert(0, %r)
import torch
torch.set_num_threads(1)
import oracle
from paged_kv_decode_27_gb300 import workloads as W
wl = W.%s()
def npv(t):
    t = t.contiguous()
    return t.view(torch.int16).numpy().view('uint16') if t.dtype == torch.bfloat16 else t.numpy()
kp, vp = npv(wl.k_pool), npv(wl.v_pool)
bt = wl.decode_block_tables.contiguous().numpy()
el = 0.0; b = 0; tok = 0; steps = 0
e = 2; hkv, d, hq = wl.num_kv_heads, wl.head_dim, wl.num_q_heads
for t in range(wl.steps):
    st = wl.step(t)
    kp, vp = oracle.append_ref(kp, vp, st.slot_mapping.numpy(), npv(st.k_new), npv(st.v_new))
    ctx = st.context_lens.numpy()
    t0 = time.perf_counter()
    oracle.decode_ref(npv(st.q), kp, vp, bt, ctx, wl.scale)
    el += time.perf_counter() - t0
    b += sum(int(c) * 2 * hkv * d * e + 2 * hq * d * e + 4 * ((int(c) + 15) // 16) + 4 for c in ctx)
    tok += int(ctx.sum()); steps += 1
    if el > %f: break
print(json.dumps({"seconds": el, "steps": steps, "bytes": b, "tokens": tok}))
""" % (ROOT, WORKLOAD, max_seconds)
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env, timeout=900)
    if r.returncode != 0:
        tail = r.stderr.strip().splitlines()[-1] if r.stderr.strip() else "no output"
        return {"value": None, "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": "failed: " + tail}
    rec = json.loads(r.stdout.strip().splitlines()[-1])
    return {"value": rec["bytes"] / rec["seconds"] / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"float64 numpy oracle on {WORKLOAD}: decode steps 0..{rec['steps'] - 1} in full "
                      f"(64 sequences x 32 q heads each, {rec['tokens']} context tokens in total), "
                      f"{rec['seconds']:.2f} s of decode time, 1 thread; appends untimed",
            "seconds": rec["seconds"]}


def cpu_oracle_more(max_seconds: float = 6.0):
    """The float64 oracle on the host cores, beyond the 1-thread headline
    figure: (1) the same headline decode steps spread over every core the
    process may use (one single-threaded worker process per core, each taking
    whole sequences), wall clock; (2) one decode step of every benchmark
    configuration on one thread (the mixed step's prompt pass on its
    512-token prompt only).  Runs in a fresh process with no GPU."""
    code = r"""
import json, os, sys, time
sys.path.insert(0, %r)
import numpy as np
import torch
torch.set_num_threads(1)
import multiprocessing as mp
import oracle
from paged_kv_decode_27_gb300 import workloads as W
def npv(t):
    t = t.contiguous()
    return t.view(torch.int16).numpy().view('uint16') if t.dtype == torch.bfloat16 else t.numpy()
cores = len(os.sched_getaffinity(0))
res = {"cores": cores}
# (1) headline steps 0..n-1 on all cores: the pool after the appends of steps 0..n-1 serves
# every one of those steps (a step reads only positions below its own contexts)
wl = W.llama3_8b_decode()
kp, vp = npv(wl.k_pool), npv(wl.v_pool)
n = 4
sts = [wl.step(t) for t in range(n)]
for st in sts:
    kp, vp = oracle.append_ref(kp, vp, st.slot_mapping.numpy(), npv(st.k_new), npv(st.v_new))
bt = wl.decode_block_tables.contiguous().numpy()
QS = [npv(st.q) for st in sts]
CT = [st.context_lens.numpy() for st in sts]
jobs = [(t, s) for t in range(n) for s in range(64)]
def work(part):
    for t, s in part:
        oracle.decode_ref(QS[t], kp, vp, bt, CT[t], wl.scale, seqs=[s])
    return len(part)
# workers are forked here, in a process that never touched a GPU
ctx = mp.get_context("fork")
parts = [jobs[i::cores] for i in range(cores)]
with ctx.Pool(cores) as pool:
    pool.map(work, [parts[0][:1]] * cores)      # start-up, untimed
    t0 = time.perf_counter()
    pool.map(work, parts)
    el = time.perf_counter() - t0
b = sum(int(c) * 2 * 8 * 128 * 2 + 2 * 32 * 128 * 2 + 4 * ((int(c) + 15) // 16) + 4 for ct in CT for c in ct)
res["all_cores"] = {"value": b / el / 1e9, "unit": "GB/s", "cores": cores, "seconds": el,
                    "sample": f"decode steps 0..{n-1} of llama3_8b_decode in full (64 sequences x 32 q heads), "
                              f"one single-threaded worker process per core, whole sequences per task"}
# (2) one step of every configuration, one thread
per = {}
for name in %r:
    w = wl if name == wl.name else W.WORKLOADS[name]()
    st = w.step(0)
    k2, v2 = oracle.append_ref(npv(w.k_pool), npv(w.v_pool), st.slot_mapping.numpy(), npv(st.k_new), npv(st.v_new))
    t0 = time.perf_counter()
    oracle.decode_ref(npv(st.q), k2, v2, w.decode_block_tables.contiguous().numpy(), st.context_lens.numpy(), w.scale)
    rec = {"decode_s": time.perf_counter() - t0, "decode_bytes": w.decode_bytes(0)}
    if w.prompt_lens:
        rows = list(range(int(st.cu_q_lens[0]), int(st.cu_q_lens[1])))
        t0 = time.perf_counter()
        oracle.prefill_ref(npv(st.q_prefill), k2, v2, w.prefill_block_tables.contiguous().numpy(),
                           st.cu_q_lens.numpy(), st.prefill_context_lens.numpy(), w.scale, rows=rows)
        rec["prefill_first_prompt_s"] = time.perf_counter() - t0
        rec["prefill_first_prompt_tokens"] = len(rows)
    per[name] = rec
res["per_config_1_thread"] = per
print(json.dumps(res))
""" % (ROOT, [c for c in CONFIGS])
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    try:
        r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env, timeout=600)
    except Exception as exc:
        return {"failed": type(exc).__name__}
    if r.returncode != 0:
        return {"failed": (r.stderr.strip().splitlines() or ["no output"])[-1]}
    return json.loads(r.stdout.strip().splitlines()[-1])


# ---------------------------------------------------------------------------
# reference arm: the oracle, timed on the host cores
# ---------------------------------------------------------------------------

def run_reference(args, rank, world):
    if rank != 0:
        return
    import numpy as np
    import torch
    torch.set_num_threads(1)
    import oracle
    from paged_kv_decode_27_gb300 import workloads as W
    wl = W.llama3_8b_decode()

    def npv(t):
        t = t.contiguous()
        return t.view(torch.int16).numpy().view(np.uint16) if t.dtype == torch.bfloat16 else t.numpy()
    kp, vp = npv(wl.k_pool), npv(wl.v_pool)
    bt = wl.decode_block_tables.contiguous().numpy()
    per_step = 2   # sequences of the batch per step: a bounded sample

    def one(i):
        st = wl.step(i % wl.steps)
        seqs = [(2 * i + j) % 64 for j in range(per_step)]
        k2, v2 = oracle.append_ref(kp, vp, st.slot_mapping.numpy()[seqs], npv(st.k_new)[seqs],
                                   npv(st.v_new)[seqs])
        ctx = st.context_lens.numpy()
        t0 = time.perf_counter()
        oracle.decode_ref(npv(st.q), k2, v2, bt, ctx, wl.scale, seqs=seqs)
        el = time.perf_counter() - t0
        b = sum(int(ctx[s]) * 2 * 8 * 128 * 2 + 2 * 32 * 128 * 2 + 4 * ((int(ctx[s]) + 15) // 16) + 4 for s in seqs)
        return el, b, seqs
    for i in range(args.warmup):
        one(i)
    tot_t = tot_b = 0.0
    for i in range(args.steps):
        el, b, _ = one(args.warmup + i)
        tot_t += el
        tot_b += b
    value = tot_b / tot_t / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot_t / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": WORKLOAD_DESC},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": f"float64 numpy oracle: {per_step} sequences (all 32 q heads, their full "
                                       f"contexts) of each step's batch, rotating; append of those sequences "
                                       f"untimed"},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    import __graft_entry__
    __graft_entry__.build()
    from paged_kv_decode_27_gb300 import binding as pa
    from paged_kv_decode_27_gb300 import workloads as W

    # the CPU oracle baseline runs first, in its own 1-thread process, then on all cores
    cpu = None
    if rank == 0 and not (args.no_cpu_baseline or args.quick):
        cpu = cpu_baseline()
        if world == 1:
            more = cpu_oracle_more()
            cpu["host_cores"] = more.get("cores", len(os.sched_getaffinity(0)))
            cpu["all_cores"] = more.get("all_cores", more)
            cpu["per_config_1_thread"] = more.get("per_config_1_thread")

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    wl = W.llama3_8b_decode()
    S, hq, hkv, d = wl.num_decode_seqs, wl.num_q_heads, wl.num_kv_heads, wl.head_dim
    kp, vp = wl.k_pool.to(dev), wl.v_pool.to(dev)
    bt_cpu = wl.decode_block_tables.contiguous()
    bt = bt_cpu.to(dev)
    steps_in = [wl.step(t) for t in range(wl.steps)]
    dev_in = [(s.slot_mapping.to(dev), s.k_new.to(dev), s.v_new.to(dev), s.q.to(dev), s.context_lens.to(dev))
              for s in steps_in]
    max_ctx = wl.max_context_len(wl.steps - 1)
    part = pa.pa_decode_partition_size(S, max_ctx, kp, args.partition)
    ws = torch.zeros(max(1, pa.pa_decode_workspace_size(S, hq, max_ctx, kp, args.partition)),
                     dtype=torch.uint8, device=dev)
    out = torch.empty((S, hq, d), dtype=wl.dtype, device=dev)
    stream = torch.cuda.current_stream()
    max_splits = -(-((max_ctx + 15) // 16) // (part // 16))
    launches_per_step = 1   # decode_tc_kernel with the step's append fused in (pa_decode_step)

    def step(i):
        _, kn, vn, q, ctx = dev_in[i % wl.steps]
        pa.pa_decode_step(out, q, kp, vp, kn, vn, bt, ctx, wl.scale, max_context_len=max_ctx,
                          partition_size=args.partition, workspace=ws, stream=stream)

    # untimed: >= 1 s of steps so the clock sampler sees the GPU under load, then W warm-ups
    sampler = ClockSampler(local_rank) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    t_busy0 = time.time()
    i = 0
    while not args.quick and time.time() - t_busy0 < 1.0:
        step(i)
        i += 1
        if i % 64 == 0:
            torch.cuda.synchronize()
    for w in range(args.warmup):
        step(w)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()

    # timed: exactly K steps issued back to back, CUDA events on the launching stream
    # around the whole region (an event between two launches would stop the next one
    # from starting while the previous drains)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t_wall0 = time.time()
    ev0.record(stream)
    for k in range(args.steps):
        step(args.warmup + k)
    ev1.record(stream)
    torch.cuda.synchronize()
    total_ms = ev0.elapsed_time(ev1)
    # the same K steps again with an event pair around every call: the per-launch
    # duration of the roofline
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    for k in range(args.steps):
        ev[k][0].record(stream)
        step(args.warmup + k)
        ev[k][1].record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    if world > 1:
        dist.barrier()
    if sampler:
        time.sleep(0.25)
        sampler.stop()
    attn_ms = [ev[k][0].elapsed_time(ev[k][1]) for k in range(args.steps)]
    total_ms = max_over_ranks(total_ms, dev, world)

    dec_b = [wl.decode_bytes((args.warmup + k) % wl.steps) for k in range(args.steps)]
    app_b = wl.append_bytes()
    step_bytes = sum(dec_b) + args.steps * app_b
    value = replica_gbs(step_bytes, total_ms * 1e-3, world)
    ms_per_step = total_ms / args.steps
    peak, peak_kind = peak_hbm()
    attn_avg_ms = statistics.mean(attn_ms)
    achieved = statistics.mean(dec_b) / (attn_avg_ms * 1e-3) / 1e9
    kv_ratio = statistics.mean(dec_b) / wl.decode_bytes(0)

    # e2e through the public API with host buffers: each step's inputs (new K/V, q, context
    # lengths, block tables) sit packed in one pinned host buffer and go to the device in one H2D
    # copy; then the step call, a D2H copy of the attention output, and a synchronise
    def pack(st):
        parts = [st.k_new, st.v_new, st.q, st.context_lens, bt_cpu]
        flat = [x.contiguous().view(torch.uint8).reshape(-1) for x in parts]
        pad = [(-f.numel()) % 16 for f in flat]   # keep every view 16-byte aligned
        buf = torch.cat([torch.cat([f, torch.zeros(p_, dtype=torch.uint8)]) for f, p_ in zip(flat, pad)])
        return buf.pin_memory(), [(x.dtype, tuple(x.shape), f.numel() + p_) for x, f, p_ in zip(parts, flat, pad)]
    packed = [pack(st) for st in steps_in]
    layout = packed[0][1]
    def unpack_views(buf):
        views, off = [], 0
        for dt, shp, nb in layout:
            n = int(torch.Size(shp).numel()) * torch.empty((), dtype=dt).element_size()
            views.append(buf[off:off + n].view(dt).view(shp))
            off += nb
        return views
    d_buf = torch.empty(packed[0][0].numel(), dtype=torch.uint8, device=dev)
    d_kn, d_vn, d_q, d_ctx, d_bt = unpack_views(d_buf)
    out_host = torch.empty((S, hq, d), dtype=wl.dtype).pin_memory()
    h2d = packed[0][0].numel()
    d2h = out_host.numel() * out_host.element_size()

    def enqueue(t, st):
        d_buf.copy_(packed[t % wl.steps][0], non_blocking=True)
        pa.pa_decode_step(out, d_q, kp, vp, d_kn, d_vn, d_bt, d_ctx, wl.scale, max_context_len=max_ctx,
                          partition_size=args.partition, workspace=ws, stream=st)
        out_host.copy_(out, non_blocking=True)

    # The library allocates nothing and never synchronises, so a step (H2D of
    # its packed inputs, the append + decode call, D2H of the output) can be captured in
    # a CUDA graph once per input buffer and replayed: one launch per step.
    graphs, e2e_mode = [], "eager"
    if not args.quick:
        try:
            torch.cuda.synchronize()
            for t in range(wl.steps):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g):
                    enqueue(t, torch.cuda.current_stream())
                graphs.append(g)
            e2e_mode = "cuda_graph"
        except Exception as exc:   # capture unsupported here: time the eager calls instead
            graphs, e2e_mode = [], f"eager ({type(exc).__name__})"
            torch.cuda.synchronize()

    def e2e_step(t):
        if graphs:
            graphs[t % wl.steps].replay()
        else:
            enqueue(t, stream)
        stream.synchronize()
    e2e_s = float("nan")
    if not args.quick:
        for w in range(args.warmup):
            e2e_step(w)
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        te0 = time.perf_counter()
        for k in range(args.steps):
            e2e_step(args.warmup + k)
        te1 = time.perf_counter()
        e2e_s = te1 - te0
    e2e_s = max_over_ranks(e2e_s, dev, world)
    e2e_value = replica_gbs(step_bytes, e2e_s, world)

    # Pipelined, as a serving loop runs it: step t's inputs go up on an H2D stream
    # while step t-1 computes, its output comes back on a D2H stream while step
    # t+1 computes, and the host waits for each step's output one step later.
    # Two input/output buffer pairs; events keep every reuse ordered.
    NB = 2
    p_bufs = [torch.empty_like(d_buf) for _ in range(NB)]
    p_views = [unpack_views(b) for b in p_bufs]
    p_outs = [torch.empty_like(out) for _ in range(NB)]
    p_host = [torch.empty((S, hq, d), dtype=wl.dtype).pin_memory() for _ in range(NB)]
    s_h2d, s_d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(NB)]
    ev_k = [torch.cuda.Event() for _ in range(NB)]
    ev_out = [torch.cuda.Event() for _ in range(NB)]

    def e2e_pipelined(t_first, n):
        for b in range(NB):
            ev_k[b].record(stream)
            ev_out[b].record(s_d2h)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for i in range(n):
            t, b = t_first + i, i % NB
            s_h2d.wait_event(ev_k[b])            # step t-2 has finished reading input buffer b
            with torch.cuda.stream(s_h2d):
                p_bufs[b].copy_(packed[t % wl.steps][0], non_blocking=True)
            ev_in[b].record(s_h2d)
            stream.wait_event(ev_in[b])          # this step's inputs are on the device
            stream.wait_event(ev_out[b])         # step t-2's output has left buffer b
            kn, vn, qq, cc, bb = p_views[b]
            pa.pa_decode_step(p_outs[b], qq, kp, vp, kn, vn, bb, cc, wl.scale, max_context_len=max_ctx,
                              partition_size=args.partition, workspace=ws, stream=stream)
            ev_k[b].record(stream)
            s_d2h.wait_event(ev_k[b])
            with torch.cuda.stream(s_d2h):
                p_host[b].copy_(p_outs[b], non_blocking=True)
            ev_out[b].record(s_d2h)
            if i >= 1:
                ev_out[(i - 1) % NB].synchronize()   # the host holds step t-1's output
        ev_out[(n - 1) % NB].synchronize()
        return time.perf_counter() - t0

    pipe_s = float("nan")
    if not args.quick:
        e2e_pipelined(0, args.warmup)
        if world > 1:
            dist.barrier()
        pipe_s = e2e_pipelined(args.warmup, args.steps)
        # the pipelined steps wrote the same new tokens as the timed steps: check one output
        if not torch.equal(p_host[(args.steps - 1) % NB], p_outs[(args.steps - 1) % NB].cpu()):
            raise RuntimeError("pipelined e2e: host copy differs from the device output")
    pipe_s = max_over_ranks(pipe_s, dev, world)
    pipe_value = replica_gbs(step_bytes, pipe_s, world)

    status = pa.pa_device_status()
    if rank != 0:
        return
    clocks = sampler.summary(t_busy0, t_wall1 + 0.1) if sampler else None
    # every configuration of the workload list, per call (L2 evicted), after the timed region
    configs = None
    others = None
    if world == 1 and not args.quick:
        del kp, vp, dev_in, p_bufs, p_views, graphs
        torch.cuda.empty_cache()
        configs = measure_configs(pa, W, torch, dev)
        others = measure_other_workloads(pa, W, torch, dev)
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD_DESC, "partition_tokens": part, "max_splits": max_splits,
                   "l2": "inputs larger than L2: ~726 MB of K/V read per step vs 129 MB L2, no flush",
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "step": "pa_decode_step: each sequence's new token appended by the decode launch itself",
                   "timing": "value: K steps back to back between two CUDA events; roofline: a second pass "
                             "of the same K steps with an event pair around each call"},
        "pct_of_peak": value / peak,
        "decode_tokens_per_s": world * S * args.steps / (total_ms * 1e-3),
        "attention_us": 1e3 * attn_avg_ms, "append_us": None,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": measured_traffic(kv_ratio),
                     "kernel": "pa_decode_step (decode_tc_kernel: append and split-K merge fused), "
                               "CUDA events per call",
                     "peak_kind": f"{peak_kind} (STREAM-like copy, burst)"},
        "e2e": {"value": pipe_value, "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "mode": "pipelined: H2D of step t+1 and D2H of step t-1 on their own streams beside step t; "
                        "the host waits for every step's output",
                "value_synchronous": e2e_value,
                "mode_synchronous": f"{e2e_mode}: H2D, step call, D2H, synchronise, one step at a time"},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks, "device_status": status,
        "cpu_baseline": cpu,
        "configs": configs,
        "other_workloads": others,
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# per-call figures of the other workloads
# ---------------------------------------------------------------------------

# Layers of the model each workload's head shape comes from (attention-only
# per-model figures divide the one-layer rate by this).
N_LAYERS = {"tiny_fp32": 1, "llama32_1b_decode": 16, "llama3_8b_decode": 32, "prefix_shared_8k": 32,
            "mixed_mistral7b": 32, "llama3_8b_long_b1": 32, "llama3_8b_long_b4": 32,
            "llama32_1b_decode_int8": 16, "llama3_8b_decode_int8": 32, "llama3_8b_verify": 32,
            "llama3_8b_verify_int8": 32, "llama3_8b_decode_rope": 32, "mixed_mistral7b_int8": 32}
# The five configurations of the benchmark's workload list, then the small-batch
# end of its decode range (batch 1 and 4 at contexts up to 8192).
CONFIGS = ["tiny_fp32", "llama32_1b_decode", "llama3_8b_decode", "prefix_shared_8k", "mixed_mistral7b",
           "llama3_8b_long_b1", "llama3_8b_long_b4"]
# The other calls of the path on the same head shapes: the INT8 cache (decode,
# and the mixed step with its INT8 prompt pass) and the verification pass of
# speculative decoding over both cache formats.
OTHER_WORKLOADS = ["llama3_8b_decode_int8", "mixed_mistral7b_int8", "llama3_8b_verify", "llama3_8b_verify_int8"]


def peak_bf16():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return 1900.0, "fallback"


def l2_flusher(torch, dev):
    """A read of twice the L2 size (L2 from the device attribute), which
    evicts every line without leaving dirty ones behind (a write would make the
    timed call pay for their write-back)."""
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size or (129 << 20)
    buf = torch.ones(max(2 * l2, 256 << 20) // 2, dtype=torch.float16, device=dev)
    return lambda: buf.sum()


def measure_workload(name, pa, W, torch, dev, reps, warmup, partition=0, flush=None):
    """Append / prefill / attention times of one workload, each call bracketed by
    CUDA events on its stream, with L2 evicted before every repetition so that
    each call reads its inputs from HBM.  Median and p90 over `reps` calls."""
    wl = W.WORKLOADS[name]()
    kp, vp = wl.k_pool.to(dev), wl.v_pool.to(dev)
    ks = wl.k_scales.to(dev) if wl.kv_int8 else None
    vs = wl.v_scales.to(dev) if wl.kv_int8 else None
    bt = wl.decode_block_tables.contiguous().to(dev)
    pbt = wl.prefill_block_tables.contiguous().to(dev) if wl.prompt_lens else None
    steps_in = [wl.step(t) for t in range(wl.steps)]
    d_in = []
    for st in steps_in:
        d = {"slots": st.slot_mapping.to(dev), "kn": st.k_new.to(dev), "vn": st.v_new.to(dev),
             "q": st.q.to(dev), "ctx": st.context_lens.to(dev)}
        if wl.prompt_lens:
            d.update(qp=st.q_prefill.to(dev), cu=st.cu_q_lens.to(dev), pctx=st.prefill_context_lens.to(dev),
                     pout=torch.empty_like(st.q_prefill, device=dev))
        d_in.append(d)
    max_ctx = wl.max_context_len(wl.steps - 1)
    S, hq, dh = wl.num_decode_seqs, wl.num_q_heads, wl.head_dim
    ws = torch.zeros(max(1, pa.pa_decode_workspace_size(S, hq, max_ctx, kp, partition)),
                     dtype=torch.uint8, device=dev)
    out = torch.empty((S, hq, dh), dtype=wl.dtype, device=dev)
    vq = wl.extra.get("verify_q_len", 0)
    if vq:   # a verification pass replaces the decode: q_len query rows per sequence
        for t, d in enumerate(d_in):
            d["vq"] = wl.verify_queries(t, vq).to(dev)
        out = torch.empty((S, vq, hq, dh), dtype=wl.dtype, device=dev)
        ws = torch.zeros(max(1, pa.pa_verify_workspace_size(S, vq, hq, max_ctx, kp, partition)),
                         dtype=torch.uint8, device=dev)
    theta = wl.extra.get("rope_theta")
    if theta:   # RoPE: K rotated on the append, q rotated at position context - 1
        cos_sin = torch.empty((max_ctx + 1, dh // 2, 2), dtype=torch.float32, device=dev)
        pa.pa_rope_cache(cos_sin, theta)
        for d in d_in:
            d["pos"] = (d["ctx"] - 1).to(torch.int32)
            d["q0"] = d["q"].clone()
    pws = None
    if wl.prompt_lens and wl.kv_int8:   # the INT8 prompt pass dequantises into its workspace
        mp = max(wl.prompt_lens)
        pws = torch.empty(max(1, pa.pa_prefill_int8_workspace_size(len(wl.prompt_lens), mp, kp)),
                          dtype=torch.uint8, device=dev)
    flush = flush or l2_flusher(torch, dev)
    stream = torch.cuda.current_stream()
    rec = {"append": [], "prefill": [], "decode": []}

    def step(t, timed):
        d = d_in[t % wl.steps]
        if timed:
            flush()
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        if theta:
            d["q"].copy_(d["q0"])   # the queries arrive unrotated every step
        evs[0].record(stream)
        if wl.kv_int8:
            pa.pa_append_kv_int8(kp, vp, ks, vs, d["slots"], d["kn"], d["vn"], stream=stream)
        elif theta:
            pa.pa_append_kv_rope(kp, vp, d["slots"], d["pos"], d["kn"], d["vn"], cos_sin, stream=stream)
            pa.pa_apply_rope(d["q"], d["pos"], cos_sin, stream=stream)
        else:
            pa.pa_append_kv(kp, vp, d["slots"], d["kn"], d["vn"], stream=stream)
        evs[1].record(stream)
        if wl.prompt_lens and wl.kv_int8:
            pa.pa_prefill_attention_int8(d["pout"], d["qp"], kp, vp, ks, vs, pbt, d["cu"], d["pctx"], wl.scale,
                                         max_q_len=max(wl.prompt_lens), max_context_len=max(wl.prompt_lens),
                                         workspace=pws, stream=stream)
        elif wl.prompt_lens:
            pa.pa_prefill_attention(d["pout"], d["qp"], kp, vp, pbt, d["cu"], d["pctx"], wl.scale,
                                    max_q_len=max(wl.prompt_lens), max_context_len=max(wl.prompt_lens),
                                    stream=stream)
        evs[2].record(stream)
        if vq and wl.kv_int8:
            pa.pa_verify_attention_int8(out, d["vq"], kp, vp, ks, vs, bt, d["ctx"], wl.scale,
                                        max_context_len=max_ctx, partition_size=partition, workspace=ws,
                                        stream=stream)
        elif vq:
            pa.pa_verify_attention(out, d["vq"], kp, vp, bt, d["ctx"], wl.scale, max_context_len=max_ctx,
                                   partition_size=partition, workspace=ws, stream=stream)
        elif wl.kv_int8:
            pa.pa_decode_attention_int8(out, d["q"], kp, vp, ks, vs, bt, d["ctx"], wl.scale, max_context_len=max_ctx,
                                        partition_size=partition, workspace=ws, stream=stream)
        else:
            pa.pa_decode_attention(out, d["q"], kp, vp, bt, d["ctx"], wl.scale, max_context_len=max_ctx,
                                   partition_size=partition, workspace=ws, stream=stream)
        evs[3].record(stream)
        return evs
    for w in range(warmup):
        step(w, False)
    torch.cuda.synchronize()
    # a ~50 ms device-side delay lets the host enqueue every timed step before the GPU starts on
    # them, so that the events time the GPU work and not the host's enqueue of small calls
    torch.cuda._sleep(100_000_000)
    evl = [step(warmup + k, True) for k in range(reps)]
    torch.cuda.synchronize()
    for e in evl:
        rec["append"].append(e[0].elapsed_time(e[1]) * 1e3)
        rec["prefill"].append(e[1].elapsed_time(e[2]) * 1e3)
        rec["decode"].append(e[2].elapsed_time(e[3]) * 1e3)
    med = {k: statistics.median(v) for k, v in rec.items()}
    p90 = {k: sorted(v)[int(0.9 * (reps - 1))] for k, v in rec.items()}
    t_mid = (warmup + reps // 2) % wl.steps
    dec_b = wl.verify_bytes(t_mid, vq) if vq else wl.decode_bytes(t_mid)
    peak, kind = peak_hbm()
    nl = N_LAYERS.get(wl.name, 1)
    tok_s = S / ((med["append"] + med["decode"] + med["prefill"]) * 1e-6)
    line = {"workload": wl.name, "description": wl.description, "reps": reps, "warmup": warmup,
            "l2": "evicted before every repetition (a read of 2x the L2 size)",
            # the decode's partition (a verification pass chooses its own split)
            "partition_tokens": None if vq else pa.pa_decode_partition_size(S, max_ctx, kp, partition),
            "append_us": med["append"], "append_p90_us": p90["append"],
            "append_gbs": wl.append_bytes() / (med["append"] * 1e-6) / 1e9,
            "attention_us": med["decode"], "attention_p90_us": p90["decode"],
            "attention_gbs": dec_b / (med["decode"] * 1e-6) / 1e9,
            "attention_frac_of_hbm_peak": dec_b / (med["decode"] * 1e-6) / 1e9 / peak,
            "hbm_peak_gbs": peak, "hbm_peak_kind": kind, "attention_bytes": dec_b,
            "decode_tokens_per_s": tok_s, "n_layers": nl,
            "decode_tokens_per_s_attention_only_per_model": tok_s / nl}
    if theta:
        line["rope_theta"] = theta
        line["append_note"] = "append_us covers the RoPE append of K and the in-place rotation of q"
    if wl.prompt_lens:
        fl = wl.prefill_flops()
        pk, pkind = peak_bf16()
        line.update(prefill_us=med["prefill"], prefill_p90_us=p90["prefill"],
                    prefill_tflops=fl / (med["prefill"] * 1e-6) / 1e12,
                    prefill_frac_of_bf16_peak=fl / (med["prefill"] * 1e-6) / 1e12 / pk,
                    bf16_peak_tflops=pk, bf16_peak_kind=pkind, prefill_flops=fl)
    line["device_status"] = pa.pa_device_status()
    return line


def measure_model_step(name, pa, W, torch, dev, reps, warmup):
    """One decode step of the whole model's attention: n_layers fused append +
    decode calls (pa_decode_step), back to back on one stream, each layer over
    its own K/V pool (n_layers distinct pools, together larger than L2, so every
    layer reads its cache from HBM).  Timed with one CUDA event pair around the
    n_layers calls, median over `reps` steps."""
    wl = W.WORKLOADS[name]()
    nl = N_LAYERS.get(wl.name, 1)
    st = wl.step(0)
    kp0, vp0 = wl.k_pool.to(dev), wl.v_pool.to(dev)
    pools = [(kp0.clone(), vp0.clone()) for _ in range(nl)]
    del kp0, vp0
    bt = wl.decode_block_tables.contiguous().to(dev)
    q, kn, vn, ctx = st.q.to(dev), st.k_new.to(dev), st.v_new.to(dev), st.context_lens.to(dev)
    S, hq = wl.num_decode_seqs, wl.num_q_heads
    mc = wl.max_context_len(0)
    ws = torch.zeros(max(1, pa.pa_decode_workspace_size(S, hq, mc, pools[0][0])), dtype=torch.uint8, device=dev)
    outs = [torch.empty_like(q) for _ in range(nl)]
    stream = torch.cuda.current_stream()

    def model_step():
        for layer, (kp, vp) in enumerate(pools):
            pa.pa_decode_step(outs[layer], q, kp, vp, kn, vn, bt, ctx, wl.scale, max_context_len=mc,
                              workspace=ws, stream=stream)
    for _ in range(warmup):
        model_step()
    torch.cuda.synchronize()
    torch.cuda._sleep(100_000_000)
    evs = []
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        model_step()
        e1.record(stream)
        evs.append((e0, e1))
    torch.cuda.synchronize()
    t = sorted(a.elapsed_time(b) * 1e3 for a, b in evs)
    med = statistics.median(t)
    peak, _ = peak_hbm()
    b = nl * (wl.decode_bytes(0) + wl.append_bytes())
    return {"n_layers": nl, "layer_pools_mb": round(nl * 2 * wl.k_pool.numel() * wl.k_pool.element_size() / 1e6, 1),
            "model_step_us": med, "model_step_p90_us": t[int(0.9 * (reps - 1))], "per_layer_us": med / nl,
            "gbs": b / (med * 1e-6) / 1e9, "frac_of_hbm_peak": b / (med * 1e-6) / 1e9 / peak,
            "decode_tokens_per_s_attention_only_per_model": S / (med * 1e-6),
            "how": f"{nl} pa_decode_step calls back to back, one per layer pool, one event pair around them"}


def measure_configs(pa, W, torch, dev, reps=60, warmup=5):
    flush = l2_flusher(torch, dev)
    res = {}
    for name in CONFIGS:
        res[name] = measure_workload(name, pa, W, torch, dev, reps, warmup, flush=flush)
        if name in ("llama32_1b_decode", "llama3_8b_long_b1", "llama3_8b_long_b4"):
            res[name]["model_step"] = measure_model_step(name, pa, W, torch, dev, max(reps // 3, 20), 3)
        torch.cuda.empty_cache()
    return res


def measure_other_workloads(pa, W, torch, dev, reps=30, warmup=3):
    """OTHER_WORKLOADS per call, as measure_configs; a workload that fails is
    reported by its error, after the headline and the configurations."""
    flush = l2_flusher(torch, dev)
    res = {}
    for name in OTHER_WORKLOADS:
        try:
            res[name] = measure_workload(name, pa, W, torch, dev, reps, warmup, flush=flush)
        except Exception as e:   # keep the line: the headline was measured already
            res[name] = {"error": repr(e)[:300]}
        torch.cuda.empty_cache()
    return res


def run_other(args):
    """Per-call figures of one workload (L2 evicted before every step)."""
    import torch

    import __graft_entry__
    __graft_entry__.build()
    from paged_kv_decode_27_gb300 import binding as pa
    from paged_kv_decode_27_gb300 import workloads as W

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    line = measure_workload(args.workload, pa, W, torch, dev, args.steps, args.warmup, args.partition)
    print(json.dumps(line), flush=True)


def run_serving(args):
    """Decode steps driven by the block manager with a prefix cache: 64
    sequences whose prompts share a 208-token system prompt (13 blocks) and
    whose contexts are log-uniform in [512, 8192] (the Llama-3-8B-shaped
    decode batch).  Every step appends one token per sequence through the
    manager (host), uploads slots and block tables, appends K/V and decodes.
    Reports the manager's host time per step beside the GPU time."""
    import math
    import numpy as np
    import torch

    import __graft_entry__
    __graft_entry__.build()
    from paged_kv_decode_27_gb300 import binding as pa

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    S, hq, hkv, d, sys_len = 64, 32, 8, 128, 208
    g = torch.Generator().manual_seed(2024)
    u = torch.rand((S,), generator=g, dtype=torch.float64)
    ctx0 = torch.floor(torch.exp(math.log(512) + u * (math.log(8192) - math.log(512)))).to(torch.int64)
    steps_total = args.warmup + args.steps
    mb = (int(ctx0.max()) + steps_total + 15) // 16
    nb = int(1.1 * (sum((int(c) + steps_total + 15) // 16 for c in ctx0)))
    bm = pa.pa_bm_create(nb, mb, S)
    system = torch.randint(0, 32000, (sys_len,), generator=g).tolist()
    t0 = time.perf_counter()
    cached = 0
    for s in range(S):
        prompt = system + torch.randint(0, 32000, (int(ctx0[s]) - sys_len,), generator=g).tolist()
        cached += pa.pa_bm_add_sequence(bm, s, prompt)[0]
    add_s = time.perf_counter() - t0
    kp = torch.randn((nb, hkv, 16, d), generator=g).to(torch.bfloat16).to(dev)
    vp = torch.randn((nb, hkv, 16, d), generator=g).to(torch.bfloat16).to(dev)
    q = torch.randn((S, hq, d), generator=g).to(torch.bfloat16).to(dev)
    kn = torch.randn((S, hkv, d), generator=g).to(torch.bfloat16).to(dev)
    vn = torch.randn((S, hkv, d), generator=g).to(torch.bfloat16).to(dev)
    out = torch.empty_like(q)
    max_ctx = mb * 16
    ws = torch.zeros(max(1, pa.pa_decode_workspace_size(S, hq, max_ctx, kp)), dtype=torch.uint8, device=dev)
    slot_h = torch.empty((S,), dtype=torch.int64).pin_memory()
    tab_h = torch.empty((S, mb), dtype=torch.int32).pin_memory()
    ctx_h = torch.empty((S,), dtype=torch.int32).pin_memory()
    slot_d = torch.empty((S,), dtype=torch.int64, device=dev)
    tab_d = torch.empty((S, mb), dtype=torch.int32, device=dev)
    ctx_d = torch.empty((S,), dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()
    host_us, step_us, gpu_us = [], [], []
    ids_np = np.arange(S, dtype=np.int32)
    for it in range(steps_total):
        tw0 = time.perf_counter()
        toks = np.full(S, it % 32000, dtype=np.int32)
        _, copies = pa.pa_bm_append_step(bm, ids_np, toks, slots_out=slot_h)
        pa.pa_bm_block_tables_into(bm, ids_np, tab_h, ctx_h)
        th = time.perf_counter()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        slot_d.copy_(slot_h, non_blocking=True)
        tab_d.copy_(tab_h, non_blocking=True)
        ctx_d.copy_(ctx_h, non_blocking=True)
        e0.record(stream)
        pa.pa_append_kv(kp, vp, slot_d, kn, vn, stream=stream)
        pa.pa_decode_attention(out, q, kp, vp, tab_d, ctx_d, 1.0 / math.sqrt(d), max_context_len=max_ctx,
                               workspace=ws, stream=stream)
        e1.record(stream)
        stream.synchronize()
        te = time.perf_counter()
        if it >= args.warmup:
            host_us.append((th - tw0) * 1e6)
            step_us.append((te - tw0) * 1e6)
            gpu_us.append(e0.elapsed_time(e1) * 1e3)
    st = pa.pa_bm_get_stats(bm)
    pa.pa_bm_destroy(bm)
    line = {"workload": "llama3_8b_prefix_serving",
            "description": "64 sequences sharing a 208-token system prompt, contexts log-uniform in [512, 8192], "
                           "one token per sequence per step through the block manager",
            "steps": args.steps, "warmup": args.warmup,
            "prompt_tokens_from_prefix_cache": cached, "add_sequences_ms": add_s * 1e3,
            "manager_host_us_per_step": statistics.median(host_us),
            "manager_host_us_per_token": statistics.median(host_us) / S,
            "gpu_us_per_step": statistics.median(gpu_us), "wall_us_per_step": statistics.median(step_us),
            "manager_stats": st, "device_status": pa.pa_device_status()}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if args.workload != WORKLOAD:
        if world > 1:
            raise SystemExit("--workload other than the headline runs on one GPU")
        if args.workload == "llama3_8b_prefix_serving":
            run_serving(args)
        else:
            run_other(args)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    try:
        run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
