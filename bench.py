"""Benchmark of one hybrid-batch attention step (KV append + attention).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl native|reference] [--sweep chunk]

A step is one pass of the hot path over one synthetic hybrid batch: the KV
append of the batch's new tokens and the attention of every new token (decode
rows and prefill chunks) over the paged cache, through the C ABI.  The batch
layout (q_len, context_len, block tables) is fixed per workload, so the plan
is built once.  The default workload is the largest single-GPU batch: the
Yi-34B attention shape at a 2048-token budget (32 decode rows over long
contexts + one 2016-token chunk at offset 6048).

Printed (rank 0, one JSON line): tokens/s over the timed steps with inputs
resident in HBM (`value`), the same through host buffers with the copies in
the timed region (`e2e`), the dominant kernel's roofline figures, the whole
step's fraction of its roofline, the CPU oracle timed on a bounded sample, and
the SM clocks sampled during the timed region.

`--impl reference` times the fp64 CPU oracle instead (rank 0 only).
`--layer` times one whole transformer block of the batch instead (the
linear layers on synthetic weights around the attention step).
`--sweep chunk` prefills one 8192-token prompt in chunks of several sizes,
with and without decode rows beside each chunk, and prints one JSON line per
chunk size (the chunk-size sweep; not the step benchmark).
Under torchrun (N > 1) each rank runs an independent replica of the workload;
timing is the max over ranks and `value` counts every rank's tokens.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from chunked_prefill_decode_gb300 import workloads  # noqa: E402

METRIC = "mixed-batch paged attention tokens/s; % of roofline (HBM GB/s or TC util)"
L2_BYTES = 129 * 1024 * 1024


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


ATTN_SOURCES = ("attention.cu", "decode_body.cuh", "chunk_body.cuh", "ptx.cuh",
                "hb_internal.h", "decode_plan.h", "api.cu")


def source_code_tokens(text):
    """C/C++/CUDA source with its comments removed and every run of
    whitespace made one space: what the compiler sees, so that a change to a
    comment or to the layout of the text does not count as a change of the
    kernel.  String and character literals are kept as they are."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c == "/" and i + 1 < n and text[i + 1] == "/":
            j = text.find("\n", i)
            i = n if j < 0 else j
            out.append(" ")
        elif c == "/" and i + 1 < n and text[i + 1] == "*":
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        elif c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def attention_sources_digest(root=None):
    """First 16 hex digits of the sha256 over the attention launch's sources
    (comments and layout ignored), as recorded in its ncu summaries."""
    import hashlib
    h = hashlib.sha256()
    for src in ATTN_SOURCES:
        with open(os.path.join(root or ROOT, "chunked_prefill_decode_gb300", "csrc", src)) as f:
            h.update(source_code_tokens(f.read()).encode())
        h.update(b"\0")
    return h.hexdigest()[:16]


def profiled_traffic(workload):
    """DRAM bytes per attention launch from the committed ncu summary of this
    workload, if the summary was taken on the current kernel code."""
    path = os.path.join(ROOT, "profiles", f"attention_{workload}.md")
    if not os.path.exists(path):
        return None
    fields = {}
    for line in open(path):
        if ":" in line and line.split(":")[0] in ("traffic_bytes_per_launch", "code_sha256"):
            k, v = line.split(":", 1)
            fields[k.strip()] = v.strip()
    if fields.get("code_sha256") != attention_sources_digest():
        return None
    return int(fields["traffic_bytes_per_launch"])


def algorithmic_counts(layout):
    """FLOPs and bytes of one step, by kernel, counted from the definition.

    attention FLOPs: 4 * Hq * D * sum over new tokens of (keys it sees);
    decode bytes: K and V of every decode row's context once per kv head,
    plus its q row and output; chunk bytes: K and V of the chunk's context
    once per kv head, plus q and out; append bytes: new K and V read and
    written."""
    sh = layout.shape
    Hq, Hkv, D = sh.num_q_heads, sh.num_kv_heads, sh.head_dim
    W = sh.sliding_window
    kv_tok = 2 * Hkv * D * 2               # K+V bytes per cached token
    qo_tok = 2 * Hq * D * 2                # q read + out written per new token
    c = {"decode_bytes": 0, "decode_flops": 0, "chunk_bytes": 0, "chunk_flops": 0}
    for q, ctx in zip(layout.q_len.tolist(), layout.context_len.tolist()):
        # keys each new token sees (a sliding window caps them at W), and the
        # keys the row needs at all
        seen = sum(min(ctx - q + j + 1, W) if W > 0 else ctx - q + j + 1 for j in range(q))
        first_key = max(0, ctx - q - W + 1) if W > 0 else 0
        flops = 4 * Hq * D * seen
        byts = (ctx - first_key) * kv_tok + q * qo_tok
        kind = "decode" if q == 1 else "chunk"
        c[kind + "_bytes"] += byts
        c[kind + "_flops"] += flops
    c["append_bytes"] = 2 * layout.total_q * kv_tok
    c["bytes"] = c["decode_bytes"] + c["chunk_bytes"] + c["append_bytes"]
    c["flops"] = c["decode_flops"] + c["chunk_flops"]
    return c


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index, period_ms=20):
        self.proc = None
        self.idx = device_index
        self.period = period_ms

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", str(self.period)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is None:
            return False
        time.sleep(0.05)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        self.lines = [l for l in out.splitlines() if l.strip()]
        return False

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def _dist(backend="nccl"):
    n = int(os.environ.get("WORLD_SIZE", "1"))
    if n > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend)
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return n, rank, local


def replica_launch(gpus, argv, env=None):
    """--gpus N against the process's rank environment.  Under a launcher
    (WORLD_SIZE set) N must equal WORLD_SIZE: a mismatch ends the run with
    exit code 2 instead of timing the wrong number of GPUs.  Without one, N > 1
    starts N replica ranks through torch.distributed.run on this node (127.0.0.1)
    and returns their exit code; N = 1 returns None (run here)."""
    env = os.environ if env is None else env
    if gpus < 1:
        print(f"bench.py: --gpus {gpus} must be >= 1", file=sys.stderr)
        return 2
    if "WORLD_SIZE" in env:
        ws = int(env["WORLD_SIZE"])
        if ws != gpus:
            print(f"bench.py: --gpus {gpus} but WORLD_SIZE={ws}", file=sys.stderr)
            return 2
        return None
    if gpus == 1:
        return None
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes", "1",
           "--nproc-per-node", str(gpus), "--master-addr", "127.0.0.1",
           "--master-port", str(port), os.path.abspath(__file__)] + list(argv)
    return subprocess.run(cmd).returncode


def _barrier(n):
    if n > 1:
        torch.distributed.barrier()


def max_over_ranks(x: float, n: int) -> float:
    """Largest value over the ranks (the job ends when its slowest rank does)."""
    if n <= 1:
        return x
    dev = "cuda" if torch.distributed.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(tokens_per_step: int, steps: int, n: int, ms_local: float) -> float:
    """Whole-job rate of n independent replicas: every rank's tokens over the
    slowest rank's time."""
    return n * tokens_per_step * steps / (max_over_ranks(ms_local, n) / 1e3)


# ---------------------------------------------------------------------------
def oracle_sample_rate(layout, ten_host, budget_s=12.0, rows=None):
    """Time the fp64 oracle on the CPU on a sample of the batch's rows:
    decode rows first (each is one token), then single chunk tokens, until
    `budget_s` seconds have been spent.  Returns (tokens/s, description)."""
    from oracle import paged_attention as pa
    sh = layout.shape
    bits = workloads.bf16_bits
    q = bits(ten_host.q)
    kc, vc = bits(ten_host.k_cache), bits(ten_host.v_cache)
    kn, vn = bits(ten_host.k_new), bits(ten_host.v_new)
    kp, vp = pa.kv_append(kc, vc, kn, vn, layout.q_len, layout.context_len,
                          layout.block_table, sh.page_size)
    cu = layout.cu_q_len
    order = rows
    if order is None:
        dec = [int(cu[s]) for s in range(layout.num_seqs) if layout.q_len[s] == 1]
        chk = [int(cu[s] + j) for s in range(layout.num_seqs) if layout.q_len[s] > 1
               for j in range(0, int(layout.q_len[s]), 7)]
        order = dec + chk
    scale = 1.0 / math.sqrt(sh.head_dim)
    done, t0 = 0, time.perf_counter()
    while time.perf_counter() - t0 < budget_s:
        tok = order[done % len(order)]
        pa.attention(q, kp, vp, layout.q_len, layout.context_len, layout.block_table,
                     sh.page_size, sh.num_q_heads, sh.num_kv_heads, scale, tokens=[tok],
                     window=sh.sliding_window)
        done += 1
    dt = time.perf_counter() - t0
    return done / dt, f"{done} new tokens (all {sh.num_q_heads} heads) of this batch, " \
                      f"decode rows then every 7th chunk token, cycled, {dt:.1f} s"


_ONE_THREAD_ENV = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS",
                   "BLIS_NUM_THREADS", "VECLIB_MAXIMUM_THREADS")


def oracle_sample_rate_one_thread(workload, budget_s):
    """The same oracle sample with BLAS held to one thread: a fresh process
    (the thread count of a BLAS library is fixed when it loads).  Returns
    (tokens/s, description) or (None, reason)."""
    import subprocess
    env = dict(os.environ)
    for k in _ONE_THREAD_ENV:
        env[k] = "1"
    env.pop("RANK", None), env.pop("WORLD_SIZE", None)
    try:
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-sample",
                            "--workload", workload, "--cpu-seconds", str(budget_s)],
                           env=env, capture_output=True, text=True, timeout=300)
        d = json.loads(r.stdout.strip().splitlines()[-1])
        return d["value"], d["sample"]
    except Exception as e:   # reported, not fatal: the GPU numbers stand alone
        return None, f"one-thread sample failed: {type(e).__name__}"


def run_oracle_sample(args):
    """Print one JSON line with the oracle's sample rate (used by
    oracle_sample_rate_one_thread in a child process)."""
    layout = workloads.WORKLOADS[args.workload]()
    v, desc = oracle_sample_rate(layout, workloads.make_tensors(layout, seed=1),
                                 budget_s=args.cpu_seconds)
    print(json.dumps({"value": v, "sample": desc}), flush=True)


def plan_host_us(db, layout, sms, reps=200):
    """Median host time of hb_plan for this batch, the host part only (no
    upload): (the C call with its arguments marshalled once, the same call
    through the Python binding)."""
    import ctypes
    from chunked_prefill_decode_gb300 import hb
    plan, _ = hb.hb_plan(db.batch, layout.q_len, layout.context_len, sms, upload=False)
    ql = np.ascontiguousarray(layout.q_len, dtype=np.int32)
    cl = np.ascontiguousarray(layout.context_len, dtype=np.int32)
    L = hb.load()
    pb, wb = ctypes.c_size_t(plan.nbytes), ctypes.c_size_t(0)
    args = (ctypes.byref(db.batch), ql.ctypes.data_as(ctypes.c_void_p),
            cl.ctypes.data_as(ctypes.c_void_p), int(sms), plan.ctypes.data_as(ctypes.c_void_p),
            ctypes.byref(pb), None, ctypes.byref(wb), None)
    c_ts, py_ts = [], []
    for _ in range(reps):
        t0 = time.perf_counter()
        st = L.hb_plan(*args)
        c_ts.append((time.perf_counter() - t0) * 1e6)
        if st != 0:
            raise RuntimeError(f"hb_plan failed ({st})")
        t0 = time.perf_counter()
        hb.hb_plan(db.batch, layout.q_len, layout.context_len, sms, plan=plan, upload=False)
        py_ts.append((time.perf_counter() - t0) * 1e6)
    return float(np.median(c_ts)), float(np.median(py_ts))


def builder_host_us(layout, reps=60, num_pages=200_000):
    """Median host time of one stall-free batch build (hb_builder_step and
    hb_builder_complete through the binding) in a steady state shaped like
    this batch: its decode rows running and a long prompt chunked into the
    rest of the budget (budget = the batch's tokens), on a pool of
    `num_pages` pages."""
    from chunked_prefill_decode_gb300 import hb
    n_dec = int((layout.q_len == 1).sum())
    budget = int(layout.total_q)
    page = layout.shape.page_size
    max_pages = max(int(layout.block_table.shape[1]), -(-(reps + 16) // page))
    b = hb.Builder(budget, page, num_pages, max_pages)
    for rid in range(n_dec):
        b.add_request(rid, 1, reps + 16)                  # decodes from the first step on
    for _ in range(-(-n_dec // budget)):                  # admit them all
        b.step()
        b.complete()
    prompt = max(1, max_pages * page // 2)
    rid = n_dec
    b.add_request(rid, prompt, 1)
    ts = []
    for _ in range(reps):
        t0 = time.perf_counter()
        b.step()
        fin = b.complete()
        ts.append((time.perf_counter() - t0) * 1e6)
        if rid in fin:
            rid += 1
            b.add_request(rid, prompt, 1)
    b.close()
    return float(np.median(ts[reps // 5:]))


def run_reference(args):
    """The fp64 CPU oracle as the reference arm (rank 0 only)."""
    n, rank, _ = _dist() if int(os.environ.get("WORLD_SIZE", "1")) > 1 else (1, 0, 0)
    if rank != 0:
        return
    layout = workloads.WORKLOADS[args.workload]()
    ten = workloads.make_tensors(layout, seed=1)
    cu = layout.cu_q_len
    dec = [int(cu[s]) for s in range(layout.num_seqs) if layout.q_len[s] == 1]
    from oracle import paged_attention as pa
    sh = layout.shape
    bits = workloads.bf16_bits
    kp, vp = pa.kv_append(bits(ten.k_cache), bits(ten.v_cache), bits(ten.k_new),
                          bits(ten.v_new), layout.q_len, layout.context_len,
                          layout.block_table, sh.page_size)
    qb = bits(ten.q)
    scale = 1.0 / math.sqrt(sh.head_dim)

    def step(i):
        tok = dec[i % len(dec)]
        pa.attention(qb, kp, vp, layout.q_len, layout.context_len, layout.block_table,
                     sh.page_size, sh.num_q_heads, sh.num_kv_heads, scale, tokens=[tok],
                     window=sh.sliding_window)

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(args.warmup + i)
    dt = time.perf_counter() - t0
    v = args.steps / dt
    cores = len(os.sched_getaffinity(0))
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s",
        "n_gpus": n, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * dt / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload},
        "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": "each step: one decode row (all q heads) of the batch, "
                                   "rows cycled, fp64 numpy oracle"},
        "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


TIMING_EVERY = 16   # --layer: timed steps per step with per-kernel CUDA events
KERNEL_TIMING_STEPS = 100   # steps of the per-kernel timing pass (>= 50 launches each)


def run_native(args):
    n, rank, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import __graft_entry__
    __graft_entry__.build()
    from chunked_prefill_decode_gb300 import hb
    from chunked_prefill_decode_gb300.device import device_batch

    layout = workloads.WORKLOADS[args.workload]()
    sh = layout.shape
    ten = workloads.make_tensors(layout, seed=1 + rank, device=dev)
    db = device_batch(layout.q_len, layout.context_len, layout.block_table,
                      layout.num_pages, sh.num_q_heads, sh.num_kv_heads, sh.head_dim,
                      sh.page_size, dev, sliding_window=sh.sliding_window)
    scale = 1.0 / math.sqrt(sh.head_dim)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    out = torch.empty_like(ten.q)
    kc, vc = ten.k_cache, ten.v_cache
    plan, ws = hb.hb_plan(db.batch, db.q_len, db.context_len, sms)
    T = layout.total_q
    stream = torch.cuda.current_stream(dev)

    def step():
        hb.hb_kv_append(db.batch, ten.k_new, ten.v_new, kc, vc)
        hb.hb_attention_new_kv(db.batch, plan, ten.q, ten.k_new, ten.v_new, kc, vc, scale, out, ws)

    for _ in range(max(args.warmup, 3)):
        step()
    hb.hb_check()
    # ---- timed region: inputs resident in HBM
    _barrier(n)
    torch.cuda.synchronize(dev)
    launches0 = hb.hb_launch_count()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        ev0.record(stream)
        for _ in range(args.steps):
            step()
        ev1.record(stream)
        torch.cuda.synchronize(dev)
    launches = hb.hb_launch_count() - launches0
    hb.hb_check()
    _barrier(n)
    # ---- per-kernel durations, in a pass of their own after the timed
    # region: CUDA events around every launch of KERNEL_TIMING_STEPS steps
    # (an event between two kernels stops the second from starting under the
    # first one's tail, so the headline loop above carries none)
    k_steps = max(KERNEL_TIMING_STEPS, 1)
    hb.hb_timing_enable(True)
    for _ in range(k_steps):
        step()
    hb.hb_timing_enable(False)
    torch.cuda.synchronize(dev)
    kdur = {k: hb.hb_timing_durations(k) for k in ("kv_append", "attention")}
    hb.hb_check()
    ms = ev0.elapsed_time(ev1)
    ms_max = max_over_ranks(ms, n)
    value = job_tokens_per_s(T, args.steps, n, ms)

    # ---- end to end through the public API with host buffers: hb_step, one
    # library call per step that plans, copies the step's inputs (q, k_new,
    # v_new, descriptors: one packed page-locked block) to the device, runs
    # append + attention and copies the output back.  Its slots order an
    # input-copy stream, the kernels' stream and an output-copy stream, so
    # a step's copies overlap the neighbouring steps' kernels, as a serving
    # loop would run them.
    from chunked_prefill_decode_gb300.device import StepStaging
    stages = [StepStaging(layout.num_seqs, T, layout.block_table.shape[1], layout.num_pages,
                          sh.num_q_heads, sh.num_kv_heads, sh.head_dim, sh.page_size,
                          sh.sliding_window, dev) for _ in range(args.e2e_stages)]
    q_len_h = np.ascontiguousarray(layout.q_len, dtype=np.int32)
    ctx_h = np.ascontiguousarray(layout.context_len, dtype=np.int32)
    for stg in stages:
        stg.h_q.copy_(ten.q.cpu())
        stg.h_k_new.copy_(ten.k_new.cpu())
        stg.h_v_new.copy_(ten.v_new.cpu())
        stg.h_cu_q_len.copy_(torch.from_numpy(layout.cu_q_len))
        stg.h_context_len.copy_(torch.from_numpy(layout.context_len))
        stg.h_block_table.copy_(torch.from_numpy(np.ascontiguousarray(layout.block_table)))
        plan_h, stg.ws = hb.hb_plan(stg.batch, layout.q_len, layout.context_len, sms)
        # the plan buffer hb_step rewrites and uploads every step, page-locked
        # so that its copy is asynchronous like the inputs'
        stg.plan = torch.empty(plan_h.nbytes, dtype=torch.uint8, pin_memory=True).numpy()
        stg.plan[:] = plan_h
        stg.slot = hb.StepSlot()
        stg.bufs = stg.step_buffers(stg.plan, stg.ws)
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    e2e_steps = max(1, min(args.steps, 200))
    h2d = stages[0].in_bytes
    d2h = stages[0].out_bytes

    def e2e_step(i):
        stg = stages[i % len(stages)]
        hb.hb_step(stg.batch, q_len_h, ctx_h, sms, stg.slot, stg.bufs, kc, vc, scale,
                   s_in, stream, s_out)

    for i in range(4):
        e2e_step(i)
    torch.cuda.synchronize(dev)
    _barrier(n)
    t0 = time.perf_counter()
    for i in range(e2e_steps):
        e2e_step(i)
    torch.cuda.synchronize(dev)
    e2e_s = max_over_ranks(time.perf_counter() - t0, n)
    hb.hb_check()
    plan_bytes = int(hb.plan_header(plan)["items_bytes"])
    e2e = {"value": n * T * e2e_steps / e2e_s, "unit": "tokens/s",
           "h2d_bytes_per_step": h2d + plan_bytes, "d2h_bytes_per_step": d2h,
           "api": "hb_step (one C call per step)",
           "copies": "per step: the plan (page-locked) and one packed page-locked block (q, "
                     "k_new, v_new, descriptors) up on an input-copy stream, which then raises "
                     "the slot's flag for the append kernel; the output down on an "
                     "output-copy stream, ordered by the slot's events; "
                     f"{len(stages)} staging buffers in flight"}

    if rank != 0:
        return
    peaks = _peaks()
    cnt = algorithmic_counts(layout)
    t_att = float(np.median(kdur["attention"]))
    t_app = float(np.median(kdur["kv_append"]))
    # the attention launch (decode and chunk CTAs together) is the dominant
    # kernel; its bound is the larger of its two roofline terms
    att_bytes = cnt["decode_bytes"] + cnt["chunk_bytes"]
    att_flops = cnt["flops"]
    t_hbm = att_bytes / (peaks["hbm_gbs"] * 1e9)
    t_tc = att_flops / (peaks["bf16_tflops"] * 1e12)
    if t_hbm >= t_tc:
        achieved = att_bytes / (t_att / 1e3) / 1e9
        roof = {"kernel": "attention", "bound": "hbm", "achieved": achieved,
                "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "traffic": None}
    else:
        achieved = att_flops / (t_att / 1e3) / 1e12
        roof = {"kernel": "attention", "bound": "tensor", "achieved": achieved,
                "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "frac": achieved / peaks["bf16_tflops"], "traffic": None}
    roof["peak_source"] = peaks["source"]
    roof["traffic"] = profiled_traffic(args.workload)
    roof["algorithmic"] = {"bytes": att_bytes, "flops": att_flops}
    roof["kernel_roofline_frac"] = max(t_hbm, t_tc) * 1e3 / t_att
    roof["median_launch_ms"] = {"attention": t_att, "kv_append": t_app}
    roof["mean_launch_ms"] = {k: float(np.mean(v)) for k, v in kdur.items()}
    roof["timed_launches"] = {"attention": len(kdur["attention"]),
                              "kv_append": len(kdur["kv_append"]),
                              "sample": f"median of CUDA events around each launch of "
                                        f"{k_steps} steps run after the timed region"}
    app_bytes = cnt["append_bytes"]
    roof["kv_append"] = {"bound": "hbm", "algorithmic_bytes": app_bytes,
                         "achieved": app_bytes / (t_app / 1e3) / 1e9, "unit": "GB/s",
                         "frac": app_bytes / (t_app / 1e3) / 1e9 / peaks["hbm_gbs"]}
    step_roof_s = max(cnt["flops"] / (peaks["bf16_tflops"] * 1e12),
                      cnt["bytes"] / (peaks["hbm_gbs"] * 1e9))
    ms_step = ms_max / args.steps
    cpu_v, cpu_desc = oracle_sample_rate(layout, workloads.make_tensors(layout, seed=1),
                                         budget_s=args.cpu_seconds)
    cpu1_v, cpu1_desc = oracle_sample_rate_one_thread(args.workload, args.cpu_seconds / 2)
    plan_us, plan_binding_us = plan_host_us(db, layout, sms)
    try:                        # an auxiliary host figure: never costs the line
        build_us = builder_host_us(layout)
    except Exception as e:      # noqa: BLE001
        build_us = f"failed: {e}"
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": n,
        "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": args.workload, "num_q_heads": sh.num_q_heads,
                   "num_kv_heads": sh.num_kv_heads, "head_dim": sh.head_dim,
                   "page_size": sh.page_size, "sliding_window": sh.sliding_window,
                   "tokens_per_step": T,
                   "decode_rows": int((layout.q_len == 1).sum()),
                   "chunk_rows": int((layout.q_len > 1).sum()),
                   "kv_bytes_per_step": cnt["bytes"],
                   "l2": "inputs larger than L2 (KV read per step %.0f MB > 129 MB)" % (cnt["bytes"] / 1e6),
                   "parallelism": f"replicas{n}" if n > 1 else "single"},
        "roofline": roof,
        "step_roofline": {"frac": (step_roof_s * 1e3) / ms_step,
                          "roofline_ms": step_roof_s * 1e3,
                          "flops": cnt["flops"], "bytes": cnt["bytes"],
                          "bound": "hbm" if cnt["bytes"] / (peaks["hbm_gbs"] * 1e9) >=
                          cnt["flops"] / (peaks["bf16_tflops"] * 1e12) else "tensor"},
        "cpu_baseline": {"value": cpu_v, "unit": "tokens/s",
                         "cores": len(os.sched_getaffinity(0)), "kind": "oracle",
                         "sample": cpu_desc,
                         "one_thread": {"value": cpu1_v, "unit": "tokens/s", "cores": 1,
                                        "sample": cpu1_desc}},
        "plan_host_us": plan_us,
        "plan_binding_us": plan_binding_us,
        "builder_host_us": build_us,
        "e2e": e2e,
        "gpu_launches": int(launches),
        "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)


SWEEP_CHUNKS = (256, 257, 512, 1024, 2048, 8192)


def run_seed_sweep(args):
    """The workload's batch drawn with seeds 0..4 (lengths, page permutation
    and tensor contents): tokens/s and the attention launch's roofline
    fraction per seed (append + attention back to back, inputs larger than
    L2), one JSON line per seed and a summary line."""
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    import __graft_entry__
    __graft_entry__.build()
    from chunked_prefill_decode_gb300 import hb
    from chunked_prefill_decode_gb300.device import device_batch

    peaks = _peaks()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    stream = torch.cuda.current_stream(dev)
    steps = max(10, min(args.steps, 500))
    rows = []
    with ClockSampler(0) as clk:
        for seed in range(5):
            lay = workloads.WORKLOADS[args.workload](seed)
            sh = lay.shape
            ten = workloads.make_tensors(lay, seed=seed, device=dev)
            db = device_batch(lay.q_len, lay.context_len, lay.block_table, lay.num_pages,
                              sh.num_q_heads, sh.num_kv_heads, sh.head_dim, sh.page_size, dev,
                              sliding_window=sh.sliding_window)
            plan, ws = hb.hb_plan(db.batch, db.q_len, db.context_len, sms)
            out = torch.empty_like(ten.q)
            scale = 1.0 / math.sqrt(sh.head_dim)

            def step():
                hb.hb_kv_append(db.batch, ten.k_new, ten.v_new, ten.k_cache, ten.v_cache)
                hb.hb_attention_new_kv(db.batch, plan, ten.q, ten.k_new, ten.v_new, ten.k_cache,
                                       ten.v_cache, scale, out, ws)
            for _ in range(max(args.warmup, 3)):
                step()
            torch.cuda.synchronize(dev)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(steps):
                step()
            e1.record(stream)
            torch.cuda.synchronize(dev)
            hb.hb_check()
            ms = e0.elapsed_time(e1) / steps
            cnt = algorithmic_counts(lay)
            step_roof = max(cnt["flops"] / (peaks["bf16_tflops"] * 1e12),
                            cnt["bytes"] / (peaks["hbm_gbs"] * 1e9)) * 1e3
            r = {"sweep": "seed", "workload": args.workload, "seed": seed,
                 "tokens_per_step": lay.total_q, "ms_per_step": ms,
                 "tokens_per_s": lay.total_q / (ms * 1e-3), "step_roofline_frac": step_roof / ms,
                 "kv_bytes": cnt["bytes"], "flops": cnt["flops"]}
            rows.append(r)
            print(json.dumps(r), flush=True)
    v = [r["tokens_per_s"] for r in rows]
    f = [r["step_roofline_frac"] for r in rows]
    print(json.dumps({"sweep": "seed", "workload": args.workload, "seeds": 5, "steps": steps,
                      "tokens_per_s": {"mean": statistics.mean(v), "min": min(v), "max": max(v)},
                      "step_roofline_frac": {"mean": statistics.mean(f), "min": min(f), "max": max(f)},
                      "clocks": clk.summary()}), flush=True)


def run_chunk_sweep(args):
    """Prefill of one 8192-token prompt in chunks of c tokens, each chunk in a
    hybrid batch with 32 decode rows at context 2048, and the same chunks
    alone.  Per c: the summed step time over all chunks of the prompt (append
    + attention, L2 flushed before every timed step, median over repetitions),
    the chunk work's FLOPs and the KV bytes its re-reads of earlier chunks
    cost.  One JSON line per chunk size; c = 8192 is the unchunked prefill."""
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    import __graft_entry__
    __graft_entry__.build()
    from chunked_prefill_decode_gb300 import hb
    from chunked_prefill_decode_gb300.device import device_batch

    peaks = _peaks()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    reps = max(3, args.sweep_reps)

    def time_layout(lay):
        sh = lay.shape
        ten = workloads.make_tensors(lay, seed=7, device=dev)
        db = device_batch(lay.q_len, lay.context_len, lay.block_table, lay.num_pages,
                          sh.num_q_heads, sh.num_kv_heads, sh.head_dim, sh.page_size, dev)
        plan, ws = hb.hb_plan(db.batch, db.q_len, db.context_len, sms)
        out = torch.empty_like(ten.q)
        scale = 1.0 / math.sqrt(sh.head_dim)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(reps + 3)]
        for e0, e1 in evs:
            flush.fill_(1)
            e0.record(stream)
            hb.hb_kv_append(db.batch, ten.k_new, ten.v_new, ten.k_cache, ten.v_cache)
            hb.hb_attention_new_kv(db.batch, plan, ten.q, ten.k_new, ten.v_new, ten.k_cache,
                                   ten.v_cache, scale, out, ws)
            e1.record(stream)
        torch.cuda.synchronize(dev)
        hb.hb_check()
        return statistics.median(e0.elapsed_time(e1) for e0, e1 in evs[3:])

    rows = []
    chunks = SWEEP_CHUNKS if not args.sweep_chunks else tuple(args.sweep_chunks)
    with ClockSampler(0) as clk:
        for c in chunks:
            n_chunks = -(-8192 // c)
            iters = range(n_chunks) if args.sweep_iters is None else \
                [i for i in args.sweep_iters if i < n_chunks]
            r = {"sweep": "chunk", "chunk": c, "n_chunks": n_chunks, "prefill_ms_with_decodes": 0.0,
                 "prefill_ms_chunk_only": 0.0, "chunk_flops": 0, "chunk_kv_bytes": 0,
                 "iterations": []}
            for i in iters:
                alone = workloads.chunk_sweep(c, i, n_decode=0)
                cnt = algorithmic_counts(alone)
                t_alone = time_layout(alone)
                t_dec = time_layout(workloads.chunk_sweep(c, i)) if not args.sweep_chunk_only else 0.0
                r["chunk_flops"] += cnt["chunk_flops"]
                r["chunk_kv_bytes"] += cnt["chunk_bytes"]
                r["prefill_ms_chunk_only"] += t_alone
                r["prefill_ms_with_decodes"] += t_dec
                r["iterations"].append({"index": i, "ms_chunk_only": t_alone, "ms_with_decodes": t_dec,
                                        "chunk_kv_bytes": cnt["chunk_bytes"],
                                        "chunk_flops": cnt["chunk_flops"]})
            t = r["prefill_ms_chunk_only"] * 1e-3
            r["chunk_only_tflops"] = r["chunk_flops"] / t / 1e12
            r["chunk_only_tc_frac"] = r["chunk_only_tflops"] / peaks["bf16_tflops"]
            r["decode_ms_per_iteration"] = (r["prefill_ms_with_decodes"] -
                                            r["prefill_ms_chunk_only"]) / n_chunks
            rows.append(r)
    base = rows[-1]
    clocks = clk.summary()
    for r in rows:
        r["chunk_only_vs_unchunked"] = r["prefill_ms_chunk_only"] / max(base["prefill_ms_chunk_only"], 1e-12)
        r["with_decodes_vs_unchunked"] = (r["prefill_ms_with_decodes"] /
                                          max(base["prefill_ms_with_decodes"], 1e-12))
        r["peak"] = {"bf16_tflops": peaks["bf16_tflops"], "source": peaks["source"]}
        r["l2"] = "flushed before every timed step (%d MB written)" % (flush.numel() >> 20)
        r["reps"] = reps
        r["clocks"] = clocks
        print(json.dumps(r), flush=True)


def run_layer(args):
    """One transformer block of the workload's hybrid batch (linear layers
    around the attention step, synthetic weights) timed on the device: QKV
    projection, KV append, attention, output projection, gated MLP and down
    projection, all in this library's kernels.  One JSON line."""
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    import __graft_entry__
    __graft_entry__.build()
    from chunked_prefill_decode_gb300 import hb, layer
    from chunked_prefill_decode_gb300.device import from_layout

    lay = workloads.WORKLOADS[args.workload]()
    sh = lay.shape
    bshape = {32: layer.MISTRAL_7B, 56: layer.YI_34B}.get(sh.num_q_heads)
    if bshape is None or sh.head_dim != 128:
        raise SystemExit("--layer supports the Mistral-7B and Yi-34B attention shapes")
    blk = layer.HybridBlock(bshape, seed=1)
    ten = workloads.make_tensors(lay, seed=1, device=dev)
    db = from_layout(lay)
    T = lay.total_q
    x = torch.randn(T, bshape.hidden, device=dev).to(torch.bfloat16)
    bufs = blk.buffers(T)
    for _ in range(max(args.warmup, 3)):
        blk.forward(x, db, ten.k_cache, ten.v_cache, bufs=bufs, plan=False)
    torch.cuda.synchronize(dev)
    hb.hb_check()
    steps = max(1, min(args.steps, 500))
    hb.hb_timing_enable(True)
    hb.hb_timing_enable(False)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n_sampled = 0
    with ClockSampler(0) as clk:
        ev0.record()
        for i in range(steps):
            sampled = i % TIMING_EVERY == 0
            if sampled:
                hb.hb_timing_enable(True, keep=True)
                n_sampled += 1
            blk.forward(x, db, ten.k_cache, ten.v_cache, bufs=bufs, plan=False)
            if sampled:
                hb.hb_timing_enable(False)
        ev1.record()
        torch.cuda.synchronize(dev)
    kt = hb.hb_timing_read()
    hb.hb_check()
    ms = ev0.elapsed_time(ev1) / steps
    peaks = _peaks()
    lin_ms = kt["linear"][0] / n_sampled
    lin_flops = blk.flops(T)
    weight_bytes = 2.0 * bshape.params()
    line = {
        "mode": "layer", "workload": args.workload, "tokens_per_step": T, "steps": steps,
        "ms_per_step": ms, "tokens_per_s": T / (ms * 1e-3),
        "ms_by_kernel": {k: v[0] / n_sampled for k, v in kt.items()},
        "launches_per_step": {k: v[1] / n_sampled for k, v in kt.items()},
        "linear": {"flops": lin_flops, "weight_bytes": weight_bytes,
                   "tflops": lin_flops / (lin_ms * 1e-3) / 1e12,
                   "roofline_ms": max(lin_flops / (peaks["bf16_tflops"] * 1e12),
                                      weight_bytes / (peaks["hbm_gbs"] * 1e9)) * 1e3},
        "attention_share": (kt["attention"][0] + kt["kv_append"][0]) / n_sampled / ms,
        "kernel_timing": f"CUDA events around each launch of every {TIMING_EVERY}th timed step",
        "block": {"hidden": bshape.hidden, "ffn": bshape.ffn, "params": bshape.params()},
        "weights": "synthetic N(0, 1/fan_in)", "data": "synthetic", "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="yi_b2048", choices=sorted(workloads.WORKLOADS))
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--sweep", choices=["chunk", "seed"], default=None,
                    help="instead of the step benchmark: 'chunk' prefills one 8192-token "
                         "prompt in chunks of 256/257/512/1024/2048/8192 tokens; 'seed' draws "
                         "the workload's batch with seeds 0..4")
    ap.add_argument("--sweep-reps", type=int, default=10)
    ap.add_argument("--sweep-chunks", type=int, nargs="+", default=None,
                    help="chunk sweep: only these chunk sizes (the ratios are then relative "
                         "to the last size given)")
    ap.add_argument("--sweep-iters", type=int, nargs="+", default=None,
                    help="chunk sweep: only these iterations (chunk indices) of each size")
    ap.add_argument("--sweep-chunk-only", action="store_true",
                    help="chunk sweep: skip the iterations with decode rows beside the chunk")
    ap.add_argument("--e2e-stages", type=int, default=2,
                    help="staging buffers of the end-to-end loop (steps whose copies may be "
                         "in flight at once)")
    ap.add_argument("--layer", action="store_true",
                    help="instead of the attention step: one transformer block of the "
                         "batch (linear layers on synthetic weights around attention)")
    ap.add_argument("--oracle-sample", action="store_true", help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.oracle_sample:
        run_oracle_sample(args)
        return
    rc = replica_launch(args.gpus, sys.argv[1:])
    if rc is not None:
        sys.exit(rc)
    if args.sweep == "chunk":
        run_chunk_sweep(args)
    elif args.sweep == "seed":
        run_seed_sweep(args)
    elif args.layer:
        run_layer(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_native(args)
    if torch.distributed.is_initialized():
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
