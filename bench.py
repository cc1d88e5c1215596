#!/usr/bin/env python3
"""Benchmark: GDN decode tokens/s per layer and achieved HBM GB/s on one GB300.

Headline workload: the Qwen3.5-shaped GDN layer (16 QK heads, 32 V heads,
dk = dv = 128, conv width 4 over 8192 channels, bf16 activations and conv
history, fp32 state), batch 64, over a 512-slot pool.  One step = one
gdn_decode_step launch (conv1d update + SiLU + L2 norm + gates + gated delta
rule + readout for 64 requests).  Consecutive steps rotate over 8 disjoint
64-slot sets of the pool, so the state touched between two visits of a slot
(1.1 GB) is far larger than the 129 MB L2: every step streams its state from
HBM.

The other hot-path rows (batch sweep, speculative verify + commit, chunked
prefill, slot copy / zero) are timed after the headline and reported under
"rows"; they are not part of the headline number.

`--impl reference` times the CPU oracle (the reference arm of this build).
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
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "GDN decode tokens/s per layer & achieved HBM GB/s (% of roofline), 1×GB300"
UNIT = "tokens/s"
B_HEAD = 64
SETS = 8
POOL = 512

# bytes per decode token, Qwen3.5-shaped layer (bf16 activations / history):
#   state 2 x 32 x 128 x 128 x 4, conv history 2 x 3 x 8192 x 2, qkv 8192 x 2,
#   a and b 2 x 32 x 2, out 32 x 128 x 2, slot id 4
DECODE_TOKEN_BYTES = 2 * 2097152 + 2 * 49152 + 16384 + 128 + 8192 + 4
DECODE_STEP_PARAM_BYTES = 8192 * 4 * 4 + 2 * 32 * 4

# ncu DRAM traffic (read + write bytes per launch) of the decode kernel on the
# headline workload itself (profiles/decode_tma_kernel_b64_pool512_dram.md),
# with the sha256 of the kernel's sources (DECODE_SOURCES) it was captured on;
# reported only while they are unchanged.
DECODE_TRAFFIC = {
    "bytes_per_launch": 138596096 + 76754432,
    "source_sha256": "42d6dd52e9e6106fe1c06ee851ae482d4de2862e4f71eb27aef542749b838bd3",
    "case": "batch 64 over the 512-slot pool with the headline's 8-set rotation, the sixth launch "
            "(ncu dram__bytes_read.sum + dram__bytes_write.sum, one pass): reads are exactly the algorithmic "
            "138.6 MB; part of the 134 MB of state written is still in L2 when the launch ends and leaves it "
            "during the next launches, so the launch's own DRAM writes are 77 MB",
}


def _sha(*paths):
    """sha256 of the files' contents, in order."""
    h = hashlib.sha256()
    for path in paths:
        with open(path, "rb") as f:
            h.update(f.read())
    return h.hexdigest()


# the sources of the headline decode kernel
DECODE_SOURCES = [os.path.join("hybrid_linear_attention_gdn_gb300", "csrc", f)
                  for f in ("decode_tma.cu", "decode_tma_item.cuh", "gdn_common.cuh")]


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d.get("hbm_gbs", 6800.0), d.get("bf16_tflops", 1900.0), d.get(
            "bf16_tflops_sustained", 1700.0), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled in the background."""

    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self, t_lo: float, t_hi: float):
        """Summary of the samples taken between wall times t_lo and t_hi."""
        import datetime
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        lines = self.file.read().splitlines()
        os.unlink(self.file.name)
        win = []
        for ln in lines:
            r = [x.strip() for x in ln.split(",")]
            if len(r) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(r[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                sm, mx = float(r[2]), float(r[3])
            except ValueError:
                continue
            if t_lo - 0.15 <= ts <= t_hi + 0.15:
                win.append((sm, mx, r[6:10]))
        reasons = sorted({n for _, _, rs in win for n, v in zip(self.REASONS, rs)
                          if v.lower() == "active"})
        return {"sm_mhz": statistics.median(w[0] for w in win) if win else None,
                "sm_max_mhz": max(w[1] for w in win) if win else None,
                "reasons": reasons, "samples": len(win)}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def reduce_max(value: float, device=None) -> float:
    """Maximum of `value` over the ranks of the default process group (the
    value itself when there is no group or one rank)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, world: int, ms_max: float) -> float:
    """Units processed by all ranks per second, timed by the slowest rank."""
    return world * units_per_rank / (ms_max * 1e-3)


def headline_config(n_slots: int, n_sets: int, ws: int) -> dict:
    return {"workload": f"qwen35_gdn_decode_b64_h16x32_d128_pool{n_slots}",
            "batch": B_HEAD, "pool_slots": n_slots,
            "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU",
            "l2": f"inputs larger than L2: steps rotate over {n_sets} disjoint 64-slot "
                  f"sets ({n_sets * 0.137:.2f} GB of state between visits of a slot)",
            "activations": "bf16", "state": "fp32"}


# --------------------------------------------------------------- reference arm

def run_reference(args):
    """The oracle on the host cores, same metric and workload, bounded sample."""
    ws, rank, _ = _dist()
    if rank != 0:
        return
    import numpy as np
    import oracle
    from hybrid_linear_attention_gdn_gb300 import synth
    shape = synth.QWEN
    g = synth.generator(1)
    conv_w, A_log, dt_bias = synth.params(shape, g)
    sample_b = 8  # requests per reference step (a bounded sample of the 64)
    ssm, conv = synth.pool(shape, g, sample_b)
    od = oracle.Dims(shape.hk, shape.hv, shape.dk, shape.dv, shape.w)
    op = oracle.Params(conv_w.double().numpy(), A_log.double().numpy(), dt_bias.double().numpy())
    pool = oracle.Pool(ssm.double().numpy(), conv.double().numpy())
    ids = np.arange(sample_b, dtype=np.int32)
    qkv, a, b = synth.tokens(shape, g, (sample_b,))
    qkv, a, b = (t.double().numpy() for t in (qkv, a, b))
    for _ in range(args.warmup):
        oracle.decode_step(od, pool, op, ids, qkv, a, b)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.decode_step(od, pool, op, ids, qkv, a, b)
    dt = time.perf_counter() - t0
    value = sample_b * args.steps / dt
    cores = oracle.num_threads()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": headline_config(POOL, SETS, ws),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"each step a bounded sample: {sample_b} of the {B_HEAD} "
                                   f"requests, double precision; {args.steps} steps"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------- our arm

def _events_time(fn, reps, stream):
    import torch
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for i in range(reps):
        fn(i)
    e1.record(stream)
    e1.synchronize()
    return e0.elapsed_time(e1) / reps  # ms


def _cpu_baseline(budget_s=12.0):
    """The oracle as it stands, on the host cores, on a bounded sample."""
    import numpy as np
    import oracle
    from hybrid_linear_attention_gdn_gb300 import synth
    shape = synth.QWEN
    g = synth.generator(7)
    conv_w, A_log, dt_bias = synth.params(shape, g)
    B = B_HEAD
    ssm, conv = synth.pool(shape, g, B)
    od = oracle.Dims(shape.hk, shape.hv, shape.dk, shape.dv, shape.w)
    op = oracle.Params(conv_w.double().numpy(), A_log.double().numpy(), dt_bias.double().numpy())
    pool = oracle.Pool(ssm.double().numpy(), conv.double().numpy())
    ids = np.arange(B, dtype=np.int32)
    qkv, a, b = (t.double().numpy() for t in synth.tokens(shape, g, (B,)))
    oracle.decode_step(od, pool, op, ids, qkv, a, b)  # warm
    steps, t0 = 0, time.perf_counter()
    while True:
        oracle.decode_step(od, pool, op, ids, qkv, a, b)
        steps += 1
        dt = time.perf_counter() - t0
        if dt > budget_s:
            break
    return {"value": B * steps / dt, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{steps} decode steps of the batch-64 workload ({B * steps} tokens), "
                      f"{dt:.1f} s"}


def run_ours(args):
    import torch
    import hybrid_linear_attention_gdn_gb300 as gdn
    from hybrid_linear_attention_gdn_gb300 import synth

    ws, rank, local = _dist()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    gdn.load()
    hbm_peak, bf16_peak, bf16_sust, peak_src = _peaks()
    shape = synth.QWEN
    dims = gdn.Dims.of(shape)
    g = synth.generator(1000 + rank)
    conv_w, A_log, dt_bias = synth.params(shape, g)
    params = gdn.LayerParams(conv_w.to(dev), A_log.to(dev), dt_bias.to(dev))
    n_slots = args.pool
    ssm, conv = synth.pool(shape, g, n_slots)
    pool = gdn.StatePool(ssm.to(dev), conv.to(dev))
    del ssm, conv
    perm = torch.randperm(n_slots, generator=g).to(torch.int32)
    n_sets = max(1, min(SETS, n_slots // B_HEAD))
    id_sets = [perm[k * B_HEAD:(k + 1) * B_HEAD].to(dev) for k in range(n_sets)]
    inputs = [tuple(t.to(dev) for t in synth.tokens(shape, g, (B_HEAD,))) for _ in range(n_sets)]
    out = torch.empty((B_HEAD, shape.hv, shape.dv), dtype=shape.act_dtype, device=dev)
    stream = torch.cuda.current_stream()

    def step(i):
        q, a, b = inputs[i % n_sets]
        gdn.decode_step(dims, pool, params, id_sets[i % n_sets], q, a, b, out)

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    # make sure the clock sampler sees a loaded window even for short runs
    t_soak = time.time()
    while not args.no_soak and time.time() - t_soak < 1.0:
        for i in range(200):
            step(i)
        torch.cuda.synchronize()
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    n0 = sum(gdn.launch_counts())
    t_lo = time.time()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        step(i)
    e1.record(stream)
    e1.synchronize()
    torch.cuda.synchronize()
    t_hi = time.time()
    launches = sum(gdn.launch_counts()) - n0
    ms = reduce_max(e0.elapsed_time(e1), dev)
    clocks = sampler.stop(min(t_soak, t_lo), t_hi)
    ms_step = ms / args.steps
    tok_s = whole_job_rate(B_HEAD * args.steps, ws, ms)
    step_bytes = B_HEAD * DECODE_TOKEN_BYTES + DECODE_STEP_PARAM_BYTES
    achieved = step_bytes / (ms_step * 1e-3) / 1e9
    # per-step distribution: a separate pass after the timed one, an event
    # around every step (the events themselves add a little to each step)
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    evs[0].record(stream)
    for i in range(args.steps):
        step(i)
        evs[i + 1].record(stream)
    evs[-1].synchronize()
    per_step = sorted(evs[i].elapsed_time(evs[i + 1]) for i in range(args.steps))

    def pct(q):
        return per_step[min(len(per_step) - 1, int(q * (len(per_step) - 1) + 0.5))]
    step_stats = {"median": statistics.median(per_step), "p10": pct(0.10), "p90": pct(0.90),
                  "how": "separate pass, CUDA events around each step"}
    srcs = [os.path.join(ROOT, f) for f in DECODE_SOURCES]
    traffic = DECODE_TRAFFIC["bytes_per_launch"] if DECODE_TRAFFIC["source_sha256"] == _sha(*srcs) else None

    # ---- end to end through the public API with host buffers: every step's
    # inputs are copied in from pinned host memory and its output read back,
    # all inside the timed region.  As a serving loop would run it, step i+1's
    # upload and step i-1's read-back overlap step i's kernel (two copy
    # streams, double-buffered device inputs and outputs).
    # one pinned byte buffer per input set: [qkv | a | b | slot ids], 256-byte
    # aligned parts, so a step's upload is a single copy
    parts = list(inputs[0]) + [id_sets[0]]
    offs, o = [], 0
    for t in parts:
        offs.append(o)
        o += (t.numel() * t.element_size() + 255) // 256 * 256
    packed_bytes = o

    def pack(ts):
        buf = torch.empty(packed_bytes, dtype=torch.uint8).pin_memory()
        for t, off in zip(ts, offs):
            nb = t.numel() * t.element_size()
            buf[off:off + nb].copy_(t.cpu().contiguous().view(torch.uint8).reshape(-1))
        return buf

    pin = [pack(list(inp) + [ids]) for inp, ids in zip(inputs, id_sets)]
    d_raw = [torch.empty(packed_bytes, dtype=torch.uint8, device=dev) for _ in range(2)]
    d_in = [tuple(raw[off:off + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
                  for t, off in zip(parts, offs)) for raw in d_raw]
    out_host = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
    d_out = [torch.empty_like(out) for _ in range(2)]
    s_up, s_down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]    # inputs of buffer k uploaded
    ev_used = [torch.cuda.Event() for _ in range(2)]  # kernel done with buffer k
    ev_out = [torch.cuda.Event() for _ in range(2)]   # output of buffer k read back
    h2d = sum(t.numel() * t.element_size() for t in parts)
    d2h = out_host[0].numel() * out_host[0].element_size()

    def upload(i):
        k = i % 2
        with torch.cuda.stream(s_up):
            s_up.wait_event(ev_used[k])
            d_raw[k].copy_(pin[i % n_sets], non_blocking=True)
            ev_in[k].record(s_up)

    def e2e_run(n):
        start = torch.cuda.Event()
        start.record(stream)
        s_up.wait_event(start)
        upload(0)
        for i in range(n):
            k = i % 2
            stream.wait_event(ev_in[k])
            stream.wait_event(ev_out[k])
            q, a, b, ids = d_in[k]
            gdn.decode_step(dims, pool, params, ids, q, a, b, d_out[k], stream=stream)
            ev_used[k].record(stream)
            if i + 1 < n:
                upload(i + 1)
            with torch.cuda.stream(s_down):
                s_down.wait_event(ev_used[k])
                out_host[k].copy_(d_out[k], non_blocking=True)
                ev_out[k].record(s_down)
        stream.wait_event(ev_out[(n - 1) % 2])

    e2e_run(args.warmup)
    torch.cuda.synchronize()
    if ws > 1:
        torch.distributed.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    e2e_run(args.steps)
    e1.record(stream)
    e1.synchronize()
    e2e_ms = reduce_max(e0.elapsed_time(e1) / args.steps, dev)
    e2e = {"value": whole_job_rate(B_HEAD, ws, e2e_ms), "unit": UNIT, "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h, "overlap": "uploads and read-backs on two copy streams beside the kernel"}

    rows = {} if args.no_rows else measure_rows(gdn, synth, dev, stream, hbm_peak, bf16_peak,
                                                args.rows, args.prefill_len)

    if rank != 0:
        return
    cpu = None if (ws > 1 or args.no_cpu) else _cpu_baseline()
    line = {
        "metric": METRIC, "value": tok_s, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "step_ms": step_stats, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": headline_config(n_slots, n_sets, ws),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                     "frac": achieved / hbm_peak, "traffic": traffic,
                     "traffic_case": DECODE_TRAFFIC["case"] if traffic else None,
                     "kernel": "decode_tma_kernel<bf16,bf16,10>",
                     "algorithmic_bytes_per_launch": step_bytes, "peak_source": peak_src},
        "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches, "clocks": clocks,
        "rows": rows,
    }
    print(json.dumps(line), flush=True)


def _graph_time(f, n_steps, n_replays, dev):
    """ms per step of n_steps calls of f captured in one CUDA graph (None if
    the capture is refused)."""
    import torch
    try:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(n_steps):
                f(i)
        g.replay()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(n_replays):
            g.replay()
        e1.record()
        e1.synchronize()
        return e0.elapsed_time(e1) / (n_steps * n_replays)
    except RuntimeError:
        return None


ROW_GROUPS = ("all", "sweep", "slots", "verify", "prefill", "kda_decode", "kda_verify", "kda_prefill",
              "mixed", "epilogue")


def measure_rows(gdn, synth, dev, stream, hbm_peak, bf16_peak, which="all", prefill_len=8192):
    """Every other row of the hot path, timed with CUDA events (not headline).
    which: "all", or one group of ROW_GROUPS alone (for profiling one kernel;
    prefill_len sets the tokens per sequence of both 4-sequence prefills)."""
    import torch
    shape = synth.QWEN
    dims = gdn.Dims.of(shape)
    g = synth.generator(77)
    conv_w, A_log, dt_bias = synth.params(shape, g)
    params = gdn.LayerParams(conv_w.to(dev), A_log.to(dev), dt_bias.to(dev))
    ssm, conv = synth.pool(shape, g, POOL)
    pool = gdn.StatePool(ssm.to(dev), conv.to(dev))
    del ssm, conv
    rows = {}
    reps = 50

    def frac(nbytes, ms):
        gbs = nbytes / (ms * 1e-3) / 1e9
        return {"ms": ms, "algorithmic_GBps": gbs, "frac_hbm": gbs / hbm_peak}

    def want(group):
        return which in ("all", group)

    # batch sweep (state rotates over POOL // B disjoint sets where possible)
    sweep = {}
    for B in ([1, 2, 4, 8, 16, 32, 64, 128, 256] if want("sweep") else []):
        nsets = max(1, min(8, POOL // B))
        perm = torch.randperm(POOL, generator=g).to(torch.int32)
        sets = [perm[k * B:(k + 1) * B].to(dev) for k in range(nsets)]
        inp = [tuple(t.to(dev) for t in synth.tokens(shape, g, (B,))) for _ in range(nsets)]
        out = torch.empty((B, 32, 128), dtype=torch.bfloat16, device=dev)

        def f(i, sets=sets, inp=inp, out=out):
            q, a, b = inp[i % len(sets)]
            gdn.decode_step(dims, pool, params, sets[i % len(sets)], q, a, b, out)
        for i in range(10):
            f(i)
        ms = _events_time(f, reps, stream)
        r = frac(B * DECODE_TOKEN_BYTES + DECODE_STEP_PARAM_BYTES, ms)
        r["tokens_per_s"] = B / (ms * 1e-3)
        # the same steps replayed from a CUDA graph: the GPU-side time per step
        # without the per-call host cost (what a graph-captured serving loop sees)
        r["ms_graph"] = _graph_time(f, 20, 10, dev)
        sweep[str(B)] = r
    if sweep:
        rows["decode_sweep"] = sweep

    slot_bytes = 2097152 + 49152
    perm = torch.randperm(POOL, generator=g).to(torch.int32)
    pair_sets = [(perm[k * 128:k * 128 + 64].to(dev), perm[k * 128 + 64:(k + 1) * 128].to(dev))
                 for k in range(4)]

    def slot_rows():
        def fc(i):
            s, d = pair_sets[i % 4]
            gdn.slot_copy(dims, pool, pool, s, d)
        fc(0)
        rows["slot_copy_64"] = frac(64 * 2 * slot_bytes, _events_time(fc, reps, stream))

        def fz(i):
            gdn.slot_zero(dims, pool, pair_sets[i % 4][1])
        fz(0)
        rows["slot_zero_64"] = frac(64 * slot_bytes, _events_time(fz, reps, stream))

        # state pack / unpack of 64 slots through one contiguous staging buffer
        rec = gdn.state_record_bytes(dims)
        staging = torch.empty(64 * rec, dtype=torch.uint8, device=dev)

        def fpk(i):
            gdn.state_pack(dims, pool, pair_sets[i % 4][0], staging)
        fpk(0)
        rows["state_pack_64"] = frac(64 * 2 * rec, _events_time(fpk, reps, stream))

        def fup(i):
            gdn.state_unpack(dims, staging, pool, pair_sets[i % 4][1])
        fup(0)
        rows["state_unpack_64"] = frac(64 * 2 * rec, _events_time(fup, reps, stream))
        del staging

    def spec_rows():
        # speculative verify, batch 16, T = 8, spec cache of 16 x 8 slots, then commit
        B, T = 16, 8
        spec = gdn.StatePool.empty(dims, 4 * B * T, dev)
        spec_sets = [torch.arange(k * B * T, (k + 1) * B * T, dtype=torch.int32,
                                  device=dev).reshape(B, T) for k in range(4)]
        work_sets = [perm[k * B:(k + 1) * B].to(dev) for k in range(4)]
        vin = [tuple(t.to(dev) for t in synth.tokens(shape, g, (B, T))) for _ in range(4)]
        vout = torch.empty((B, T, 32, 128), dtype=torch.bfloat16, device=dev)
        L = synth.accept_lengths(B, T, g).to(dev)

        def fv(i):
            q, a, b = vin[i % 4]
            gdn.spec_verify(dims, pool, spec, params, work_sets[i % 4], spec_sets[i % 4], q, a, b,
                            vout)
        fv(0)
        vbytes = B * (slot_bytes + T * (16384 + 128) + T * slot_bytes + T * 8192)
        r = frac(vbytes, _events_time(fv, reps, stream))
        r["draft_tokens_per_s"] = B * T / (r["ms"] * 1e-3)
        rows["spec_verify_b16_t8"] = r

        def fm(i):
            gdn.spec_commit(dims, spec, pool, spec_sets[i % 4], L, work_sets[i % 4])
        fm(0)
        rows["spec_commit_b16"] = frac(B * 2 * slot_bytes, _events_time(fm, reps, stream))
        del spec

        # index-update commit of the same batch: only int32 indices move
        idx_slots = work_sets[0].clone()
        freed = torch.empty((B, T), dtype=torch.int32, device=dev)

        def fi(i):
            gdn.spec_commit_index(spec_sets[i % 4], L, idx_slots, freed)
        fi(0)
        ms_i = _events_time(fi, reps, stream)
        rows["spec_commit_index_b16"] = {"ms": ms_i, "ms_graph": _graph_time(fi, 20, 10, dev),
                                         "bytes_moved": B * (T + 1 + 2 * T + 2) * 4}

        # verify at larger batches (T = 8), two alternating request / spec-cache sets
        vsweep = {}
        for Bv in (32, 64, 128):
            spec_v = gdn.StatePool.empty(dims, 2 * Bv * T, dev)
            ss = [torch.arange(k * Bv * T, (k + 1) * Bv * T, dtype=torch.int32, device=dev).reshape(Bv, T)
                  for k in range(2)]
            ws_ = [perm[k * Bv:(k + 1) * Bv].to(dev) for k in range(2)]
            vi = [tuple(t.to(dev) for t in synth.tokens(shape, g, (Bv, T))) for _ in range(2)]
            vo = torch.empty((Bv, T, 32, 128), dtype=torch.bfloat16, device=dev)

            def fvb(i, spec_v=spec_v, ss=ss, ws_=ws_, vi=vi, vo=vo):
                q, a, b = vi[i % 2]
                gdn.spec_verify(dims, pool, spec_v, params, ws_[i % 2], ss[i % 2], q, a, b, vo)
            fvb(0)
            nb = Bv * (slot_bytes + T * (16384 + 128) + T * slot_bytes + T * 8192)
            rv = frac(nb, _events_time(fvb, reps, stream))
            rv["draft_tokens_per_s"] = Bv * T / (rv["ms"] * 1e-3)
            vsweep[str(Bv)] = rv
            del spec_v
            torch.cuda.empty_cache()
        rows["spec_verify_sweep_t8"] = vsweep

    def prefill_row():
        # chunked prefill: 4 sequences x prefill_len tokens, checkpoints every 256
        n_seq, S = 4, prefill_len
        total = n_seq * S
        qkv, a, b = (t.to(dev) for t in synth.tokens(shape, g, (total,)))
        cu = torch.arange(0, total + 1, S, dtype=torch.int32, device=dev)
        sp = torch.zeros(n_seq, dtype=torch.int64, device=dev)
        n_ck = S // 256
        ck = gdn.StatePool.empty(dims, 4 * n_ck, dev)
        ck_ids = torch.arange(4 * n_ck, dtype=torch.int32, device=dev).reshape(4, n_ck)
        pout = torch.empty((total, 32, 128), dtype=torch.bfloat16, device=dev)
        wsb = gdn.chunk_prefill_workspace_size(dims, n_seq, total)
        wsp = torch.empty(wsb, dtype=torch.uint8, device=dev)
        pids = [perm[k * 4:(k + 1) * 4].to(dev) for k in range(4)]

        def fp(i):
            gdn.chunk_prefill(dims, pool, ck, params, pids[i % 4], cu, sp, total, ck_ids, 256, qkv, a,
                              b, pout, wsp)
        fp(0)
        pms = _events_time(fp, 5, stream)
        # qkv, a, b and out per token; checkpoints plus each sequence's state read and written
        pbytes = total * (16384 + 128 + 8192) + (4 * n_ck + 8) * slot_bytes
        # ~11.7 MFLOP per (64-token chunk, V head) for the chunk form
        pflop = total / 64 * 32 * 11.7e6
        rows[f"chunk_prefill_4x{S}"] = {
            "ms": pms, "tokens_per_s": total / (pms * 1e-3),
            "algorithmic_GBps": pbytes / (pms * 1e-3) / 1e9,
            "frac_hbm": pbytes / (pms * 1e-3) / 1e9 / hbm_peak,
            "TFLOPs": pflop / (pms * 1e-3) / 1e12,
            "frac_bf16_peak": pflop / (pms * 1e-3) / 1e12 / bf16_peak,
            "workspace_bytes": wsb}
        # the same prefill with the readout epilogue (gated RMS norm): fused
        # into the prefill's output, against the prefill then the epilogue
        z = synth.normal((total, 32, 128), 1.5, g, shape.act_dtype).to(dev)
        nw = torch.ones(128, dtype=torch.float32, device=dev)

        def fg(i):
            gdn.chunk_prefill_gated(dims, pool, ck, params, pids[i % 4], cu, sp, total, ck_ids, 256, qkv, a,
                                    b, z, nw, 1e-6, pout, wsp)

        def fs(i):
            fp(i)
            gdn.gated_rmsnorm(dims, pout, z, nw, 1e-6)
        fg(0)
        fs(0)
        rows[f"chunk_prefill_gated_4x{S}"] = {"ms_fused": _events_time(fg, 5, stream),
                                              "ms_prefill_then_epilogue": _events_time(fs, 5, stream)}
        del qkv, a, b, pout, wsp, z
        torch.cuda.synchronize()

    def kda_rows():
        # KDA decode, batch 64: the per-channel gate logits replace the per-head
        # ones (+ 32 x 128 x 2 bytes per token) and dt_bias is per channel
        kp = gdn.LayerParams(params.conv_w, params.A_log,
                             synth.normal((shape.hv, shape.dk), 0.5, g).to(dev))
        ksets = [perm[k * 64:(k + 1) * 64].to(dev) for k in range(8)]
        kin = [(synth.tokens(shape, g, (64,))[0].to(dev),
                synth.normal((64, shape.hv, shape.dk), 1.0, g, shape.act_dtype).to(dev),
                synth.tokens(shape, g, (64,))[2].to(dev)) for _ in range(8)]
        kout = torch.empty((64, shape.hv, shape.dv), dtype=torch.bfloat16, device=dev)

        def fk(i):
            q, ka, kb = kin[i % 8]
            gdn.kda_decode_step(dims, pool, kp, ksets[i % 8], q, ka, kb, kout)
        if want("kda_decode"):
            fk(0)
            kbytes = 64 * (DECODE_TOKEN_BYTES - 2 * 32 * 2 + 32 * 128 * 2 + 32 * 2) \
                + DECODE_STEP_PARAM_BYTES + 32 * 128 * 4
            rk = frac(kbytes, _events_time(fk, reps, stream))
            rk["tokens_per_s"] = 64 / (rk["ms"] * 1e-3)
            rows["kda_decode_b64"] = rk
        if want("kda_verify"):
            kda_verify_row(kp)
        if want("kda_prefill"):
            kda_prefill_row(kp)

    def kda_verify_row(kp):
        # KDA verify, batch 32, T = 8, snapshots into a separate spec pool
        Bk, Tk = 32, 8
        kspec = gdn.StatePool.empty(dims, 2 * Bk * Tk, dev)
        kss = [torch.arange(k * Bk * Tk, (k + 1) * Bk * Tk, dtype=torch.int32, device=dev).reshape(Bk, Tk)
               for k in range(2)]
        kws = [perm[k * Bk:(k + 1) * Bk].to(dev) for k in range(2)]
        kvin = [(synth.tokens(shape, g, (Bk, Tk))[0].to(dev),
                 synth.normal((Bk, Tk, shape.hv, shape.dk), 1.0, g, shape.act_dtype).to(dev),
                 synth.tokens(shape, g, (Bk, Tk))[2].to(dev)) for _ in range(2)]
        kvo = torch.empty((Bk, Tk, shape.hv, shape.dv), dtype=torch.bfloat16, device=dev)

        def fkv(i):
            q, ka, kb = kvin[i % 2]
            gdn.kda_spec_verify(dims, pool, kspec, kp, kws[i % 2], kss[i % 2], q, ka, kb, kvo)
        fkv(0)
        kvb = Bk * (slot_bytes + Tk * (16384 + 32 * 128 * 2 + 64) + Tk * slot_bytes + Tk * 8192)
        rkv = frac(kvb, _events_time(fkv, reps, stream))
        rkv["draft_tokens_per_s"] = Bk * Tk / (rkv["ms"] * 1e-3)
        rows["kda_verify_b32_t8"] = rkv
        del kspec

    def kda_prefill_row(kp):
        # KDA prefill (the 64-token chunk form on the tensor cores), 4 sequences x prefill_len tokens,
        # checkpoints every 256: per token qkv, the per-channel gate logits, beta and out
        nK, SK = 4, prefill_len
        kt = nK * SK
        kpq = synth.tokens(shape, g, (kt,))
        kpin = (kpq[0].to(dev), synth.normal((kt, shape.hv, shape.dk), 1.0, g, shape.act_dtype).to(dev),
                kpq[2].to(dev))
        del kpq
        kcu = torch.arange(0, kt + 1, SK, dtype=torch.int32, device=dev)
        ksp = torch.zeros(nK, dtype=torch.int64, device=dev)
        kck = gdn.StatePool.empty(dims, nK * (SK // 256), dev)
        kck_ids = torch.arange(nK * (SK // 256), dtype=torch.int32, device=dev).reshape(nK, SK // 256)
        kpo = torch.empty((kt, shape.hv, shape.dv), dtype=torch.bfloat16, device=dev)
        kpids = [perm[k * nK:(k + 1) * nK].to(dev) for k in range(4)]

        def fkp(i):
            gdn.kda_prefill(dims, pool, kck, kp, kpids[i % 4], kcu, ksp, kt, kck_ids, 256, *kpin, kpo)
        fkp(0)
        kpbytes = kt * (16384 + 32 * 128 * 2 + 64 + 8192) + (nK * (SK // 256) + 2 * nK) * slot_bytes
        rkp = frac(kpbytes, _events_time(fkp, 3, stream))
        rkp["tokens_per_s"] = kt / (rkp["ms"] * 1e-3)
        rows[f"kda_prefill_{nK}x{SK}"] = rkp
        del kpin, kck, kpo

    def epilogue_row():
        # readout epilogue over a 4 x 8192-token prefill output: o and z read,
        # y written in place (3 x 256 bytes per (token, V head) row)
        n_tok = 32768
        eo = synth.normal((n_tok, shape.hv, shape.dv), 0.7, g, shape.act_dtype).to(dev)
        ez = synth.normal((n_tok, shape.hv, shape.dv), 1.5, g, shape.act_dtype).to(dev)
        ew = torch.ones(shape.dv, dtype=torch.float32, device=dev)

        def fe(i):
            gdn.gated_rmsnorm(dims, eo, ez, ew, 1e-6)
        fe(0)
        rows["gated_rmsnorm_32768_tokens"] = frac(3 * n_tok * shape.hv * shape.dv * 2,
                                                  _events_time(fe, 20, stream))
        del eo, ez

    if want("slots"):
        slot_rows()
    if want("verify"):
        spec_rows()
    if want("prefill"):
        prefill_row()
    if want("kda_decode") or want("kda_verify") or want("kda_prefill"):
        kda_rows()
    if want("mixed"):
        rows["mixed_b64_plus_4x256"] = _mixed_row(gdn, synth, dims, pool, params, perm, g, dev, stream)
    if want("epilogue"):
        epilogue_row()
    return rows


def _mixed_row(gdn, synth, dims, pool, params, perm, g, dev, stream):
    """Decode-first mixed batch: 64 decode tokens plus 4 continuations of 256
    tokens from unaligned prefixes, through gdn_mixed_step; beside it the same
    batch sent whole through the chunked prefill (decode rows as 1-token
    sequences)."""
    import torch
    shape = synth.QWEN
    n_dec, L, starts = 64, 256, [1000, 3077, 517, 8191]
    lens = [1] * n_dec + [L] * 4
    n = len(lens)
    total = sum(lens)
    cu = torch.tensor([0] + list(torch.tensor(lens).cumsum(0).tolist()), dtype=torch.int32, device=dev)
    sp = torch.tensor([4096 + 7 * i for i in range(n_dec)] + starts, dtype=torch.int64, device=dev)
    sets = [perm[k * n:(k + 1) * n].to(dev) for k in range(2 if perm.numel() >= 2 * n else 1)]
    qkv, a, b = (t.to(dev) for t in synth.tokens(shape, g, (total,)))
    out = torch.empty((total, shape.hv, shape.dv), dtype=torch.bfloat16, device=dev)
    ck = gdn.StatePool.empty(dims, 2 * n, dev)
    ck_ids = torch.arange(2 * n, dtype=torch.int32, device=dev).reshape(n, 2)
    ws = torch.empty(gdn.chunk_prefill_workspace_size(dims, n, total), dtype=torch.uint8, device=dev)

    def fm(i):
        gdn.mixed_step(dims, pool, ck, params, sets[i % len(sets)], cu, sp, total, n_dec, ck_ids, 256, qkv, a, b,
                       out, ws)

    def fp(i):
        gdn.chunk_prefill(dims, pool, ck, params, sets[i % len(sets)], cu, sp, total, ck_ids, 256, qkv, a, b, out,
                          ws)
    fm(0)
    fp(0)
    ms_m = _events_time(fm, 20, stream)
    ms_p = _events_time(fp, 20, stream)
    # the same call as separate launches (decode kernel, chains, histories)
    import os
    os.environ["GDN_MIXED"] = "split"
    try:
        fm(0)
        ms_s = _events_time(fm, 20, stream)
    finally:
        del os.environ["GDN_MIXED"]
    return {"ms": ms_m, "tokens_per_s": total / (ms_m * 1e-3), "ms_split_launches": ms_s,
            "ms_all_through_prefill": ms_p, "batch": f"{n_dec} decode + 4 x {L} continuation tokens"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-rows", action="store_true", help="headline only")
    ap.add_argument("--rows", default="all", choices=list(ROW_GROUPS),
                    help="which secondary rows to time: all, or one group alone (for profiling)")
    ap.add_argument("--prefill-len", type=int, default=8192,
                    help="tokens per sequence of the 4-sequence GDN and KDA prefill rows (multiple of 256)")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--no-soak", action="store_true",
                    help="skip the untimed 1 s warm loop that gives the clock sampler a window")
    ap.add_argument("--pool", type=int, default=POOL,
                    help="slots in the pool (the headline uses 512; smaller for profiling)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
