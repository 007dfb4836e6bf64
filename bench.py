"""Benchmark: one relay decode-attention step (system attention + context
attention + relay fusion, one attention layer) on synthetic Llama-2-7B
shapes, through the C ABI of librelay.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl relay|reference]
                    [--workload llama2_7b] [--Ls L]

Prints ONE JSON line (rank 0).  `value` is tokens/s over the whole job (a
token = one query row of one request, all heads), measured with CUDA events
around each step's kernel on device-resident inputs, L2 flushed between
steps: a 256 MB buffer is written and then a second 256 MB buffer read, so
each step starts with L2 holding clean, unrelated lines (a write-only flush
would leave ~128 MB of dirty lines whose write-back the next step would pay).
The step itself is replayed from a CUDA graph.  `e2e` repeats the measurement through the public API with the
step's per-request inputs (q, block tables, lengths) copied from pinned host
memory and the output copied back inside the timed region; the KV caches are
persistent device state, as in a serving system.  `--impl reference` times
the fp64 CPU oracle on the host cores instead.

Under torchrun (N > 1) every rank runs an independent batch (weak scaling):
there is no exchange step in the path, so no collective touches the data.
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

import synth  # noqa: E402

METRIC = "relay decode-attention step µs, tokens/s & HBM GB/s (% of 8 TB/s), Llama2-7B"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}
KERNEL_SOURCES = ["shared_prompt_decode_gb300/csrc/relay.cu", "shared_prompt_decode_gb300/csrc/relay_kernels.cuh",
                  "shared_prompt_decode_gb300/csrc/sys_tc.cuh"]
# The library runs the system step on the tcgen05 kernel, a third launch per
# step, when D = 128, Ls > 0 and the batch holds more than this many virtual
# rows per KV head (query rows x query heads per KV head; the dispatch rule of
# relay.cu).
TC_MIN_ROWS = 256


def launches_per_step(case):
    rows = case.total_q() * (case.H // case.Hkv)
    return 3 if (case.D == 128 and case.Ls > 0 and rows > TC_MIN_ROWS) else 2


# ----------------------------------------------------------------------------- helpers
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world, backend):
    if world > 1 and not torch.distributed.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        torch.distributed.init_process_group(backend)


def max_over_ranks(x: float, world: int, device=None) -> float:
    if world <= 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]), "source": "measured"}
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS, source="fallback")


def kernel_hash():
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload):
    """DRAM bytes per launch of the relay kernel from a committed ncu summary,
    or None if the kernel changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", "relay_kernel_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    if rec.get("kernel_hash") != kernel_hash():
        return None
    entry = rec.get("workloads", {}).get(workload)
    return None if entry is None else entry.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks/throttle reasons sampled every 200 ms while running."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index=0):
        self.index = index
        self.proc = None
        self.lines = []
        self.thread = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        time.sleep(0.3)
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
            self.thread.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        loaded = [s for s in sm if s >= 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def build_case(args, rank):
    over = {}
    if args.Ls is not None:
        over["Ls"] = args.Ls
    wl = synth.workload(args.workload, **over)
    return synth.make_case(wl, seed=args.seed + rank)


def algorithmic_bytes(case):
    kv_tok = 2 * case.Hkv * case.D * 2          # K and V of one token, every KV head
    rows = case.total_q()
    return case.Ls * kv_tok + int(case.ctx_lens.sum()) * kv_tok + 2 * rows * case.H * case.D * 2


def workload_config(case, args):
    return {"workload": case.wl.name, "B": case.B, "H": case.H, "Hkv": case.Hkv, "D": case.D, "Ls": case.Ls,
            "Lq": case.Lq, "query_rows": case.total_q(), "ctx_tokens": int(case.ctx_lens.sum()),
            "block_size": 16, "seed": args.seed,
            "l2": "flushed between steps: 256 MB written, then another 256 MB read (L2 clean and cold)",
            "parallelism": f"replicas x{args.world} (independent batches)"}


# ----------------------------------------------------------------------------- oracle (CPU) timing
def time_oracle(case, frac_rows: float, min_seconds: float, max_reps: int):
    import oracle
    oracle.build()
    rows = oracle.all_rows(case)
    stride = max(1, int(round(1.0 / frac_rows)))
    sample = rows[::stride]
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle.attention_rows(case, sample)
        reps += 1
        el = time.perf_counter() - t0
        if el >= min_seconds or reps >= max_reps:
            break
    tokens = reps * len(sample) / case.H
    cores = oracle.max_threads()
    # one thread on a bounded sample (about 2 s), for the per-core rate
    one = sample[: max(1, len(sample) // 16)]
    n1, t1 = 0, time.perf_counter()
    while time.perf_counter() - t1 < 2.0:
        oracle.attention_rows(case, one, threads=1)
        n1 += 1
    e1 = time.perf_counter() - t1
    return {"value": tokens / el, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{len(sample)} of {len(rows)} (request, row, head) outputs per step, {reps} steps, "
                      f"{el:.1f} s wall; fp64 C with OpenMP",
            "single_thread": {"value": n1 * len(one) / case.H / e1, "unit": "tokens/s",
                              "sample": f"{len(one)} outputs x {n1} repetitions, {e1:.1f} s"}}


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    case = build_case(args, 0)
    import oracle
    oracle.build()
    rows = oracle.all_rows(case)
    stride = args.ref_stride
    sample = rows[::stride]
    for _ in range(args.warmup):
        oracle.attention_rows(case, sample[: max(1, len(sample) // 8)])
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.attention_rows(case, sample)
    el = time.perf_counter() - t0
    tokens = args.steps * len(sample) / case.H
    value = tokens / el
    cpu = {"value": value, "unit": "tokens/s", "cores": oracle.max_threads(), "kind": "oracle",
           "sample": f"{len(sample)} of {len(rows)} (request, row, head) outputs per step (every {stride}th), "
                     f"fp64 C with OpenMP"}
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": 0,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(case, args), "cpu_baseline": cpu,
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- the other workloads
def measure_workload(relay, case, dev, timed, as_graph, steps, warmup, baseline=True, sys_step=False):
    """Relay step (and optionally the non-relay baseline and the system step
    alone) of one workload, timed like the headline: graph replay, L2 flushed
    before every step, CUDA events on the launching stream."""
    g = {k: getattr(case, k).to(dev) for k in ("q", "sys_k", "sys_v", "k_cache", "v_cache", "block_tables",
                                              "ctx_lens")}
    ql = None if case.q_lens is None else case.q_lens.to(dev)
    mq = case.total_q() if ql is not None else 0
    dims = relay.make_dims(g["q"], case.Ls, case.num_blocks, case.max_blocks, Hkv=case.Hkv, max_q_total=mq)
    ws = relay.make_workspace(dims, dev)
    out = torch.empty_like(g["q"])

    def step():
        relay.relay_attention_decode(g["q"], g["sys_k"], g["sys_v"], g["k_cache"], g["v_cache"], g["block_tables"],
                                     g["ctx_lens"], ql, out=out, workspace=ws, dims=dims)
    ms, _ = timed(as_graph(step), steps, warmup)
    abytes = algorithmic_bytes(case)
    us = 1e3 * statistics.mean(ms)
    res = {"step_us": us, "algorithmic_bytes": abytes, "hbm_gbs": abytes / (us * 1e-6) / 1e9,
           "tokens_per_s": case.total_q() / (us * 1e-6), "requests_per_s": case.B / (us * 1e-6),
           "launches_per_step": launches_per_step(case)}
    if sys_step:
        # the system step alone (relay_sys_attn: the tensor-core kernel, then its partials fused into o_sys)
        o_s = torch.empty(*g["q"].shape, dtype=torch.float32, device=dev)
        l_s = torch.empty(*g["q"].shape[:3], dtype=torch.float32, device=dev)

        def sys_only():
            relay.relay_sys_attn(g["q"], g["sys_k"], g["sys_v"], ql, o_sys=o_s, lse_sys=l_s, workspace=ws,
                                 max_q_total=mq)
        ms_s, _ = timed(as_graph(sys_only), steps, warmup)
        sus = 1e3 * statistics.mean(ms_s)
        flops = 4 * case.total_q() * case.Ls * case.D * case.H
        res["system_step"] = {"us": sus, "flops": flops, "tflops": flops / (sus * 1e-6) / 1e12,
                              "what": "relay_sys_attn: sys_tc_kernel (tcgen05) + fusion of its partials into o_sys"}
        del o_s, l_s
    if baseline:
        kp, vp, ids = synth.with_system_in_pool(case)
        kp, vp, ids = kp.to(dev), vp.to(dev), ids.to(dev)
        dims_b = relay.make_dims(g["q"], case.Ls, kp.shape[0], case.max_blocks, max_q_total=mq, Hkv=case.Hkv)
        ws_b = relay.make_workspace(dims_b, dev)
        out_b = torch.empty_like(out)

        def base_step():
            relay.relay_baseline_decode(g["q"], kp, vp, ids, case.Ls, g["block_tables"], g["ctx_lens"], ql,
                                        out=out_b, workspace=ws_b, dims=dims_b)
        ms_b, _ = timed(as_graph(base_step), steps, warmup)
        bus = 1e3 * statistics.mean(ms_b)
        res["nonrelay_us"] = bus
        res["relay_speedup"] = bus / us
        del kp, vp, ids, ws_b, out_b
    del g, ws, out
    return res


def run_configs(args, relay, dev, timed, as_graph, peaks):
    """The other workloads of the study at their full sizes (one line each in
    `configs`): the Llama-30B system-prompt-length sweep with the non-relay
    baseline ("flat in Ls"), the batch-256 Llama-2-7B step, and the Llama-2-13B
    mixed step whose system step runs on the tensor cores."""
    steps = max(3, args.steps // 4)
    hbm = peaks["hbm_gbs"]
    out = {"timing": f"{steps} timed steps per point after {args.warmup} warm-up steps, graph replay, "
                     "L2 flushed before every step, CUDA events"}
    pts = []
    for Ls in synth.SWEEP_LS:
        case = synth.make_case(synth.workload("llama30b_sweep", Ls=Ls), seed=args.seed)
        r = measure_workload(relay, case, dev, timed, as_graph, steps, args.warmup)
        pts.append({"Ls": Ls, "relay_us": r["step_us"], "nonrelay_us": r["nonrelay_us"],
                    "relay_speedup": r["relay_speedup"], "algorithmic_bytes": r["algorithmic_bytes"],
                    "hbm_gbs": r["hbm_gbs"], "frac": r["hbm_gbs"] / hbm})
        del case
    out["llama30b_sweep"] = {
        "shape": "H=52, D=128, B=32, 1 query row each, ctx U[128,512], Ls swept", "points": pts,
        "relay_growth_16384_over_512": pts[-1]["relay_us"] / pts[0]["relay_us"],
        "nonrelay_growth_16384_over_512": pts[-1]["nonrelay_us"] / pts[0]["nonrelay_us"],
        "algorithmic_bytes_growth_16384_over_512": pts[-1]["algorithmic_bytes"] / pts[0]["algorithmic_bytes"]}
    case = synth.make_case("llama2_7b_b256", seed=args.seed)
    r = measure_workload(relay, case, dev, timed, as_graph, steps, args.warmup)
    r["frac"] = r["hbm_gbs"] / hbm
    out["llama2_7b_b256"] = dict(r, shape="H=32, D=128, B=256, Ls=4096, ctx lognormal(256, 1) in [1, 2048]")
    del case
    case = synth.make_case("llama2_13b_mixed", seed=args.seed)
    r = measure_workload(relay, case, dev, timed, as_graph, steps, args.warmup, sys_step=True)
    tf = peaks["bf16_tflops"]
    flops = r["system_step"]["flops"]
    hbm_floor = r["algorithmic_bytes"] / (hbm * 1e9) * 1e6
    tensor_floor = flops / (tf * 1e12) * 1e6
    r["roofline"] = {"hbm_floor_us": hbm_floor, "tensor_floor_us": tensor_floor,
                     "frac_of_max_floor": max(hbm_floor, tensor_floor) / r["step_us"],
                     "system_step_tensor_frac": r["system_step"]["tflops"] / tf,
                     "peaks": f"{peaks['source']} copy bandwidth {hbm:.0f} GB/s, dense bf16 {tf:.0f} TFLOP/s "
                              "(fp16 has the same nominal tensor rate)"}
    out["llama2_13b_mixed"] = dict(r, shape="H=40, D=128, B=64 (56 x 1 row, 8 x 128-row chunks), Ls=32768, "
                                            "ctx U[1,4096]")
    del case
    return out


# ----------------------------------------------------------------------------- GPU timing
def run_relay(args):
    world, rank, local = dist_env()
    if not torch.cuda.is_available():
        print(json.dumps({"metric": METRIC, "error": "no CUDA device"}))
        return 1
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    init_dist(world, "nccl")
    args.world = world

    from shared_prompt_decode_gb300 import build as relay_build
    if rank == 0 or world == 1:
        relay_build.build()
    barrier(world)
    import shared_prompt_decode_gb300 as relay

    case = build_case(args, rank)
    g = {k: getattr(case, k).to(dev) for k in ("q", "sys_k", "sys_v", "k_cache", "v_cache", "block_tables",
                                              "ctx_lens")}
    g["q_lens"] = None if case.q_lens is None else case.q_lens.to(dev)
    mq = case.total_q() if case.q_lens is not None else 0
    rows = case.total_q()
    dims = relay.make_dims(g["q"], case.Ls, case.num_blocks, case.max_blocks, Hkv=case.Hkv, ctx_split=args.ctx_split,
                           sys_range=args.sys_range, max_q_total=mq)
    ws = relay.make_workspace(dims, dev)
    out = torch.empty_like(g["q"])
    flush_w = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    flush_r = torch.ones(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def flush():
        flush_w.zero_()
        flush_r.sum()

    def as_graph(fn):
        """Capture one call of fn (after two eager calls) and return a replay function."""
        side = torch.cuda.Stream(dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):
            fn()
            fn()
        torch.cuda.current_stream(dev).wait_stream(side)
        torch.cuda.synchronize(dev)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            fn()
        return graph.replay

    def step():
        relay.relay_attention_decode(g["q"], g["sys_k"], g["sys_v"], g["k_cache"], g["v_cache"],
                                     g["block_tables"], g["ctx_lens"], g["q_lens"], out=out, workspace=ws,
                                     dims=dims)

    def timed(fn, steps, warmup, cold=True):
        for _ in range(warmup):
            if cold:
                flush()
            fn()
        torch.cuda.synchronize(dev)
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        barrier(world)
        torch.cuda.synchronize(dev)
        w0 = time.perf_counter()
        for i in range(steps):
            if cold:
                flush()
            starts[i].record(stream)
            fn()
            ends[i].record(stream)
        torch.cuda.synchronize(dev)
        barrier(world)
        wall = time.perf_counter() - w0
        ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
        return ms, wall

    step_graph = as_graph(step)
    with ClockSampler(local) as clk:
        ms, wall = timed(step_graph, args.steps, args.warmup)
    ms_hot, _ = timed(step_graph, max(10, args.steps // 4), args.warmup, cold=False)    # L2 left warm
    clocks = clk.summary()
    mean_ms = max_over_ranks(sum(ms) / len(ms), world, dev)
    value = world * rows / (mean_ms * 1e-3)
    abytes = algorithmic_bytes(case)
    peaks = load_peaks()
    achieved = abytes / (statistics.mean(ms) * 1e-3) / 1e9
    traffic = recorded_traffic(case.wl.name if args.Ls is None else f"{case.wl.name}_Ls{args.Ls}")
    if args.quick:
        if rank == 0:
            print(json.dumps({"metric": METRIC, "value": value, "unit": "tokens/s", "step_us": 1e3 * mean_ms,
                              "hbm_gbs": achieved, "frac": achieved / peaks["hbm_gbs"], "ctx_split": args.ctx_split,
                              "sys_range": args.sys_range, "config": workload_config(case, args)}), flush=True)
        return 0

    # non-relay baseline: same requests, system KV re-read per request from the paged pool
    kp, vp, ids = synth.with_system_in_pool(case)
    kp, vp, ids = kp.to(dev), vp.to(dev), ids.to(dev)
    dims_b = relay.make_dims(g["q"], case.Ls, kp.shape[0], case.max_blocks, max_q_total=mq, Hkv=case.Hkv)
    ws_b = relay.make_workspace(dims_b, dev)
    out_b = torch.empty_like(out)

    def base_step():
        relay.relay_baseline_decode(g["q"], kp, vp, ids, case.Ls, g["block_tables"], g["ctx_lens"], g["q_lens"],
                                    out=out_b, workspace=ws_b, dims=dims_b)
    ms_b, _ = timed(as_graph(base_step), max(5, args.steps // 2), args.warmup)
    del kp, vp

    # end to end through the public API, host buffers, copies inside the timed region: the step's inputs
    # (q, block tables, context lengths, query lengths) staged in one pinned buffer and copied in one
    # transfer, as a serving loop would, into one device buffer that the call reads through typed views
    parts = [case.q, case.block_tables, case.ctx_lens] + ([] if case.q_lens is None else [case.q_lens])
    offs, nbytes = [], 0
    for t in parts:
        offs.append(nbytes)
        nbytes += (t.numel() * t.element_size() + 255) // 256 * 256
    hin = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    din = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    views_h, views_d = [], []
    for t, o in zip(parts, offs):
        n = t.numel() * t.element_size()
        views_h.append(hin[o:o + n].view(t.dtype).view(t.shape))
        views_d.append(din[o:o + n].view(t.dtype).view(t.shape))
    for t, v in zip(parts, views_h):
        v.copy_(t)
    dq, dbt, dcl = views_d[0], views_d[1], views_d[2]
    dql = views_d[3] if case.q_lens is not None else None
    hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()

    def e2e_step():
        din.copy_(hin, non_blocking=True)
        relay.relay_attention_decode(dq, g["sys_k"], g["sys_v"], g["k_cache"], g["v_cache"], dbt, dcl, dql, out=out,
                                     workspace=ws, dims=dims, stream=stream)
        hout.copy_(out, non_blocking=True)
    ms_e, _ = timed(e2e_step, args.steps, args.warmup)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(sum(ms_e) / len(ms_e), world, dev)
    h2d = nbytes
    d2h = hout.numel() * hout.element_size()

    # the cache write that precedes the step: this step's new K/V rows into the pool (timed like the step)
    gk = torch.Generator().manual_seed(args.seed + 7)
    kv_shape = (case.B, case.Lq, case.Hkv, case.D)
    k_new = torch.randn(*kv_shape, generator=gk).half().to(dev)
    v_new = torch.randn(*kv_shape, generator=gk).half().to(dev)
    kc_scratch, vc_scratch = g["k_cache"].clone(), g["v_cache"].clone()
    ws_a = torch.zeros(256, dtype=torch.uint8, device=dev)

    def append_step():
        relay.relay_kv_append(k_new, v_new, g["block_tables"], g["ctx_lens"], kc_scratch, vc_scratch,
                              q_lens=g["q_lens"], workspace=ws_a)
    ms_a, _ = timed(as_graph(append_step), max(5, args.steps // 4), args.warmup)
    # rotary positions of the step's q and new k, offset by the system prompt (in place on scratch copies)
    q_rot, k_rot = g["q"].clone(), k_new.clone()

    def rope_step():
        relay.relay_rope(q_rot, g["ctx_lens"], case.Ls, k_new=k_rot, q_lens=g["q_lens"], workspace=ws_a)
    ms_r, _ = timed(as_graph(rope_step), max(5, args.steps // 4), args.warmup)
    rope_bytes = 2 * rows * (case.H + case.Hkv) * case.D * 2    # q and k rows, read and written
    del q_rot, k_rot
    append_bytes = 2 * 2 * rows * case.Hkv * case.D * 2          # K and V rows, read once and written once
    del kc_scratch, vc_scratch

    # the system prompt's own prefill attention (causal, compute-bound: tcgen05), timed like the step
    prefill = None
    if case.D == 128 and case.Ls > 0:
        gp = torch.Generator().manual_seed(args.seed + 9)
        q_sys = (torch.randn(case.Ls, case.H, case.D, generator=gp) * 0.5).half().to(dev)
        out_p = torch.empty_like(q_sys)
        ws_p = torch.zeros(256, dtype=torch.uint8, device=dev)

        def prefill_step():
            relay.relay_sys_prefill(q_sys, g["sys_k"], g["sys_v"], out=out_p, workspace=ws_p)
        ms_p, _ = timed(as_graph(prefill_step), max(5, args.steps // 40), args.warmup)
        flops = 2 * case.D * case.H * case.Ls * (case.Ls + 1)    # QK^T and PV over the t+1 visible keys of row t
        tflops = flops / (statistics.mean(ms_p) * 1e-3) / 1e12
        peaks_p = load_peaks()
        prefill = {"kernel": "sys_tc_kernel<prefill> (relay_sys_prefill: causal self-attention of the system prompt)",
                   "us": 1e3 * statistics.mean(ms_p), "flops": flops, "tflops": tflops,
                   "peak_tflops": peaks_p["bf16_tflops"], "frac": tflops / peaks_p["bf16_tflops"],
                   "peak_source": f"{peaks_p['source']} dense bf16 (fp16 has the same nominal tensor rate)"}
        del q_sys, out_p

    # a two-level prefix tree on this batch: the workload's system prompt shared by every request plus one
    # 512-token prompt per group of requests (4 groups), served as a tree (global and group prompts each read
    # once, K = 6 parts merged by relay_fuse_n) and flattened (one relay call per group with its prompts
    # concatenated, the global prompt re-read per group)
    tree = None
    if case.q_lens is None and case.Ls > 0 and case.B % 4 == 0:
        groups, Lp = 4, 512
        gt = torch.Generator().manual_seed(args.seed + 11)
        grp = [((torch.randn(Lp, case.Hkv, case.D, generator=gt) * 0.5).half().to(dev),
                (torch.randn(Lp, case.Hkv, case.D, generator=gt) * 0.5).half().to(dev)) for _ in range(groups)]
        masks = [torch.tensor([1 if b % groups == p else 0 for b in range(case.B)], dtype=torch.int32, device=dev)
                 for p in range(groups)]
        shp = (case.B, case.Lq, case.H)
        o_parts = [torch.zeros(*shp, case.D, dtype=torch.float32, device=dev) for _ in range(groups + 2)]
        l_parts = [torch.full(shp, float("-inf"), dtype=torch.float32, device=dev) for _ in range(groups + 2)]
        ws_t = [relay.make_workspace(relay.make_dims(g["q"], Ls_, case.num_blocks, case.max_blocks, Hkv=case.Hkv), dev)
                for Ls_ in [case.Ls] + [Lp] * groups + [0]]
        out_t = torch.empty_like(out)

        def tree_step():
            relay.relay_sys_attn(g["q"], g["sys_k"], g["sys_v"], o_sys=o_parts[0], lse_sys=l_parts[0], workspace=ws_t[0])
            for p, (k, v) in enumerate(grp):
                relay.relay_sys_attn(g["q"], k, v, q_lens=masks[p], o_sys=o_parts[1 + p], lse_sys=l_parts[1 + p],
                                     workspace=ws_t[1 + p])
            relay.relay_ctx_attn(g["q"], g["k_cache"], g["v_cache"], g["block_tables"], g["ctx_lens"],
                                 o_ctx=o_parts[-1], lse_ctx=l_parts[-1], workspace=ws_t[-1])
            relay.relay_fuse_n(o_parts, l_parts, out=out_t)
        ms_t, _ = timed(as_graph(tree_step), max(5, args.steps // 8), args.warmup)
        # flattened: each group alone, its system prompt = [global; group prompt]
        flat = []
        for p, (k, v) in enumerate(grp):
            idx = torch.tensor([b for b in range(case.B) if b % groups == p], device=dev)
            fk, fv = torch.cat([g["sys_k"], k]), torch.cat([g["sys_v"], v])
            qg = g["q"][idx].contiguous()
            fd = relay.make_dims(qg, fk.shape[0], case.num_blocks, case.max_blocks, Hkv=case.Hkv)
            flat.append((qg, fk, fv, g["block_tables"][idx].contiguous(), g["ctx_lens"][idx].contiguous(),
                         torch.empty_like(qg), relay.make_workspace(fd, dev), fd))

        def flat_step():
            for qg, fk, fv, btg, clg, og, wsg, fd in flat:
                relay.relay_attention_decode(qg, fk, fv, g["k_cache"], g["v_cache"], btg, clg, out=og, workspace=wsg,
                                             dims=fd)
        ms_f, _ = timed(as_graph(flat_step), max(5, args.steps // 8), args.warmup)
        # the same tree in one unit: five shared segments, request b sees the global prompt and its group's
        segs_k = [g["sys_k"]] + [k for k, _ in grp]
        segs_v = [g["sys_v"]] + [v for _, v in grp]
        seg_mask = torch.tensor([1 | (2 << (b % groups)) for b in range(case.B)], dtype=torch.int32, device=dev)
        dims_f = relay.make_dims(g["q"], 0, case.num_blocks, case.max_blocks, Hkv=case.Hkv)
        ws_f = torch.zeros(relay.prefixes_workspace_size(dims_f, [case.Ls] + [Lp] * groups), dtype=torch.uint8,
                           device=dev)
        out_fu = torch.empty_like(out)

        def fused_step():
            relay.relay_attention_decode_prefixes(g["q"], segs_k, segs_v, seg_mask, g["k_cache"], g["v_cache"],
                                                  g["block_tables"], g["ctx_lens"], out=out_fu, workspace=ws_f,
                                                  dims=dims_f)
        ms_fu, _ = timed(as_graph(fused_step), max(5, args.steps // 8), args.warmup)
        kv_tok = 2 * case.Hkv * case.D * 2
        tree = {"groups": groups, "group_prompt_tokens": Lp,
                "fused_us": 1e3 * statistics.mean(ms_fu),
                "tree_us": 1e3 * statistics.mean(ms_t), "flattened_us": 1e3 * statistics.mean(ms_f),
                "tree_kv_bytes": (case.Ls + groups * Lp + int(case.ctx_lens.sum())) * kv_tok,
                "flattened_kv_bytes": (groups * (case.Ls + Lp) + int(case.ctx_lens.sum())) * kv_tok,
                "launches": {"fused": "relay_attention_decode_prefixes (two kernels)",
                             "tree": "5 x relay_sys_attn + relay_ctx_attn (two kernels each) + fuse_n_kernel",
                             "flattened": "4 x relay_attention_decode (two kernels each)"}}
        del o_parts, l_parts, ws_t, flat, ws_f, out_fu

    configs = None
    if not args.no_configs:
        configs = run_configs(args, relay, dev, timed, as_graph, load_peaks())

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        cpu = time_oracle(case, frac_rows=1.0, min_seconds=10.0, max_reps=200)

    if rank != 0:
        return 0
    base_mean = statistics.mean(ms_b)
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": mean_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16 in, f32 accumulate", "data": "synthetic",
        "config": workload_config(case, args),
        "step_us": 1e3 * mean_ms,
        "step_us_hot_l2": 1e3 * statistics.mean(ms_hot),
        "requests_per_s": world * case.B / (mean_ms * 1e-3),
        "step_us_p10_p50_p90": [1e3 * x for x in statistics.quantiles(ms, n=10)[::4]] if len(ms) >= 10 else None,
        "hbm_gbs": achieved, "pct_of_8tbs": 100.0 * achieved / NOMINAL_HBM_GBS,
        "algorithmic_bytes_per_step": abytes,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm_gbs"], "traffic": traffic,
                     "kernel": ("relay_kernel<128> + merge_kernel<128> (two launches per step, one graph)"
                                if launches_per_step(case) == 2 else
                                "sys_tc_kernel + relay_kernel<128> + merge_kernel<128> (three launches per step, one graph)"),
                     "peak_source": f"{peaks['source']} copy bandwidth (burst)"},
        "nonrelay_baseline": {"kernel": "relay_baseline_decode (system KV re-read per request)",
                              "step_us": 1e3 * base_mean, "tokens_per_s": rows / (base_mean * 1e-3),
                              "relay_speedup": base_mean / statistics.mean(ms)},
        "e2e": {"value": world * rows / (e2e_ms * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
        "gpu_launches": launches_per_step(case) * args.steps,
        "sys_prefill": prefill,
        "tree_prefixes": tree,
        "rope": {"kernel": "rope_kernel (relay_rope: rotary positions offset by the system prompt)",
                 "us": 1e3 * statistics.mean(ms_r), "bytes": rope_bytes,
                 "gbs": rope_bytes / (statistics.mean(ms_r) * 1e-3) / 1e9},
        "kv_append": {"kernel": "kv_append_kernel (relay_kv_append: the step's new K/V rows into the pool)",
                      "us": 1e3 * statistics.mean(ms_a), "bytes": append_bytes,
                      "gbs": append_bytes / (statistics.mean(ms_a) * 1e-3) / 1e9},
        "clocks": clocks,
        "wall_s_timed_region": wall,
    }
    if cpu is not None:
        line["cpu_baseline"] = cpu
    if configs is not None:
        line["configs"] = configs
    print(json.dumps(line), flush=True)
    return 0


def run_profile(args):
    """A short, fixed sequence of relay launches for an external profiler."""
    dev = torch.device("cuda", 0)
    from shared_prompt_decode_gb300 import build as relay_build
    relay_build.build()
    import shared_prompt_decode_gb300 as relay
    case = build_case(args, 0)
    g = {k: getattr(case, k).to(dev) for k in ("q", "sys_k", "sys_v", "k_cache", "v_cache", "block_tables",
                                              "ctx_lens")}
    ql = None if case.q_lens is None else case.q_lens.to(dev)
    dims = relay.make_dims(g["q"], case.Ls, case.num_blocks, case.max_blocks, Hkv=case.Hkv, ctx_split=args.ctx_split,
                           sys_range=args.sys_range, max_q_total=case.total_q() if ql is not None else 0)
    ws = relay.make_workspace(dims, dev)
    out = torch.empty_like(g["q"])
    flush_w = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    flush_r = torch.ones(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    for _ in range(args.profile):
        flush_w.zero_()
        flush_r.sum()
        relay.relay_attention_decode(g["q"], g["sys_k"], g["sys_v"], g["k_cache"], g["v_cache"],
                                     g["block_tables"], g["ctx_lens"], ql, out=out, workspace=ws, dims=dims)
    torch.cuda.synchronize(dev)
    print(json.dumps({"profile_launches": args.profile, "workload": case.wl.name,
                      "algorithmic_bytes_per_launch": algorithmic_bytes(case)}))
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["relay", "reference"], default="relay")
    ap.add_argument("--workload", default="llama2_7b", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--Ls", type=int, default=None, help="override the system-prompt length")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--quick", action="store_true", help="relay timing only: no baseline, e2e or CPU legs")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the other workloads (Llama-30B sweep, batch 256, 13B mixed)")
    ap.add_argument("--ctx-split", type=int, default=0, help="context keys per decode work item (0: automatic)")
    ap.add_argument("--sys-range", type=int, default=0, help="system keys per work item (0: automatic)")
    ap.add_argument("--ref-stride", type=int, default=8, help="reference arm: time every n-th output row")
    ap.add_argument("--profile", type=int, default=0, metavar="N",
                    help="profiling driver: run N relay launches (L2 flushed between) and exit, no timing")
    args = ap.parse_args(argv)
    args.warmup = max(args.warmup, 3)
    args.world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.impl == "reference":
        return run_reference(args)
    if args.profile:
        return run_profile(args)
    return run_relay(args)


if __name__ == "__main__":
    sys.exit(main())
