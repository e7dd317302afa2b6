"""KDA prefill / decode benchmark on GB300.

One step = one kda_chunk_fwd over the packed varlen prefill workload (64
sequences of U[512, 32768] tokens, seeded; H = 32, dk = dv = 128, chunk 64,
initial states given; final states and every chunk-boundary snapshot written;
inputs far larger than L2), the largest single-GPU configuration.  The same
run reports, as their own objects, the B=4 H=16 T=8192 prefill, the
1,048,576-token prefill, the decode step (512 x 32 resident states, 1000
chained steps) and the latency of the tiny B=1 H=2 T=256 dk=dv=64 prefill.
Prints ONE JSON line on rank 0.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the fp64 CPU oracle (the reference arm of this
build) on the host cores, on a bounded sample of the same workload.
Under torchrun each rank runs its own replica (weak scaling, no collective
on the data path); timing is the maximum over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "KDA prefill tokens/s and decode steps/s on 1 GB300; % of TC / HBM roofline"
UNIT = "tokens/s"
WORKLOAD = "varlen"

# Algorithmic traffic and work per token-head at chunk 64 (bf16 in/out, fp32 states):
#   q, k, z (dk each), v, o (dv each) in bf16 plus beta: 2 (3 dk + 2 dv) + 2 bytes;
#   chunk-boundary snapshots: 4 dk dv / 64 bytes;
#   flops: 6 dk dv + 64 (3 dk + 2 dv) + 64^2 / 3 (causal halves once, masked tiles not counted).


def prefill_bytes(token_heads, seq_heads, dk, dv, snapshots=True, s0=False, s_final=True,
                  full_chunk_heads=None):
    """Bytes the prefill must move: inputs, outputs, snapshots, S0 / S_final.
    Snapshots follow every full chunk (token_heads / 64 of them for lengths
    that are multiples of 64; pass full_chunk_heads otherwise)."""
    b = token_heads * (2 * (3 * dk + 2 * dv) + 2)
    if snapshots:
        if full_chunk_heads is None:
            b += token_heads * 4 * dk * dv // 64
        else:
            b += full_chunk_heads * 4 * dk * dv
    b += seq_heads * 4 * dk * dv * (int(s0) + int(s_final))
    return b


REC_BYTES = 74240  # bytes of one (chunk, head) record the two passes exchange


def prep_bytes(token_heads, dk, dv):
    """Chunk preparation, algorithmic: it reads q, k, z, v and beta.  (It also
    writes one record per (chunk, head): traffic the two-pass design adds,
    reported apart as traffic_overhead.)"""
    return token_heads * (2 * (3 * dk + dv) + 2)


def state_bytes(token_heads, full_chunk_heads, seq_heads, dk, dv, s0=False):
    """State pass, algorithmic: it writes o, the snapshots and the final states
    (and reads S0 when given).  (It also reads the records.)"""
    return (token_heads * 2 * dv + full_chunk_heads * 4 * dk * dv +
            seq_heads * 4 * dk * dv * (1 + int(s0)))


# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one launch from
# the ncu captures summarised under profiles/, per (chunk, head) task of the
# captured launch, scaled here by the tasks of the timed launch.  They are
# reported only while the kernel's sources hash to the sha256 prefix recorded
# with the capture (else the kernel has changed since: null).  A change to the
# sources' comments alone updates the recorded prefix without a new capture.
_CSRC = os.path.join(ROOT, "linear_attention_serving_chunk_gb300", "csrc")
_TC_FILES = ("kda_tc_common.cuh", "kda_sm100.cuh", "kda_split.cuh", "kda_common.cuh", "kda_pdl.cuh")
PROFILED_TRAFFIC = {
    # the full varlen prefill step (64 sequences, 1,012,452 tokens, H = 32): 507,168 tasks
    "chunk_prep_kernel": (33.747327744e9 + 37.643570432e9, 507168, "6cbc58f518fa86b4",
                          ("kda_chunk_prep.cu",) + _TC_FILES),
    "state_pass_kernel": (37.787850240e9 + 41.482227200e9, 507168, "2282604758755b95",
                          ("kda_state_pass.cu",) + _TC_FILES),
    # decode, 512 sequences x H = 32: 16,384 (sequence, head) states
    "kda_decode_step": (1.090611e9 + 1.017599e9, 16384, "850844e37b9a8a6f",
                        ("kda_decode.cu", "kda_common.cuh", "kda_tc_common.cuh", "kda_sm100.cuh")),
    # verify: 4 tokens on each of 512 x H = 32 states (commit = 0)
    "decode_tokens_kernel": (1.141108e9 + 1.8478080e7, 16384, "850844e37b9a8a6f",
                             ("kda_decode.cu", "kda_common.cuh", "kda_tc_common.cuh",
                              "kda_sm100.cuh")),
    # restore, 512 x H = 32 states
    "snapshot_restore_kernel": (1.073760e9 + 1.025011e9, 16384, "7acfbeb05332783a",
                                ("kda_snapshot.cu", "kda_common.cuh")),
}


def profiled_traffic(kernel, tasks):
    import hashlib
    if kernel not in PROFILED_TRAFFIC:
        return None
    traffic, ptasks, digest, files = PROFILED_TRAFFIC[kernel]
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(_CSRC, f), "rb") as fh:
            h.update(fh.read())
    return traffic * tasks / ptasks if h.hexdigest()[:16] == digest else None


def prefill_flops(token_heads, dk, dv):
    return token_heads * (6 * dk * dv + 64 * (3 * dk + 2 * dv) + 64 * 64 / 3)


def decode_bytes(n_states, dk, dv):
    # state read + write, q, k, z, v, o in bf16, beta
    return n_states * (8 * dk * dv + 2 * (3 * dk + 2 * dv) + 2)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p.get(
            "bf16_tflops_sustained", p["bf16_tflops"])), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, 1900.0, 1700.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 20 ms.

    Entering starts nvidia-smi and waits (up to 5 s) for its first sample, so
    that sampling is running before the timed region starts; ``window(t0, t1)``
    then keeps the samples taken between those host times (time.monotonic())
    plus one interval, i.e. during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    INTERVAL_MS = 20

    def __init__(self, gpu_id):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []
        self.thread = None
        self.t0 = self.t1 = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_id), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", str(self.INTERVAL_MS)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            deadline = time.monotonic() + 5.0
            while not self.lines and time.monotonic() < deadline and self.proc.poll() is None:
                time.sleep(0.005)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.monotonic(), line.strip()))

    def window(self, t0, t1):
        self.t0, self.t1 = t0, t1

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(2 * self.INTERVAL_MS / 1e3)  # the sample that closes the window
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            if self.thread is not None:
                self.thread.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        lines = self.lines
        if self.t0 is not None:
            slack = self.INTERVAL_MS / 1e3
            lines = [(t, l) for t, l in lines if self.t0 <= t <= self.t1 + slack]
        for _, line in lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[3:7]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup(n_gpus):
    """Rank info; under torchrun each rank gets its own GPU (no data collective)."""
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world != n_gpus and world > 1:
        raise SystemExit(f"--gpus {n_gpus} but WORLD_SIZE={world}")
    return rank, world, local


def reduce_max(value, world):
    """Maximum of a float over ranks (identity for one rank)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def init_pg(world):
    if world > 1:
        import torch.distributed as dist
        if not dist.is_initialized():
            dist.init_process_group("gloo")


# --- workloads ---------------------------------------------------------------------------------

_OVERRIDE = {}  # --seq-len / --n-seq of the headline workload (profiling runs)


def workload_params(name):
    import kda_inputs
    w = dict(kda_inputs.WORKLOADS[name])
    if name == WORKLOAD:
        if _OVERRIDE.get("seq_len") and w["kind"] == "prefill":
            w["T"] = _OVERRIDE["seq_len"]
        if _OVERRIDE.get("n_seq"):
            w["n_seq" if w["kind"] == "varlen" else "B"] = _OVERRIDE["n_seq"]
    return w


def workload_lengths(name):
    import kda_inputs
    w = workload_params(name)
    if w["kind"] == "varlen":
        return kda_inputs.varlen_lengths(w["n_seq"], w["len_lo"], w["len_hi"], w["seed"])
    return [w["T"]] * w["B"]


def make_workload(name, device):
    import kda_inputs
    w = workload_params(name)
    return kda_inputs.make_prefill(w["H"], w["dk"], w["dv"], workload_lengths(name), w["seed"],
                                   device, S0_std=w.get("S0_std"))


def workload_config(name):
    w = workload_params(name)
    L = workload_lengths(name)
    total = sum(L)
    if w["kind"] == "varlen":
        desc = (f"kda varlen prefill: {w['n_seq']} packed sequences, lengths "
                f"U[{w['len_lo']}, {w['len_hi']}] (seed {w['seed']}, {total} tokens), "
                f"H={w['H']} dk={w['dk']} dv={w['dv']} chunk={w['chunk']}, cu_seqlens, "
                f"S0 ~ N(0, {w['S0_std']}^2), final states + chunk snapshots")
    else:
        desc = (f"kda prefill B={w['B']} H={w['H']} T={w['T']} dk={w['dk']} dv={w['dv']} "
                f"chunk={w['chunk']}, final state + chunk snapshots")
    return {"workload": desc, "global_batch": len(L), "seq_len": max(L), "tokens": total,
            "heads": w["H"], "l2": "inputs larger than L2 (129 MB) by far, no flush"}


# --- reference arm: the fp64 oracle on the host cores --------------------------------------

def oracle_sample(x, n_tokens):
    """Host fp64 copies of the first n_tokens of every sequence, all heads."""
    import numpy as np
    import kda_inputs
    cu = x["cu_seqlens"].cpu().numpy()
    parts = {n: [] for n in ("q", "k", "v", "z", "beta")}
    lens = []
    for s in range(len(cu) - 1):
        a, L = int(cu[s]), min(n_tokens, int(cu[s + 1] - cu[s]))
        lens.append(L)
        for n in parts:
            parts[n].append(kda_inputs.to_f64(x[n][a:a + L]))
    cat = {n: np.concatenate(parts[n]) for n in parts}
    cat["A"] = kda_inputs.to_f64(x["A"])
    cat["S0"] = None if x.get("S0") is None else kda_inputs.to_f64(x["S0"])
    cat["cu"] = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    return cat, int(sum(lens))


def time_oracle(cat, steps):
    import oracle
    dts = []
    for _ in range(steps):
        t = time.perf_counter()
        oracle.prefill(cat["q"], cat["k"], cat["v"], cat["z"], cat["beta"], cat["A"],
                       cu_seqlens=cat["cu"], S0=cat["S0"], snapshots=True)
        dts.append(time.perf_counter() - t)
    return dts


def sample_desc(name, n_tok_seq, n_tok):
    w = workload_params(name)
    n_seq = len(workload_lengths(name))
    return (f"first {n_tok_seq} tokens of each of the {n_seq} sequences, all {w['H']} heads "
            f"({n_tok * w['H']} token-heads per step), S0 and snapshots as the workload")


def run_reference(args, rank, world):
    """The oracle on the host cores: each step runs it over the first
    --ref-tokens tokens of every sequence of the workload (all heads), drawn
    with the workload's recipe and seed; only that sample is generated, the
    whole workload would not fit the host's time budget."""
    import kda_inputs
    import oracle
    if rank != 0:
        return
    w = workload_params(WORKLOAD)
    lens = [min(args.ref_tokens, L) for L in workload_lengths(WORKLOAD)]
    x = kda_inputs.make_prefill(w["H"], w["dk"], w["dv"], lens, w["seed"], "cpu",
                                S0_std=w.get("S0_std"))
    cat, n_tok = oracle_sample(x, args.ref_tokens)
    time_oracle(cat, args.warmup)
    dts = time_oracle(cat, args.steps)
    total = sum(dts)
    value = n_tok * args.steps / total  # tokens (all H heads) per second
    cores = oracle.num_threads()
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(WORKLOAD),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": sample_desc(WORKLOAD, args.ref_tokens, n_tok)},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# --- our arm ------------------------------------------------------------------------------------

def prefill_buffers(kda, x, dev, with_ws=True):
    import torch
    total, H, dk = x["k"].shape
    dv = x["v"].shape[2]
    n_seq = len(x["lengths"])
    offs = kda.snapshot_offsets(x["lengths"], device=dev)
    b = {"offs": offs,
         "snaps": torch.empty((int(offs[-1]), H, dk, dv), dtype=torch.float32, device=dev),
         "S_final": torch.empty((n_seq, H, dk, dv), dtype=torch.float32, device=dev),
         "o": torch.empty((total, H, dv), dtype=torch.bfloat16, device=dev)}
    if with_ws:
        b["ws"] = torch.empty(max(kda.workspace_bytes(n_seq, total, H, dk, dv), 1),
                              dtype=torch.uint8, device=dev)
    b["tiny_ws"] = torch.empty(16, dtype=torch.uint8, device=dev)  # too small: single pass
    return b


def time_two_pass(kda, x, b, stream, steps, warmup, world, clock_gpu=None, single_pass=False):
    """Time `steps` prefill steps, each the two passes as split-phase calls
    (chunk preparation, then the state pass) with CUDA events around each on
    the launching stream; returns the per-pass mean times, the step time and
    the clock summary when a GPU id is given.  single_pass: one call without
    a workspace per step instead (the single-pass kernel; its time is
    reported as the state pass, the preparation time as 0)."""
    import torch

    def step(e=None):
        if single_pass:
            if e is not None:
                e[0].record(stream)
                e[1].record(stream)
            kda.chunk_fwd(x["q"], x["k"], x["v"], x["z"], x["beta"], x["A"],
                          cu_seqlens=x["cu_seqlens"], S0=x.get("S0"), o=b["o"],
                          S_final=b["S_final"], snaps=b["snaps"], snap_offsets=b["offs"],
                          workspace=b["tiny_ws"], stream=stream)
            if e is not None:
                e[2].record(stream)
            return
        if e is not None:
            e[0].record(stream)
        kda.chunk_fwd(x["q"], x["k"], x["v"], x["z"], x["beta"], x["A"],
                      cu_seqlens=x["cu_seqlens"], S0=x.get("S0"), o=b["o"],
                      S_final=b["S_final"], snaps=b["snaps"], snap_offsets=b["offs"],
                      workspace=b["ws"], pre=kda.PASS_PREPARE, stream=stream)
        if e is not None:
            e[1].record(stream)
        kda.chunk_fwd(x["q"], x["k"], x["v"], x["z"], x["beta"], x["A"],
                      cu_seqlens=x["cu_seqlens"], S0=x.get("S0"), o=b["o"],
                      S_final=b["S_final"], snaps=b["snaps"], snap_offsets=b["offs"],
                      workspace=b["ws"], pre=kda.PASS_STATE, stream=stream)
        if e is not None:
            e[2].record(stream)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    if kda.device_status() != 0:
        raise RuntimeError("device status word set during warm-up")
    ev = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(3)) for _ in range(steps)]
    barrier(world)
    torch.cuda.synchronize()
    clocks = ClockSampler(clock_gpu) if clock_gpu is not None else None
    if clocks is not None:
        clocks.__enter__()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    h0 = time.monotonic()
    t0.record(stream)
    for i in range(steps):
        step(ev[i])
    t1.record(stream)
    torch.cuda.synchronize()
    if clocks is not None:
        clocks.window(h0, time.monotonic())
        clocks.__exit__(None, None, None)
    barrier(world)
    if kda.device_status() != 0:
        raise RuntimeError("device status word set during the timed steps")
    return {"elapsed_ms": reduce_max(t0.elapsed_time(t1), world),
            "prep_s": statistics.mean(a.elapsed_time(bb) for a, bb, _ in ev) / 1e3,
            "state_s": statistics.mean(bb.elapsed_time(c) for _, bb, c in ev) / 1e3,
            "step_s": statistics.mean(a.elapsed_time(c) for a, _, c in ev) / 1e3,
            "clocks": clocks.summary() if clocks is not None else None}


def prefill_roofline(name, t, hbm_peak, tc_peak, peak_src, s0):
    """Roofline of the dominant kernel of one prefill step (algorithmic bytes)
    and of the whole step."""
    w = workload_params(name)
    L = workload_lengths(name)
    H, dk, dv = w["H"], w["dk"], w["dv"]
    token_heads = sum(L) * H
    chunk_heads = sum((l + 63) // 64 for l in L) * H
    full_heads = sum(l // 64 for l in L) * H
    seq_heads = len(L) * H
    kernels = {
        "chunk_prep_kernel": (t["prep_s"], prep_bytes(token_heads, dk, dv)),
        "state_pass_kernel": (t["state_s"], state_bytes(token_heads, full_heads, seq_heads, dk,
                                                        dv, s0=s0)),
    }
    dom = max(kernels, key=lambda k: kernels[k][0])
    dom_s, dom_bytes = kernels[dom]
    achieved = dom_bytes / dom_s / 1e9
    alg = prefill_bytes(token_heads, seq_heads, dk, dv, s0=s0, full_chunk_heads=full_heads)
    flops = prefill_flops(token_heads, dk, dv)
    return {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
            "frac": achieved / hbm_peak, "traffic": profiled_traffic(dom, chunk_heads),
            "kernel": dom, "bytes_per_launch": dom_bytes, "launch_ms": 1e3 * dom_s,
            "peak_source": peak_src + " (HBM copy bandwidth)",
            "passes_ms": {k: 1e3 * v[0] for k, v in kernels.items()},
            "traffic_overhead": {
                "what": "the two-pass records: written by the chunk preparation, read by the "
                        "state pass (not algorithmic bytes)",
                "bytes_per_step": 2 * chunk_heads * REC_BYTES},
            "path": {"what": "whole prefill step (both passes) against the algorithmic bytes "
                             "of its inputs and outputs",
                     "bytes": alg, "achieved": alg / t["step_s"] / 1e9,
                     "frac": alg / t["step_s"] / 1e9 / hbm_peak},
            "tensor": {"achieved_tflops": flops / t["step_s"] / 1e12, "peak_tflops": tc_peak,
                       "frac": flops / t["step_s"] / 1e12 / tc_peak}}


def run_ours(args, rank, world, local):
    import torch

    import kda_inputs
    import linear_attention_serving_chunk_gb300 as kda

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    kda.build()
    kda.lib()
    hbm_peak, tc_peak, tc_sus, peak_src = load_peaks()
    stream = torch.cuda.current_stream(dev)
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid).replace("GPU-", "")
    except Exception:
        gpu_id = local

    # the headline: the packed varlen prefill
    x = make_workload(WORKLOAD, dev)
    b = prefill_buffers(kda, x, dev, with_ws=not args.single_pass)
    t = time_two_pass(kda, x, b, stream, args.steps, args.warmup, world, clock_gpu=gpu_id,
                      single_pass=args.single_pass)
    n_tok = x["k"].shape[0]
    value = n_tok * args.steps * world / (t["elapsed_ms"] / 1e3)
    roofline = prefill_roofline(WORKLOAD, t, hbm_peak, tc_peak, peak_src,
                                s0=x.get("S0") is not None)

    # the end-to-end line first: its pinned host buffers (42 GB) are allocated
    # before the oracle sample's host arrays exist
    e2e = None if (args.no_e2e or args.single_pass) else run_e2e(args, x, b, stream, world)
    cpu_baseline = None
    if rank == 0 and not args.no_cpu_baseline:
        import oracle
        cat, n_s = oracle_sample(x, args.cpu_tokens)
        dts = time_oracle(cat, 1)
        del cat
        cpu_baseline = {"value": n_s / dts[0], "unit": UNIT, "cores": oracle.num_threads(),
                        "kind": "oracle", "sample": sample_desc(WORKLOAD, args.cpu_tokens, n_s)}
    del x, b
    torch.cuda.empty_cache()

    mid = None if args.no_mid else run_mid(args, dev, stream, hbm_peak, tc_peak, peak_src, world)
    long_ctx = None if args.no_long else run_long(args, dev, stream, hbm_peak, peak_src, world)
    decode = None if args.no_decode else run_decode(args, dev, stream, hbm_peak, peak_src, world)
    tiny = None if args.no_tiny else run_tiny(args, dev, stream, world)
    restore = None if args.no_restore else run_restore(args, dev, stream, hbm_peak, peak_src,
                                                       world)

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": t["elapsed_ms"] / args.steps, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": kda_dtype(),
                "data": "synthetic", "config": workload_config(WORKLOAD),
                "clocks": t["clocks"], "roofline": roofline, "cpu_baseline": cpu_baseline,
                "e2e": e2e, "gpu_launches": (1 if args.single_pass else 3) * args.steps,
                "prefill_path": "single pass (no workspace)" if args.single_pass else
                                "two passes (chunk preparation, state pass)",
                "mid": mid, "long_context": long_ctx, "decode": decode, "tiny": tiny,
                "restore": restore}
        print(json.dumps(line), flush=True)


def host_mem_available():
    """Bytes of host memory this process may still use (MemAvailable, capped
    by a cgroup limit when there is one)."""
    avail = None
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    avail = int(line.split()[1]) * 1024
    except OSError:
        pass
    for path in ("/sys/fs/cgroup/memory.max", "/sys/fs/cgroup/memory/memory.limit_in_bytes"):
        try:
            with open(path) as f:
                lim = f.read().strip()
            if lim.isdigit():
                used = 0
                for upath in ("/sys/fs/cgroup/memory.current",
                              "/sys/fs/cgroup/memory/memory.usage_in_bytes"):
                    try:
                        with open(upath) as g:
                            used = int(g.read().strip())
                        break
                    except OSError:
                        continue
                room = int(lim) - used
                avail = room if avail is None else min(avail, room)
        except OSError:
            continue
    return avail


def host_fits_all_ranks(nbytes, world, avail=None):
    """True on every rank when each node has nbytes of host memory for each of
    its ranks (LOCAL_WORLD_SIZE), else False on every rank: a line with
    barriers is then run by all ranks or by none."""
    if avail is None:
        avail = host_mem_available()
    local_ranks = max(1, int(os.environ.get("LOCAL_WORLD_SIZE", "1")))
    short = avail is not None and nbytes * local_ranks > avail
    return reduce_max(1.0 if short else 0.0, world) == 0.0


def agreed_capture(ms, err, world):
    """A graph-replay time agreed on by every rank: (the maximum over ranks,
    None) when every rank captured its graph (ms not None), else (None, the
    reason: this rank's own error, or "on another rank").  Collective: every
    rank calls it exactly once, whether its own capture worked or not."""
    if reduce_max(1.0 if ms is None else 0.0, world) == 0.0:
        return reduce_max(ms, world), None
    return None, (err if ms is None else "on another rank")


def run_e2e(args, x, b, stream, world):
    """The same step through the public API with host buffers: every step copies
    its inputs from pinned host memory to the device, runs kda_chunk_fwd
    (snapshots included) and copies its result, o and the final states, back
    to pinned host memory, all inside the timed region.  The chunk snapshots
    stay in device memory: they are the prefix cache, which kda_state_snapshot
    restores from there.  Steps are pipelined over two buffer slots on three
    streams (inputs in, compute, outputs out), as a serving loop would run
    them: step i's outputs go back while step i+1's inputs come in.  The
    compute of the steps is serialised on one stream, so the snapshot array
    and the workspace are shared by the slots."""
    import torch

    import linear_attention_serving_chunk_gb300 as kda
    dev = b["o"].device
    names_in = ("q", "k", "v", "z", "beta", "A", "cu_seqlens", "S0")
    h2d = sum(x[n].numel() * x[n].element_size() for n in names_in)
    d2h = sum(b[n].numel() * b[n].element_size() for n in ("o", "S_final"))
    if not host_fits_all_ranks(2 * (h2d + d2h), world):
        return {"value": None, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "skipped": f"needs {(h2d + d2h) / 1e9:.1f} GB of pinned host memory per rank, "
                           "more than some node has for all of its ranks"}
    host_in = {n: x[n].cpu().pin_memory() for n in names_in}
    host_out = {n: torch.empty_like(b[n], device="cpu").pin_memory() for n in ("o", "S_final")}
    slots = [{"in": {n: x[n] for n in names_in}, "out": {"o": b["o"], "S_final": b["S_final"]}},
             {"in": {n: torch.empty_like(x[n]) for n in names_in},
              "out": {"o": torch.empty_like(b["o"]), "S_final": torch.empty_like(b["S_final"])}}]
    s_comp, s_in, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    ev = {k: [torch.cuda.Event() for _ in range(2)] for k in ("in", "out", "comp")}
    used = [False, False]

    def e2e_step(i):
        sl = i & 1
        d = slots[sl]
        if used[sl]:  # this slot's previous compute has read its inputs
            s_in.wait_event(ev["comp"][sl])
        with torch.cuda.stream(s_in):
            for n in names_in:
                d["in"][n].copy_(host_in[n], non_blocking=True)
        ev["in"][sl].record(s_in)
        s_comp.wait_event(ev["in"][sl])
        if used[sl]:  # and its previous outputs have left
            s_comp.wait_event(ev["out"][sl])
        kda.chunk_fwd(d["in"]["q"], d["in"]["k"], d["in"]["v"], d["in"]["z"], d["in"]["beta"],
                      d["in"]["A"], cu_seqlens=d["in"]["cu_seqlens"], S0=d["in"]["S0"],
                      o=d["out"]["o"], S_final=d["out"]["S_final"], snaps=b["snaps"],
                      snap_offsets=b["offs"], workspace=b["ws"], stream=s_comp)
        ev["comp"][sl].record(s_comp)
        s_out.wait_event(ev["comp"][sl])
        with torch.cuda.stream(s_out):
            for n in ("o", "S_final"):
                host_out[n].copy_(d["out"][n], non_blocking=True)
        ev["out"][sl].record(s_out)
        used[sl] = True

    for i in range(2):  # warm-up: both slots once
        e2e_step(i)
    torch.cuda.synchronize()
    link = host_link(slots[0], host_in, host_out, names_in, s_in, s_out, h2d, d2h)
    e2e_steps = max(2, min(args.steps, 10))
    barrier(world)
    a = torch.cuda.Event(enable_timing=True)
    bb = torch.cuda.Event(enable_timing=True)
    a.record(s_comp)
    s_in.wait_event(a)
    for i in range(e2e_steps):
        e2e_step(i)
    s_comp.wait_event(ev["out"][(e2e_steps - 1) & 1])  # the end waits for the last copy out
    bb.record(s_comp)
    torch.cuda.synchronize()
    e2e_ms = reduce_max(a.elapsed_time(bb), world)
    n_tok = x["k"].shape[0]
    out = {"value": n_tok * e2e_steps * world / (e2e_ms / 1e3), "unit": UNIT,
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
           "ms_per_step": e2e_ms / e2e_steps,
           "d2h": "o and final states; the chunk snapshots are computed every step and stay in "
                  "device memory (the prefix cache)",
           "pipelined": "2 buffer slots; copies in and out on their own streams, compute on 1",
           "link": link}
    del host_in, host_out, slots
    return out


def host_link(slot, host_in, host_out, names_in, s_in, s_out, h2d, d2h):
    """The host link as this run sees it, just before the end-to-end region:
    one step's inputs copied in alone, then its outputs copied out alone, each
    timed with CUDA events on its copy stream.  floor_ms = the slower of the
    two directions, the least an end-to-end step can take; on a machine shared
    with other jobs this link's bandwidth is not constant from run to run."""
    import torch

    def timed(stream, copies):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record(stream)
        with torch.cuda.stream(stream):
            for dst, src in copies:
                dst.copy_(src, non_blocking=True)
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b)

    t_in = timed(s_in, [(slot["in"][n], host_in[n]) for n in names_in])
    t_out = timed(s_out, [(host_out[n], slot["out"][n]) for n in ("o", "S_final")])
    return {"h2d_gbs": h2d / t_in / 1e6, "d2h_gbs": d2h / t_out / 1e6,
            "floor_ms": max(t_in, t_out),
            "how": "one step's inputs in alone, then its outputs out alone, CUDA events"}


def kda_dtype():
    import linear_attention_serving_chunk_gb300 as kda
    return getattr(kda, "PREFILL_COMPUTE_DTYPE", "f32")


def run_mid(args, dev, stream, hbm_peak, tc_peak, peak_src, world):
    """The B=4 H=16 T=8192 prefill (final states and snapshots), the two passes
    timed as in the headline."""
    import torch

    import kda_inputs
    import linear_attention_serving_chunk_gb300 as kda
    x = make_workload("mid", dev)
    b = prefill_buffers(kda, x, dev)
    steps = max(args.steps, 50)
    t = time_two_pass(kda, x, b, stream, steps, args.warmup, world)
    n_tok = x["k"].shape[0]
    del x, b
    torch.cuda.empty_cache()
    return {"value": n_tok * steps * world / (t["elapsed_ms"] / 1e3), "unit": UNIT,
            "ms_per_step": t["elapsed_ms"] / steps, "steps": steps,
            "workload": workload_config("mid")["workload"],
            "roofline": prefill_roofline("mid", t, hbm_peak, tc_peak, peak_src, s0=False)}


def run_decode(args, dev, stream, hbm_peak, peak_src, world):
    """1000 chained decode steps (512 x 32 states, dk=dv=128) with fresh inputs."""
    import torch

    import kda_inputs
    import linear_attention_serving_chunk_gb300 as kda
    w = kda_inputs.WORKLOADS["decode"]
    Bd, H, dk, dv, n_steps = w["batch"], w["H"], w["dk"], w["dv"], args.decode_steps
    pool, A = kda_inputs.make_decode_state(Bd, H, dk, dv, w["seed"], device=dev,
                                           std=w["state_std"])
    toks = [kda_inputs.make_decode_token(Bd, H, dk, dv, w["seed"], s, device=dev)
            for s in range(max(n_steps, 3))]
    o = torch.empty((Bd, H, dv), dtype=torch.bfloat16, device=dev)

    def one(s):
        t = toks[s]
        kda.decode_step(t["q"], t["k"], t["v"], t["z"], t["beta"], A, pool, o=o, stream=stream)

    for s in range(3):
        one(s)
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(n_steps)]
    barrier(world)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for s in range(n_steps):
        evs[s][0].record(stream)
        one(s)
        evs[s][1].record(stream)
    b.record(stream)
    torch.cuda.synchronize()
    total_ms = reduce_max(a.elapsed_time(b), world)
    per = statistics.mean(x.elapsed_time(y) for x, y in evs) / 1e3
    nbytes = decode_bytes(Bd * H, dk, dv)
    achieved = nbytes / per / 1e9
    # the same chained steps captured in one CUDA graph, replayed once untimed
    # and once timed (the first replay uploads the graph).  No collective runs
    # inside the try: whether every rank captured is agreed on after it.
    graph_ms, graph_err = None, None
    try:
        side = torch.cuda.Stream(device=dev)  # captures need a stream other than the default
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=side):
            for s in range(n_steps):
                t = toks[s]
                kda.decode_step(t["q"], t["k"], t["v"], t["z"], t["beta"], A, pool, o=o,
                                stream=side)
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        cur = torch.cuda.current_stream(dev)
        a.record(cur)
        graph.replay()
        b.record(cur)
        torch.cuda.synchronize()
        graph_ms = a.elapsed_time(b)
        del graph
    except RuntimeError as e:  # capture not possible here: the issued figure only
        graph_err = str(e)
    graph_ms, graph_err = agreed_capture(graph_ms, graph_err, world)
    if graph_ms is not None:
        graph_line = {"value": n_steps * world / (graph_ms / 1e3), "unit": "steps/s",
                      "ms_per_step": graph_ms / n_steps,
                      "how": f"the {n_steps} steps captured in one CUDA graph, replayed once"}
    else:
        graph_line = f"not captured: {graph_err}"
    multi = run_decode_tokens(kda, pool, A, Bd, H, dk, dv, w["seed"], dev, stream, hbm_peak,
                              world)
    return {"value": n_steps * world / (total_ms / 1e3), "unit": "steps/s",
            "graph": graph_line,
            "multi_token": multi,
            "tokens_per_s": Bd * n_steps * world / (total_ms / 1e3),
            "workload": f"kda decode {Bd} sequences x H={H}, dk=dv={dk}, fp32 state in place, "
                        f"{n_steps} chained steps with fresh inputs",
            "gpu_launches": n_steps,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                         "frac": achieved / hbm_peak,
                         "traffic": profiled_traffic("kda_decode_step", Bd * H),
                         "kernel": "kda_decode_step", "peak_source": peak_src}}


def run_decode_tokens(kda, pool, A, Bd, H, dk, dv, seed, dev, stream, hbm_peak, world,
                      tokens=4, reps=20):
    """Speculative verification: `tokens` tokens per sequence on the same
    512 x 32 resident states (kda_decode_tokens, commit = 0: every state is
    read once, none is written), timed over `reps` calls."""
    import torch

    import kda_inputs
    x = kda_inputs.make_prefill(H, dk, dv, [tokens] * Bd, seed + 7, device=dev)
    slots = torch.arange(Bd, dtype=torch.int32, device=dev)
    o = torch.empty((Bd * tokens, H, dv), dtype=torch.bfloat16, device=dev)

    def call():
        kda.decode_tokens(x["q"], x["k"], x["v"], x["z"], x["beta"], A, pool, slots,
                          x["cu_seqlens"], commit=False, o=o, stream=stream)

    for _ in range(3):
        call()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(reps):
        call()
    b.record(stream)
    torch.cuda.synchronize()
    ms = reduce_max(a.elapsed_time(b), world) / reps
    # the state read once, the tokens' inputs and outputs
    nbytes = Bd * H * (dk * dv * 4 + tokens * (2 * (3 * dk + 2 * dv) + 2))
    return {"tokens_per_seq": tokens, "ms_per_call": ms, "unit": "tokens/s",
            "value": Bd * tokens * world / (ms / 1e3),
            "workload": f"kda_decode_tokens: {tokens} tokens on each of {Bd} x H={H} states, "
                        f"dk=dv={dk}, commit = 0 (verify)",
            "roofline": {"bound": "hbm", "achieved": nbytes / (ms / 1e3) / 1e9,
                         "peak": hbm_peak, "unit": "GB/s",
                         "frac": nbytes / (ms / 1e3) / 1e9 / hbm_peak,
                         "traffic": profiled_traffic("decode_tokens_kernel", Bd * H),
                         "kernel": "decode_tokens_kernel"}}


def run_long(args, dev, stream, hbm_peak, peak_src, world):
    """The long-context prefill: one sequence of 1,048,576 tokens, H = 16,
    dk = dv = 128, final state and chunk snapshots (the path the library picks
    for it: the segment-parallel scan)."""
    import torch

    import kda_inputs
    import linear_attention_serving_chunk_gb300 as kda
    w = kda_inputs.WORKLOADS["long"]
    B, H, T, dk, dv = w["B"], w["H"], args.long_len or w["T"], w["dk"], w["dv"]
    x = kda_inputs.make_workload_prefill("long", device=dev, T=T)
    snaps = torch.empty((B * (T // 64), H, dk, dv), dtype=torch.float32, device=dev)
    S_final = torch.empty((B, H, dk, dv), dtype=torch.float32, device=dev)
    o = torch.empty((B * T, H, dv), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(max(kda.workspace_bytes(B, B * T, H, dk, dv), 1), dtype=torch.uint8,
                     device=dev)

    def step():
        kda.chunk_fwd(x["q"], x["k"], x["v"], x["z"], x["beta"], x["A"], n_seq=B, o=o,
                      S_final=S_final, snaps=snaps, workspace=ws, stream=stream)

    for _ in range(2):
        step()
    torch.cuda.synchronize()
    n = args.long_steps
    barrier(world)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(n):
        step()
    b.record(stream)
    torch.cuda.synchronize()
    ms = reduce_max(a.elapsed_time(b), world) / n
    nbytes = prefill_bytes(B * T * H, B * H, dk, dv)
    del x, snaps, o, ws
    torch.cuda.empty_cache()
    return {"value": B * T * world / (ms / 1e3), "unit": UNIT, "ms_per_step": ms, "steps": n,
            "workload": f"kda prefill B={B} H={H} T={T} dk={dk} dv={dv} chunk=64, final state + "
                        "chunk snapshots",
            "path": {"what": "whole step against the algorithmic bytes of inputs and outputs",
                     "achieved": nbytes / (ms / 1e3) / 1e9,
                     "frac": nbytes / (ms / 1e3) / 1e9 / hbm_peak, "unit": "GB/s",
                     "peak": hbm_peak, "peak_source": peak_src}}


def run_restore(args, dev, stream, hbm_peak, peak_src, world):
    """Prefix-cache restore (kda_state_snapshot): 512 x 32 chunk-boundary
    states (dk = dv = 128, 1 GiB) gathered from a snapshot array into state
    slots in a permuted order; a pure HBM copy, timed over --restore-reps
    calls."""
    import torch

    import linear_attention_serving_chunk_gb300 as kda
    n, H, d, rows = 512, 32, 128, 1024
    snaps = torch.randn((rows, H, d, d), dtype=torch.float32, device=dev)
    pool = torch.empty((n, H, d, d), dtype=torch.float32, device=dev)
    g = torch.Generator(device="cpu")
    g.manual_seed(1005)
    src = torch.randperm(rows, generator=g)[:n].to(torch.int64).to(dev)
    dst = torch.randperm(n, generator=g).to(torch.int32).to(dev)
    for _ in range(3):
        kda.state_snapshot(snaps, src, pool, dst, stream=stream)
    torch.cuda.synchronize()
    reps = args.restore_reps
    a = torch.cuda.Event(enable_timing=True)
    bb = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(reps):
        kda.state_snapshot(snaps, src, pool, dst, stream=stream)
    bb.record(stream)
    torch.cuda.synchronize()
    ms = reduce_max(a.elapsed_time(bb), world) / reps
    nbytes = 2 * n * H * d * d * 4
    ok = bool(torch.equal(pool[dst[:4].long()], snaps[src[:4]]))
    del snaps, pool
    torch.cuda.empty_cache()
    return {"value": n * world / (ms / 1e3), "unit": "states/s", "ms_per_call": ms,
            "reps": reps, "workload": f"restore {n} x H={H} snapshot states, dk=dv={d}",
            "copy_exact": ok,
            "roofline": {"bound": "hbm", "achieved": nbytes / (ms / 1e3) / 1e9,
                         "peak": hbm_peak, "unit": "GB/s",
                         "frac": nbytes / (ms / 1e3) / 1e9 / hbm_peak,
                         "traffic": profiled_traffic("snapshot_restore_kernel", n * H),
                         "kernel": "snapshot_restore_kernel", "peak_source": peak_src}}


def run_tiny(args, dev, stream, world):
    """Latency of the tiny prefill (B=1, H=2, T=256, dk=dv=64, final state and
    snapshots): launch-bound, so reported as microseconds per call, back to
    back (no flush: its inputs fit in L2)."""
    import torch

    import kda_inputs
    import linear_attention_serving_chunk_gb300 as kda
    x = kda_inputs.make_workload_prefill("tiny", device=dev)
    b = prefill_buffers(kda, x, dev)

    def call(st=stream):
        kda.chunk_fwd(x["q"], x["k"], x["v"], x["z"], x["beta"], x["A"],
                      cu_seqlens=x["cu_seqlens"], o=b["o"], S_final=b["S_final"],
                      snaps=b["snaps"], snap_offsets=b["offs"], workspace=b["ws"],
                      stream=st)

    for _ in range(10):
        call()
    torch.cuda.synchronize()
    reps = args.tiny_reps
    a = torch.cuda.Event(enable_timing=True)
    bb = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(reps):
        call()
    bb.record(stream)
    torch.cuda.synchronize()
    us = reduce_max(a.elapsed_time(bb), world) * 1e3 / reps
    # the same call captured once in a CUDA graph and replayed: the GPU's own
    # latency of the three launches, without the host's per-call work
    # (argument checks, tensor-map encoding, the Python binding)
    # (no collective inside the try: whether every rank captured is agreed on after it)
    graph_ms, graph_err = None, None
    try:
        side = torch.cuda.Stream(device=dev)  # captures need a stream other than the default
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            call(side)
        side.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            call(side)
        torch.cuda.synchronize()
        for _ in range(10):
            g.replay()
        torch.cuda.synchronize()
        cur = torch.cuda.current_stream(dev)
        a.record(cur)
        for _ in range(reps):
            g.replay()
        bb.record(cur)
        torch.cuda.synchronize()
        graph_ms = a.elapsed_time(bb)
        del g
    except RuntimeError as e:  # capture not possible here: report the host-issued figure only
        graph_err = str(e)
    graph_ms, graph_err = agreed_capture(graph_ms, graph_err, world)
    graph_us = graph_ms * 1e3 / reps if graph_ms is not None else f"not captured: {graph_err}"
    if kda.device_status() != 0:
        raise RuntimeError("device status word set during the tiny prefill")
    return {"latency_us": us, "unit": "us per call", "reps": reps,
            "graph_replay_us": graph_us,
            "workload": workload_config("tiny")["workload"],
            "gpu_launches_per_call": 3,
            "note": "launch-bound: three kernels (chunk-start table, chunk preparation, state "
                    "pass) per call, back to back on one stream; latency_us issues every call "
                    "from Python, graph_replay_us replays it from a CUDA graph"}


def main(argv=None):
    global WORKLOAD
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--decode-steps", type=int, default=1000)
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-mid", action="store_true", help="skip the B=4 T=8192 prefill line")
    ap.add_argument("--no-long", action="store_true", help="skip the 1M-token prefill line")
    ap.add_argument("--no-tiny", action="store_true", help="skip the tiny-prefill latency line")
    ap.add_argument("--long-steps", type=int, default=3)
    ap.add_argument("--tiny-reps", type=int, default=1000)
    ap.add_argument("--no-restore", action="store_true", help="skip the snapshot-restore line")
    ap.add_argument("--restore-reps", type=int, default=20)
    ap.add_argument("--long-len", type=int, default=None,
                    help="override T of the long-context line (small cases for profiling)")
    ap.add_argument("--single-pass", action="store_true",
                    help="run the headline prefill without a workspace (the single-pass "
                         "kernel), for comparison and profiling")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-tokens", type=int, default=2048,
                    help="tokens per sequence in the cpu_baseline sample (one timed run)")
    ap.add_argument("--ref-tokens", type=int, default=128,
                    help="tokens per sequence in each step of the reference arm")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--workload", choices=("varlen", "mid", "long", "tiny"), default=WORKLOAD,
                    help="prefill workload of the headline (default: the varlen batch)")
    ap.add_argument("--seq-len", type=int, default=None,
                    help="override the sequence length (equal-length workloads; small cases "
                         "for profiling)")
    ap.add_argument("--n-seq", type=int, default=None,
                    help="override the number of sequences (small cases for profiling)")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)  # at least three untimed warm-up steps
    WORKLOAD = args.workload
    _OVERRIDE.update(seq_len=args.seq_len, n_seq=args.n_seq)
    if WORKLOAD == "mid":
        args.no_mid = True
    rank, world, local = dist_setup(args.gpus)
    init_pg(world)
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
