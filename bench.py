"""KDA prefill / decode benchmark on GB300.

One step = one kda_chunk_fwd over the prefill workload B=4, H=16, T=8192,
dk=dv=128, chunk=64, with the final state and every chunk-boundary snapshot
written (inputs larger than L2).  The decode step (512 x 32 resident states,
dk=dv=128, 1000 chained steps) is measured in the same run and reported as
its own object.  Prints ONE JSON line on rank 0.

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
WORKLOAD = "mid"

# Algorithmic traffic and work per token-head at chunk 64 (bf16 in/out, fp32 states):
#   q, k, z (dk each), v, o (dv each) in bf16 plus beta: 2 (3 dk + 2 dv) + 2 bytes;
#   chunk-boundary snapshots: 4 dk dv / 64 bytes;
#   flops: 6 dk dv + 64 (3 dk + 2 dv) + 64^2 / 3 (causal halves once, masked tiles not counted).


def prefill_bytes(token_heads, seq_heads, dk, dv, snapshots=True, s0=False, s_final=True):
    b = token_heads * (2 * (3 * dk + 2 * dv) + 2)
    if snapshots:
        b += token_heads * 4 * dk * dv // 64
    b += seq_heads * 4 * dk * dv * (int(s0) + int(s_final))
    return b


REC_BYTES = 74240  # bytes of one (chunk, head) record the two passes exchange


def prep_bytes(token_heads, chunk_heads, dk, dv):
    """Chunk preparation: reads q, k, z, v, beta; writes one record per chunk-head."""
    return token_heads * (2 * (3 * dk + dv) + 2) + chunk_heads * REC_BYTES


def state_bytes(token_heads, chunk_heads, full_chunk_heads, seq_heads, dk, dv):
    """State pass: reads the records; writes o, the snapshots and the final states."""
    return (chunk_heads * REC_BYTES + token_heads * 2 * dv + full_chunk_heads * 4 * dk * dv +
            seq_heads * 4 * dk * dv)


# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one launch from
# the ncu captures summarised under profiles/, taken on 4096 (chunk, head)
# tasks (B=4 H=16 T=4096) and scaled here by the tasks of the timed launch.
# They are reported only while the kernel's sources hash to the sha256 prefix
# recorded with the capture (else the kernel has changed since: null).
_CSRC = os.path.join(ROOT, "linear_attention_serving_chunk_gb300", "csrc")
PROFILED_TRAFFIC = {
    "prefill_tc_kernel<prep>": (269.252352e6 + 250.642944e6, 4096, "4e96eed0f04c6a83",
                                ("kda_prefill_tc.cu", "kda_tc_common.cuh", "kda_sm100.cuh",
                                 "kda_split.cuh", "kda_common.cuh")),
    "state_pass_kernel": (304.155136e6 + 289.254656e6, 4096, "a492962f1c96c2cf",
                          ("kda_state_pass.cu", "kda_tc_common.cuh", "kda_sm100.cuh",
                           "kda_split.cuh", "kda_common.cuh")),
    "kda_decode_step": (1.090611e9 + 1.017646e9, 16384, "d7fab05fc3519b6c",
                        ("kda_decode.cu", "kda_common.cuh")),
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


# --- reference arm: the fp64 oracle on the host cores --------------------------------------

def oracle_sample(x, n_tokens):
    """Host fp64 copies of the first n_tokens of every sequence, all heads."""
    import numpy as np
    import torch
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
    cat["cu"] = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    del torch
    return cat, int(sum(lens))


def time_oracle(cat, steps):
    import oracle
    dts = []
    for _ in range(steps):
        t = time.perf_counter()
        oracle.prefill(cat["q"], cat["k"], cat["v"], cat["z"], cat["beta"], cat["A"],
                       cu_seqlens=cat["cu"], snapshots=True)
        dts.append(time.perf_counter() - t)
    return dts


def run_reference(args, rank, world):
    import kda_inputs
    import oracle
    if rank != 0:
        return
    w = kda_inputs.WORKLOADS[WORKLOAD]
    x = kda_inputs.make_workload_prefill(WORKLOAD, device="cpu")
    cat, n_tok = oracle_sample(x, args.ref_tokens)
    H = w["H"]
    time_oracle(cat, args.warmup)
    dts = time_oracle(cat, args.steps)
    total = sum(dts)
    value = n_tok * args.steps / total  # tokens (all H heads) per second
    cores = oracle.num_threads()
    sample = (f"first {args.ref_tokens} tokens of each of the {w['B']} sequences, all {H} heads "
              f"({n_tok * H} token-heads per step), snapshots on")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": workload_config(w),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def workload_config(w):
    return {"workload": f"kda prefill B={w['B']} H={w['H']} T={w['T']} dk={w['dk']} "
                        f"dv={w['dv']} chunk={w['chunk']}, final state + chunk snapshots",
            "global_batch": w["B"], "seq_len": w["T"], "heads": w["H"],
            "l2": "inputs larger than L2 (~1.2 GB of HBM traffic per step), no flush"}


# --- our arm ------------------------------------------------------------------------------------

def run_ours(args, rank, world, local):
    import numpy as np
    import torch

    import kda_inputs
    import linear_attention_serving_chunk_gb300 as kda

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    kda.build()
    kda.lib()
    hbm_peak, tc_peak, tc_sus, peak_src = load_peaks()
    w = dict(kda_inputs.WORKLOADS[WORKLOAD])
    if args.seq_len:
        w["T"] = args.seq_len
    B, H, T, dk, dv = w["B"], w["H"], w["T"], w["dk"], w["dv"]
    x = kda_inputs.make_workload_prefill(WORKLOAD, device=dev, T=T)
    offs = kda.snapshot_offsets(x["lengths"], device=dev)
    snaps = torch.empty((int(offs[-1]), H, dk, dv), dtype=torch.float32, device=dev)
    S_final = torch.empty((B, H, dk, dv), dtype=torch.float32, device=dev)
    o = torch.empty((B * T, H, dv), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)

    ws_bytes = kda.workspace_bytes(B, B * T, H, dk, dv)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)

    # One step = the two passes of the prefill, as two split-phase calls so
    # that each pass is timed on its own: chunk preparation (the chunk-start
    # table + the preparation kernel), then the state pass.
    def step(e=None):
        if e is not None:
            e[0].record(stream)
        kda.chunk_fwd(x["q"], x["k"], x["v"], x["z"], x["beta"], x["A"],
                      cu_seqlens=x["cu_seqlens"], o=o, S_final=S_final, snaps=snaps,
                      snap_offsets=offs, workspace=ws, pre=kda.PASS_PREPARE, stream=stream)
        if e is not None:
            e[1].record(stream)
        kda.chunk_fwd(x["q"], x["k"], x["v"], x["z"], x["beta"], x["A"],
                      cu_seqlens=x["cu_seqlens"], o=o, S_final=S_final, snaps=snaps,
                      snap_offsets=offs, workspace=ws, pre=kda.PASS_STATE, stream=stream)
        if e is not None:
            e[2].record(stream)
    launches_per_step = 3  # chunk-start table, chunk preparation, state pass

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if kda.device_status() != 0:
        raise RuntimeError("device status word set during warm-up")

    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid).replace("GPU-", "")
    except Exception:
        gpu_id = local
    ev = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(3))
          for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(gpu_id) as clocks:
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        h0 = time.monotonic()
        t0.record(stream)
        for i in range(args.steps):
            step(ev[i])
        t1.record(stream)
        torch.cuda.synchronize()
        clocks.window(h0, time.monotonic())
    barrier(world)
    elapsed_ms = reduce_max(t0.elapsed_time(t1), world)
    prep_s = statistics.mean(a.elapsed_time(b) for a, b, _ in ev) / 1e3
    state_s = statistics.mean(b.elapsed_time(c) for _, b, c in ev) / 1e3
    step_s = statistics.mean(a.elapsed_time(c) for a, _, c in ev) / 1e3

    token_heads = B * T * H
    chunk_heads = B * ((T + 63) // 64) * H
    value = B * T * args.steps * world / (elapsed_ms / 1e3)
    alg_bytes = prefill_bytes(token_heads, B * H, dk, dv)
    alg_flops = prefill_flops(token_heads, dk, dv)
    kernels = {
        "prefill_tc_kernel<prep>": (prep_s, prep_bytes(token_heads, chunk_heads, dk, dv)),
        "state_pass_kernel": (state_s, state_bytes(token_heads, chunk_heads,
                                                    B * (T // 64) * H, B * H, dk, dv)),
    }
    dom = max(kernels, key=lambda k: kernels[k][0])
    dom_s, dom_bytes = kernels[dom]
    achieved = dom_bytes / dom_s / 1e9
    traffic = args.traffic if args.traffic is not None else profiled_traffic(dom, chunk_heads)
    roofline = {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                "frac": achieved / hbm_peak, "traffic": traffic, "kernel": dom,
                "bytes_per_launch": dom_bytes, "launch_ms": 1e3 * dom_s,
                "peak_source": peak_src,
                "passes_ms": {k: 1e3 * t for k, (t, _) in kernels.items()},
                "path": {"what": "whole prefill step (both passes), algorithmic bytes of the "
                                 "inputs and outputs only",
                         "achieved": alg_bytes / step_s / 1e9,
                         "frac": alg_bytes / step_s / 1e9 / hbm_peak},
                "tensor": {"achieved_tflops": alg_flops / step_s / 1e12,
                           "peak_tflops": tc_peak,
                           "frac": alg_flops / step_s / 1e12 / tc_peak}}

    e2e = None if args.no_e2e else run_e2e(args, x, o, S_final, snaps, offs, ws, stream, world,
                                           B, T)
    decode = None if args.no_decode else run_decode(args, dev, stream, hbm_peak, peak_src, world)
    long_ctx = None if args.no_long else run_long(args, dev, stream, hbm_peak, peak_src, world)

    cpu_baseline = None
    if rank == 0 and not args.no_cpu_baseline:
        import oracle
        cat, n_tok = oracle_sample(x, args.ref_tokens)
        dts = time_oracle(cat, 1)
        cpu_baseline = {"value": n_tok / dts[0], "unit": UNIT, "cores": oracle.num_threads(),
                        "kind": "oracle",
                        "sample": f"first {args.ref_tokens} tokens of each of the {B} sequences,"
                                  f" all {H} heads ({n_tok * H} token-heads), snapshots on"}

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": kda_dtype(),
                "data": "synthetic", "config": workload_config(w),
                "clocks": clocks.summary(), "roofline": roofline, "cpu_baseline": cpu_baseline,
                "e2e": e2e, "gpu_launches": launches_per_step * args.steps, "decode": decode,
                "long_context": long_ctx}
        print(json.dumps(line), flush=True)


def run_e2e(args, x, o, S_final, snaps, offs, ws, stream, world, B, T):
    """The same step through the public API with host buffers: every step copies
    its inputs from pinned host memory to the device, runs kda_chunk_fwd
    (snapshots included) and copies its result, o and the final states, back
    to pinned host memory, all inside the timed region.  The chunk snapshots
    stay in device memory: they are the prefix cache, which kda_state_snapshot
    restores from there.  Steps are pipelined over two buffer slots on three
    streams (inputs in, compute, outputs out), as a serving loop would run
    them: step i's outputs go back while step i+1's inputs come in."""
    import torch

    import linear_attention_serving_chunk_gb300 as kda
    dev = o.device
    names_in = ("q", "k", "v", "z", "beta", "A", "cu_seqlens")
    host_in = {n: x[n].cpu().pin_memory() for n in names_in}
    host_out = {"o": torch.empty_like(o, device="cpu").pin_memory(),
                "S_final": torch.empty_like(S_final, device="cpu").pin_memory()}
    slots = [{"in": {n: torch.empty_like(t, device=dev) for n, t in host_in.items()},
              "out": {"o": o if i == 0 else torch.empty_like(o),
                      "S_final": S_final if i == 0 else torch.empty_like(S_final),
                      "snaps": snaps if i == 0 else torch.empty_like(snaps)}}
             for i in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = sum(t.numel() * t.element_size() for t in host_out.values())
    # Copies can be split over NCS streams per direction (big tensors in
    # slices along their first dimension); on GB300 four streams per direction
    # measured no faster than one (the host link is the limit, ~275 GB/s for
    # both directions together), so one each.
    NCS = 1

    def pieces(src, dst):
        out = []
        for n, t in src.items():
            k = NCS if t.shape[0] >= NCS and t.numel() * t.element_size() > (64 << 20) else 1
            step = (t.shape[0] + k - 1) // k
            for a0 in range(0, t.shape[0], step):
                out.append((t[a0:a0 + step], dst[n][a0:a0 + step]))
        return out

    s_comp = torch.cuda.Stream(dev)
    s_in = [torch.cuda.Stream(dev) for _ in range(NCS)]
    s_out = [torch.cuda.Stream(dev) for _ in range(NCS)]
    ev = {"in": [[torch.cuda.Event() for _ in range(NCS)] for _ in range(2)],
          "out": [[torch.cuda.Event() for _ in range(NCS)] for _ in range(2)],
          "comp": [torch.cuda.Event() for _ in range(2)]}
    copies_in = [pieces(host_in, slots[sl]["in"]) for sl in range(2)]
    copies_out = [pieces({n: slots[sl]["out"][n] for n in host_out}, host_out) for sl in range(2)]
    used = [False, False]

    def e2e_step(i):
        sl = i & 1
        d = slots[sl]
        for j, st in enumerate(s_in):
            if used[sl]:  # this slot's previous compute has read its inputs
                st.wait_event(ev["comp"][sl])
            with torch.cuda.stream(st):
                for src, dst in copies_in[sl][j::NCS]:
                    dst.copy_(src, non_blocking=True)
            ev["in"][sl][j].record(st)
            s_comp.wait_event(ev["in"][sl][j])
        if used[sl]:  # and its previous outputs have left
            for j in range(NCS):
                s_comp.wait_event(ev["out"][sl][j])
        kda.chunk_fwd(d["in"]["q"], d["in"]["k"], d["in"]["v"], d["in"]["z"], d["in"]["beta"],
                      d["in"]["A"], cu_seqlens=d["in"]["cu_seqlens"], o=d["out"]["o"],
                      S_final=d["out"]["S_final"], snaps=d["out"]["snaps"], snap_offsets=offs,
                      workspace=ws, stream=s_comp)
        ev["comp"][sl].record(s_comp)
        for j, st in enumerate(s_out):
            st.wait_event(ev["comp"][sl])
            with torch.cuda.stream(st):
                for src, dst in copies_out[sl][j::NCS]:
                    dst.copy_(src, non_blocking=True)
            ev["out"][sl][j].record(st)
        used[sl] = True

    for i in range(2):  # warm-up: both slots once
        e2e_step(i)
    torch.cuda.synchronize()
    e2e_steps = max(2, min(args.steps, 10))
    barrier(world)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(s_comp)
    for st in s_in:
        st.wait_event(a)
    for i in range(e2e_steps):
        e2e_step(i)
    for j in range(NCS):  # the end waits for every stream's last copy
        s_comp.wait_event(ev["out"][(e2e_steps - 1) & 1][j])
    b.record(s_comp)
    torch.cuda.synchronize()
    e2e_ms = reduce_max(a.elapsed_time(b), world)
    e2e = {"value": B * T * e2e_steps * world / (e2e_ms / 1e3), "unit": UNIT,
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
           "d2h": "o and final states; the chunk snapshots are computed every step and stay in "
                  "device memory (the prefix cache)",
           "pipelined": f"2 buffer slots; copies in and out each on {NCS} streams, compute on 1"}
    del host_in, host_out, slots, copies_in, copies_out
    return e2e


def kda_dtype():
    import linear_attention_serving_chunk_gb300 as kda
    return getattr(kda, "PREFILL_COMPUTE_DTYPE", "f32")


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
            for s in range(n_steps)]
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
    return {"value": n_steps * world / (total_ms / 1e3), "unit": "steps/s",
            "tokens_per_s": Bd * n_steps * world / (total_ms / 1e3),
            "workload": f"kda decode {Bd} sequences x H={H}, dk=dv={dk}, fp32 state in place, "
                        f"{n_steps} chained steps with fresh inputs",
            "gpu_launches": n_steps,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                         "frac": achieved / hbm_peak,
                         "traffic": profiled_traffic("kda_decode_step", Bd * H),
                         "kernel": "kda_decode_step", "peak_source": peak_src}}


def run_long(args, dev, stream, hbm_peak, peak_src, world):
    """The long-context prefill: one sequence of 1,048,576 tokens, H = 16,
    dk = dv = 128, final state and chunk snapshots (the path the library picks
    for it: the segment-parallel scan)."""
    import torch

    import kda_inputs
    import linear_attention_serving_chunk_gb300 as kda
    w = kda_inputs.WORKLOADS["long"]
    B, H, T, dk, dv = w["B"], w["H"], w["T"], w["dk"], w["dv"]
    x = kda_inputs.make_workload_prefill("long", device=dev)
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
    return {"value": B * T * world / (ms / 1e3), "unit": UNIT, "ms_per_step": ms, "steps": n,
            "workload": f"kda prefill B={B} H={H} T={T} dk={dk} dv={dv} chunk=64, final state + "
                        "chunk snapshots",
            "path": {"what": "whole step against the algorithmic bytes of inputs and outputs",
                     "achieved": nbytes / (ms / 1e3) / 1e9,
                     "frac": nbytes / (ms / 1e3) / 1e9 / hbm_peak, "unit": "GB/s",
                     "peak": hbm_peak, "peak_source": peak_src}}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--decode-steps", type=int, default=1000)
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-long", action="store_true", help="skip the 1M-token prefill line")
    ap.add_argument("--long-steps", type=int, default=3)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ref-tokens", type=int, default=2048,
                    help="tokens per sequence in the oracle's bounded sample")
    ap.add_argument("--traffic", type=float, default=None,
                    help="ncu DRAM bytes per prefill launch, when measured for this kernel")
    ap.add_argument("--seq-len", type=int, default=None,
                    help="override T of the prefill workload (small cases for profiling)")
    ap.add_argument("--no-e2e", action="store_true")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)  # at least three untimed warm-up steps
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
