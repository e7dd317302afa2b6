"""Host-side logic: seeded input generators, the benchmark's accounting and
JSON line, and its multi-rank timing reduction (gloo, world size 2, CPU)."""
import io
import json
import os
import socket
import contextlib

import numpy as np
import pytest
import torch

import kda_inputs
import bench


def test_generators_are_deterministic_and_well_formed():
    a = kda_inputs.make_prefill(3, 64, 32, [70, 5, 0, 64], seed=9, S0_std=0.02)
    b = kda_inputs.make_prefill(3, 64, 32, [70, 5, 0, 64], seed=9, S0_std=0.02)
    for n in ("q", "k", "v", "z", "beta", "A", "S0", "cu_seqlens"):
        assert torch.equal(a[n], b[n]), n
    assert a["q"].shape == (139, 3, 64) and a["v"].shape == (139, 3, 32)
    assert a["q"].dtype == torch.bfloat16 and a["A"].dtype == torch.float32
    assert a["cu_seqlens"].tolist() == [0, 70, 75, 75, 139]
    for n in ("q", "k"):
        norms = torch.linalg.vector_norm(a[n].float(), dim=-1)
        assert torch.all((norms - 1).abs() < 2e-2)
    assert torch.all((a["beta"] > 0) & (a["beta"] < 1))
    assert torch.all(a["A"].abs() <= 1)
    c = kda_inputs.make_prefill(3, 64, 32, [70, 5, 0, 64], seed=10, S0_std=0.02)
    assert not torch.equal(a["q"], c["q"])


def test_varlen_lengths_in_range():
    w = kda_inputs.WORKLOADS["varlen"]
    L = kda_inputs.varlen_lengths(w["n_seq"], w["len_lo"], w["len_hi"], w["seed"])
    assert len(L) == 64 and min(L) >= 512 and max(L) <= 32768
    assert L == kda_inputs.varlen_lengths(w["n_seq"], w["len_lo"], w["len_hi"], w["seed"])


def test_decode_tokens_differ_per_step():
    t0 = kda_inputs.make_decode_token(4, 2, 64, 64, seed=3, step=0)
    t1 = kda_inputs.make_decode_token(4, 2, 64, 64, seed=3, step=1)
    assert not torch.equal(t0["q"], t1["q"])
    assert torch.equal(t0["q"], kda_inputs.make_decode_token(4, 2, 64, 64, seed=3, step=0)["q"])


def test_algorithmic_accounting():
    # per token-head at dk = dv = 128, chunk 64: 1282 B of q,k,z,v,o,beta,
    # 1024 B of snapshots, 140,629 flops (+1/3 from C^2/3)
    assert bench.prefill_bytes(1, 0, 128, 128, snapshots=False, s_final=False) == 1282
    assert bench.prefill_bytes(1, 0, 128, 128, snapshots=True, s_final=False) == 2306
    assert abs(bench.prefill_flops(1, 128, 128) - 140629.33) < 1
    # decode: state read + write dominate
    assert bench.decode_bytes(1, 128, 128) == 8 * 128 * 128 + 2 * 640 + 2


def test_reference_arm_line():
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.main(["--impl", "reference", "--steps", "1", "--warmup", "1", "--ref-tokens", "64"])
    line = json.loads(buf.getvalue().strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "tokens/s" and line["value"] > 0
    for key in ("metric", "n_gpus", "steps", "warmup", "ms_per_step", "config", "cpu_baseline",
                "e2e"):
        assert key in line
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    r, w, lr = bench.dist_setup(world)
    bench.init_pg(w)
    bench.barrier(w)
    got = bench.reduce_max(10.0 + r, w)
    q.put((r, got))
    import torch.distributed as dist
    dist.destroy_process_group()


def _fits_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank), LOCAL_WORLD_SIZE=str(world))
    r, w, lr = bench.dist_setup(world)
    bench.init_pg(w)
    # 10 GB per rank, two ranks on the node: rank 0's node has 30 GB, rank 1's 15 GB
    both = bench.host_fits_all_ranks(10e9, w, avail=30e9 if r == 0 else 15e9)
    roomy = bench.host_fits_all_ranks(10e9, w, avail=30e9)
    q.put((r, both, roomy))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_end_to_end_line_runs_on_all_ranks_or_none_gloo_world_size_2():
    """The end-to-end line pins host buffers on every rank and has barriers:
    one rank short of host memory makes every rank skip it, none hangs."""
    ctx = torch.multiprocessing.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_fits_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    assert res == [(0, False, True), (1, False, True)]


def _capture_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank), LOCAL_WORLD_SIZE=str(world))
    r, w, lr = bench.dist_setup(world)
    bench.init_pg(w)
    # rank 1's capture fails in the first round; both capture in the second
    first = bench.agreed_capture(None if r == 1 else 5.0, "no capture" if r == 1 else None, w)
    second = bench.agreed_capture(4.0 + r, None, w)
    q.put((r, first, second))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_graph_capture_is_agreed_on_by_all_ranks_gloo_world_size_2():
    """A rank whose CUDA-graph capture fails makes every rank report the
    graph figure as not captured (with the reason: its own, or 'on another
    rank'), and none waits in a collective the other skipped; when all
    capture, every rank gets the maximum."""
    ctx = torch.multiprocessing.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_capture_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    assert res == [(0, (None, "on another rank"), (5.0, None)),
                   (1, (None, "no capture"), (5.0, None))]


def test_max_over_ranks_gloo_world_size_2():
    ctx = torch.multiprocessing.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    assert res == [(0, 11.0), (1, 11.0)]
