"""kda_chunk_fwd_noalloc: the prefill entry point for callers that cannot
allocate device memory (no allocator of their own, or no cudaMalloc allowed on
their path).  Called through the C ABI, it must match the oracle and agree
with kda_chunk_fwd given a caller-allocated workspace, on two calls in a row
with different inputs (the scratch array keeps the first call's contents), and
a scan whose scratch exceeds the fixed array runs on the single-pass kernel.

This file is collected last so that a run stopping at the first failure has
already run every other test; it also passes when run alone.
"""
import ctypes

import numpy as np
import pytest
import torch

import kda_inputs
import oracle

pytestmark = pytest.mark.gpu

O_TOL = 2e-2
S_TOL = 1e-2
KDA_ERR_WORKSPACE = 5


@pytest.fixture(scope="module")
def kda():
    import linear_attention_serving_chunk_gb300 as m
    m.build()
    m.lib()
    return m


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _o_err(a, b):
    a = a.double().cpu().numpy()
    b = b.double().cpu().numpy()
    excess = np.abs(a - b) - 2.0 ** -8 * np.abs(b)
    return float(np.max(excess) / max(np.sqrt(np.mean(b * b)), 1e-30))


def _s_err(a, b):
    return float(torch.linalg.vector_norm(a.double() - b.double()) /
                 torch.linalg.vector_norm(b.double()))


def _noalloc(kda, x, n_seq, S_final, snaps, snap_offsets=None, expect=0):
    total, H, dk = x["k"].shape
    dv = x["v"].shape[2]
    o = torch.full((total, H, dv), float("nan"), dtype=torch.bfloat16, device="cuda")
    st = kda.lib().kda_chunk_fwd_noalloc(
        _ptr(x["q"]), _ptr(x["k"]), _ptr(x["v"]), _ptr(x["z"]), _ptr(x["beta"]), _ptr(x["A"]),
        -5.0, None, n_seq, total, H, dk, dv, 64, _ptr(x["S0"]), _ptr(o), _ptr(S_final),
        _ptr(snaps), _ptr(snap_offsets), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == expect, f"kda_chunk_fwd_noalloc returned {st}"
    return o


def test_noalloc_matches_the_workspace_entry_point_twice(kda):
    # two sequences of 65,536 tokens, 2 heads: the segment-parallel scan runs
    # (on the single-pass kernel: its three arrays, 12 MiB, fit the fixed
    # scratch) and is compared with the two-pass scan of kda_chunk_fwd.
    n_seq, H, T = 2, 2, 65536
    # the full workspace also holds the two-pass records; the scan's own
    # three arrays are what the fixed scratch must hold
    records = (T // 64) * n_seq * H * 73 * 1024
    need = kda.workspace_bytes(n_seq, n_seq * T, H, 128, 128) - records
    assert 0 < need <= (32 << 20)
    for seed in (31, 32):  # two calls in a row, different inputs
        x = kda_inputs.make_prefill(H, 128, 128, [T] * n_seq, seed=seed, device="cuda",
                                    S0_std=0.02)
        S_ref = torch.empty((n_seq, H, 128, 128), device="cuda")
        snaps_ref = torch.empty((n_seq * T // 64, H, 128, 128), device="cuda")
        o_ref = kda.chunk_fwd(x["q"], x["k"], x["v"], x["z"], x["beta"], x["A"], n_seq=n_seq,
                              S0=x["S0"], S_final=S_ref, snaps=snaps_ref)
        S_new = torch.full_like(S_ref, float("nan"))
        snaps_new = torch.full_like(snaps_ref, float("nan"))
        o_new = _noalloc(kda, x, n_seq, S_new, snaps_new)
        torch.cuda.synchronize()
        assert kda.device_status() == 0
        # outputs against the oracle (the two entry points run different
        # kernels here, so their bf16 outputs may round to neighbouring values)
        f64 = kda_inputs.to_f64
        ref = oracle.prefill(f64(x["q"]), f64(x["k"]), f64(x["v"]), f64(x["z"]), f64(x["beta"]),
                             f64(x["A"]), cu_seqlens=x["cu_seqlens"].cpu().numpy().astype(np.int64),
                             S0=f64(x["S0"]), snapshots=True)
        assert _o_err(o_new, torch.from_numpy(ref["o"])) <= O_TOL
        assert _o_err(o_ref, torch.from_numpy(ref["o"])) <= O_TOL
        # final states and snapshots of both entry points against the oracle
        for S_gpu, sn_gpu in ((S_new, snaps_new), (S_ref, snaps_ref)):
            assert _s_err(S_gpu.cpu(), torch.from_numpy(ref["S_final"])) <= S_TOL
            assert _s_err(sn_gpu.cpu(), torch.from_numpy(ref["snaps"])) <= S_TOL


def test_noalloc_single_pass_without_scratch(kda):
    """An equal-length 2^20-token call at 2 heads.  Without snap_offsets it
    would take the segment scan, whose 96 MiB of scratch exceed the fixed
    array: it runs on the single-pass kernel instead.  With snap_offsets
    kda_chunk_fwd never takes the scan, so neither does this entry point: the
    single pass again, no scratch.  The two calls agree exactly (the same
    kernel on the same inputs), and the second matches the oracle (every
    output, snapshot and the final state of both heads, the oracle running
    segment by segment on its own state)."""
    T, H = 1 << 20, 2
    x = kda_inputs.make_prefill(H, 128, 128, [T], seed=33, device="cuda", S0_std=0.02)
    S_a = torch.full((1, H, 128, 128), float("nan"), device="cuda")
    snaps_a = torch.full((T // 64, H, 128, 128), float("nan"), device="cuda")
    o_a = _noalloc(kda, x, 1, S_a, snaps_a)
    S_final = torch.full((1, H, 128, 128), float("nan"), device="cuda")
    snaps = torch.full((T // 64, H, 128, 128), float("nan"), device="cuda")
    offs = torch.tensor([0, T // 64], dtype=torch.int64, device="cuda")
    o = _noalloc(kda, x, 1, S_final, snaps, snap_offsets=offs)
    torch.cuda.synchronize()
    assert kda.device_status() == 0
    assert torch.equal(o_a, o) and torch.equal(S_a, S_final) and torch.equal(snaps_a, snaps)
    f64 = kda_inputs.to_f64
    seg = 1 << 17
    S = f64(x["S0"])
    worst_o = worst_sn = 0.0
    for a in range(0, T, seg):
        sl = slice(a, a + seg)
        ref = oracle.prefill(*(f64(x[n][sl]) for n in ("q", "k", "v", "z", "beta")), f64(x["A"]),
                             S0=S, snapshots=True)
        S = ref["S_final"]
        worst_o = max(worst_o, _o_err(o[sl], torch.from_numpy(ref["o"])))
        worst_sn = max(worst_sn, _s_err(snaps[a // 64:(a + seg) // 64].cpu(),
                                        torch.from_numpy(ref["snaps"])))
    assert worst_o <= O_TOL and worst_sn <= S_TOL
    assert _s_err(S_final.cpu(), torch.from_numpy(S)) <= S_TOL

