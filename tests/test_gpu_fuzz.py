"""Seeded random configurations of the public calls against the fp64 oracle:
every prefill path (two passes with all heads, two passes in head groups,
the single pass without a workspace) and kda_decode_tokens (token kernel and
chunked path), with random head shapes, lengths (empty, ragged, multi-chunk),
heads, and with or without S0, snapshots and final states.  The oracle sees
only the generated inputs; tolerances as in test_gpu_parity."""
import numpy as np
import pytest
import torch

import kda_inputs
import oracle

pytestmark = pytest.mark.gpu

O_TOL = 2e-2
S_TOL = 1e-2
BF16_ULP = 2.0 ** -8
f64 = kda_inputs.to_f64


@pytest.fixture(scope="module")
def kda():
    import linear_attention_serving_chunk_gb300 as m
    m.build()
    m.lib()
    return m


def o_err(o_gpu, o_ref):
    excess = np.abs(o_gpu - o_ref) - BF16_ULP * np.abs(o_ref)
    return float(np.max(excess) / max(np.sqrt(np.mean(o_ref ** 2)), 1e-30))


def s_err(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def draw(seed):
    r = np.random.default_rng(seed)
    dk = int(r.choice([64, 128]))
    dv = int(r.choice([64, 128]))
    H = int(r.integers(1, 4))
    n = int(r.integers(1, 6))
    lengths = [int(x) for x in r.choice([0, 1, 5, 63, 64, 65, 127, 128, 130, 200, 257, 400], n)]
    if sum(lengths) == 0:
        lengths[0] = 70
    return dict(dk=dk, dv=dv, H=H, lengths=lengths, S0=bool(r.integers(0, 2)),
                snaps=bool(r.integers(0, 2)), S_final=bool(r.integers(0, 2)),
                path=str(r.choice(["full", "groups", "single"])))


def ref_of(x, use_S0):
    cu = x["cu_seqlens"].cpu().numpy().astype(np.int64)
    return oracle.prefill(f64(x["q"]), f64(x["k"]), f64(x["v"]), f64(x["z"]), f64(x["beta"]),
                          f64(x["A"]), cu_seqlens=cu, S0=f64(x["S0"]) if use_S0 else None,
                          snapshots=True)


@pytest.mark.parametrize("seed", range(24))
def test_random_prefill_configuration(kda, seed):
    c = draw(9000 + seed)
    x = kda_inputs.make_prefill(c["H"], c["dk"], c["dv"], c["lengths"], seed=9100 + seed,
                                device="cuda", S0_std=0.02)
    n, total, H = len(c["lengths"]), sum(c["lengths"]), c["H"]
    full = kda.workspace_bytes(n, total, H, c["dk"], c["dv"])
    if c["path"] == "full":
        ws = torch.empty(max(full, 16), dtype=torch.uint8, device="cuda")
    elif c["path"] == "groups":  # the tables and one head's records: the heads one by one
        per_head = ((total + 63) // 64 + n) * 73 * 1024
        ws = torch.empty(max(full - (H - 1) * per_head, 16), dtype=torch.uint8, device="cuda")
    else:  # too small for any record: the single pass
        ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    offs = kda.snapshot_offsets(c["lengths"])
    rows = int(offs[-1])
    snaps = (torch.full((max(rows, 1), H, c["dk"], c["dv"]), float("nan"), device="cuda")
             if c["snaps"] else None)
    S_final = (torch.full((n, H, c["dk"], c["dv"]), float("nan"), device="cuda")
               if c["S_final"] else None)
    o = kda.chunk_fwd(x["q"], x["k"], x["v"], x["z"], x["beta"], x["A"],
                      cu_seqlens=x["cu_seqlens"], S0=x["S0"] if c["S0"] else None,
                      S_final=S_final, snaps=snaps, snap_offsets=offs if c["snaps"] else None,
                      workspace=ws)
    torch.cuda.synchronize()
    assert kda.device_status() == 0, c
    ref = ref_of(x, c["S0"])
    assert o_err(f64(o), ref["o"]) <= O_TOL, c
    if S_final is not None:
        assert s_err(f64(S_final), ref["S_final"]) <= S_TOL, c
    if snaps is not None and rows:
        assert s_err(f64(snaps[:rows]), ref["snaps"]) <= S_TOL, c


@pytest.mark.parametrize("seed", range(12))
def test_random_decode_tokens(kda, seed):
    """Random runs on random slots: short runs (the token kernel) and long
    ones (the chunked path), verify then commit."""
    r = np.random.default_rng(9500 + seed)
    dk, dv = int(r.choice([64, 128])), int(r.choice([64, 128]))
    H, n = int(r.integers(1, 4)), int(r.integers(2, 7))
    long = bool(seed % 2)
    lengths = [int(x) for x in r.integers(0, 90 if long else 12, n)]
    if sum(lengths) == 0:
        lengths[-1] = 3
    x = kda_inputs.make_prefill(H, dk, dv, lengths, seed=9600 + seed, device="cuda", S0_std=0.02)
    perm = torch.tensor(r.permutation(n + 2)[:n].astype(np.int32), device="cuda")
    pool = torch.zeros((n + 2, H, dk, dv), device="cuda")
    pool[perm.long()] = x["S0"]
    before = pool.clone()
    args = [x[nm] for nm in ("q", "k", "v", "z", "beta")] + [x["A"]]
    o_v = kda.decode_tokens(*args, pool, perm, x["cu_seqlens"], commit=False)
    torch.cuda.synchronize()
    assert torch.equal(pool, before)
    o_c = kda.decode_tokens(*args, pool, perm, x["cu_seqlens"], commit=True)
    torch.cuda.synchronize()
    assert kda.device_status() == 0
    assert torch.equal(o_v, o_c)
    ref = ref_of(x, True)
    assert o_err(f64(o_c), ref["o"]) <= O_TOL
    assert s_err(f64(pool[perm.long()]), ref["S_final"]) <= S_TOL
