"""GPU parity: the CUDA library (through the C ABI) against the fp64 oracle on
the same seeded inputs.

Tolerances: outputs |o - o_ref| <= 2e-2 * RMS(o_ref) + 2^-8 |o_ref| per
element (the stated 2e-2 RMS bound on the computation plus one bf16 ulp of
the exact value for the output cast: the outputs are heavy-tailed, max|o| is
about 12 RMS, so rounding the exact result to bf16 alone reaches 2.7e-2 RMS);
states (final and snapshots) relative Frobenius error <= 1e-2; decode state
trajectories relative Frobenius error <= 1e-4 per state.  The oracle never sees a value
produced by the CUDA path: its inputs are the generated inputs, copied to the
host, and it carries its own state between segments.
"""
import numpy as np
import pytest
import torch

import kda_inputs
import oracle
from oracle import preops

pytestmark = pytest.mark.gpu

O_TOL = 2e-2
S_TOL = 1e-2
DECODE_TOL = 1e-4

f64 = kda_inputs.to_f64


@pytest.fixture(scope="module")
def kda():
    import linear_attention_serving_chunk_gb300 as m
    m.build()
    m.lib()
    return m


BF16_ULP = 2.0 ** -8


def o_err(o_gpu, o_ref):
    """max over elements of (|o - o_ref| - 2^-8 |o_ref|) / RMS(o_ref): the
    output error beyond one bf16 ulp of the exact value, in units of RMS."""
    excess = np.abs(o_gpu - o_ref) - BF16_ULP * np.abs(o_ref)
    return float(np.max(excess) / max(np.sqrt(np.mean(o_ref ** 2)), 1e-30))


def s_err(S_gpu, S_ref):
    """Relative Frobenius error."""
    return float(np.linalg.norm(S_gpu - S_ref) / max(np.linalg.norm(S_ref), 1e-30))


def run_prefill(kda, x, snapshots=True, S0=True, pre=0):
    n_seq = len(x["lengths"])
    total, H, dk = x["k"].shape
    dv = x["v"].shape[2]
    dev = x["k"].device
    offs = kda.snapshot_offsets(x["lengths"], device=dev)
    snaps = (torch.full((max(int(offs[-1]), 1), H, dk, dv), float("nan"), device=dev)
             if snapshots else None)
    S_final = torch.full((n_seq, H, dk, dv), float("nan"), device=dev)
    o = torch.full((total, H, dv), float("nan"), dtype=torch.bfloat16, device=dev)
    kda.chunk_fwd(x["q"], x["k"], x["v"], x["z"], x["beta"], x["A"], cu_seqlens=x["cu_seqlens"],
                  S0=x["S0"] if S0 else None, o=o, S_final=S_final, snaps=snaps,
                  snap_offsets=offs if snapshots else None, pre=pre)
    torch.cuda.synchronize()
    assert kda.device_status() == 0
    return o, S_final, snaps, offs


def oracle_subset(x, seqs, heads, t_limit=None, snapshots=True, pre=0):
    """Oracle on sequences ``seqs`` and heads ``heads`` (optionally only the
    first t_limit tokens of each sequence).  Inputs are gathered on the host;
    ``pre`` applies the oracle's own input pre-ops to them first."""
    cu = x["cu_seqlens"].cpu().numpy().astype(np.int64)
    hs = torch.tensor(heads, device=x["k"].device)
    parts = {n: [] for n in ("q", "k", "v", "z", "beta")}
    lens = []
    for s in seqs:
        a = int(cu[s])
        L = int(cu[s + 1] - cu[s]) if t_limit is None else min(t_limit, int(cu[s + 1] - cu[s]))
        lens.append(L)
        for n in parts:
            parts[n].append(f64(x[n][a:a + L].index_select(1, hs)))
    cat = {n: np.concatenate(parts[n], axis=0) for n in parts}
    if pre:
        cat["q"], cat["k"], cat["beta"] = preops.apply(cat["q"], cat["k"], cat["beta"],
                                                       bool(pre & 1), bool(pre & 2))
    S0 = None
    if x["S0"] is not None:
        S0 = f64(x["S0"][torch.tensor(seqs, device=x["k"].device)].index_select(1, hs))
    ref = oracle.prefill(cat["q"], cat["k"], cat["v"], cat["z"], cat["beta"],
                         f64(x["A"])[heads], cu_seqlens=np.concatenate([[0], np.cumsum(lens)]),
                         S0=S0, snapshots=snapshots)
    ref["lens"] = lens
    return ref


def gather_gpu(x, o, S_final, snaps, offs, seqs, heads, t_limit=None):
    cu = x["cu_seqlens"].cpu().numpy().astype(np.int64)
    offs_h = offs.cpu().numpy()
    hs = torch.tensor(heads, device=o.device)
    oo, ss, sn = [], [], []
    for s in seqs:
        a = int(cu[s])
        L = int(cu[s + 1] - cu[s]) if t_limit is None else min(t_limit, int(cu[s + 1] - cu[s]))
        oo.append(f64(o[a:a + L].index_select(1, hs)))
        ss.append(f64(S_final[s].index_select(0, hs)))
        if snaps is not None:
            nsn = L // 64
            sn.append(f64(snaps[int(offs_h[s]):int(offs_h[s]) + nsn].index_select(1, hs)))
    return (np.concatenate(oo), np.stack(ss),
            np.concatenate(sn) if sn else None)


def check_all(x, kda, seqs=None, heads=None, t_limit=None, pre=0):
    o, S_final, snaps, offs = run_prefill(kda, x, pre=pre)
    n_seq = len(x["lengths"])
    H = x["k"].shape[1]
    seqs = list(range(n_seq)) if seqs is None else seqs
    heads = list(range(H)) if heads is None else heads
    ref = oracle_subset(x, seqs, heads, t_limit, pre=pre)
    go, gs, gsn = gather_gpu(x, o, S_final, snaps, offs, seqs, heads, t_limit)
    e_o = o_err(go, ref["o"])
    assert np.all(np.isfinite(go)), "non-finite outputs"
    assert e_o <= O_TOL, f"output error {e_o:.3e}"
    if ref["snaps"] is not None and ref["snaps"].shape[0]:
        e_sn = s_err(gsn, ref["snaps"])
        assert e_sn <= S_TOL, f"snapshot error {e_sn:.3e}"
    if t_limit is None:
        e_s = s_err(gs, ref["S_final"])
        assert e_s <= S_TOL, f"final state error {e_s:.3e}"
    return o, S_final, snaps, offs, ref


# --- the workloads ---------------------------------------------------------------------------

def test_tiny_full(kda):
    x = kda_inputs.make_workload_prefill("tiny", device="cuda")
    check_all(x, kda)


def test_mid_full(kda):
    """B=4, H=16, T=8192, dk=dv=128: every output, final state and snapshot."""
    x = kda_inputs.make_workload_prefill("mid", device="cuda")
    check_all(x, kda)


def test_varlen_64_sequences(kda):
    """64 packed sequences, lengths U[512, 32768], H=32, S0 ~ N(0, 0.02^2):
    the GPU runs everything; all 64 sequences are checked on 4 seeded heads."""
    x = kda_inputs.make_workload_prefill("varlen", device="cuda")
    heads = sorted(np.random.default_rng(2024).choice(32, size=4, replace=False).tolist())
    check_all(x, kda, heads=heads)


def test_long_context(kda):
    """T = 1,048,576, H = 16, called as the benchmark calls it (one sequence,
    no cu_seqlens, no snap_offsets): the library takes the segment-parallel
    scan on the two-pass kernels.  Heads 0 and 1 are checked over the whole
    length - every output, every chunk snapshot and the final state - against
    the oracle run segment by segment on its own carried state."""
    x = kda_inputs.make_workload_prefill("long", device="cuda")
    T, H = x["k"].shape[0], x["k"].shape[1]
    need = kda.workspace_bytes(1, T, H, 128, 128)
    assert need > (T // 64) * H * 73 * 1024  # the scan arrays plus every record
    S_final = torch.full((1, H, 128, 128), float("nan"), device="cuda")
    snaps = torch.full((T // 64, H, 128, 128), float("nan"), device="cuda")
    o = kda.chunk_fwd(x["q"], x["k"], x["v"], x["z"], x["beta"], x["A"], n_seq=1,
                      S_final=S_final, snaps=snaps)
    torch.cuda.synchronize()
    assert kda.device_status() == 0
    heads = [0, 1]
    hs = torch.tensor(heads, device="cuda")
    seg = 1 << 17
    S = None
    worst_o, worst_sn = 0.0, 0.0
    for a in range(0, T, seg):
        sl = slice(a, a + seg)
        ref = oracle.prefill(*(f64(x[n][sl].index_select(1, hs)) for n in ("q", "k", "v", "z",
                                                                            "beta")),
                             f64(x["A"])[heads], S0=S, snapshots=True)
        S = ref["S_final"]
        worst_o = max(worst_o, o_err(f64(o[sl].index_select(1, hs)), ref["o"]))
        g_sn = f64(snaps[a // 64:(a + seg) // 64].index_select(1, hs))
        worst_sn = max(worst_sn, s_err(g_sn, ref["snaps"]))
    assert worst_o <= O_TOL, f"output error {worst_o:.3e}"
    assert worst_sn <= S_TOL, f"snapshot error {worst_sn:.3e}"
    e_s = s_err(f64(S_final[0].index_select(0, hs)), S[0])
    assert e_s <= S_TOL, f"final state error {e_s:.3e}"


@pytest.mark.parametrize("S0_std", [None, 0.02])
def test_segment_scan_long_sequences(kda, S0_std):
    """Few chains and long sequences take the segment-parallel scan (2 x 65,536
    tokens, H = 2: 16 segments of 4096 tokens per chain); every output, the
    final states and all snapshots are checked against the oracle."""
    x = kda_inputs.make_prefill(2, 128, 128, [65536, 65536], seed=21, device="cuda",
                                S0_std=S0_std)
    assert kda.workspace_bytes(2, 2 * 65536, 2, 128, 128) > 0  # the scan path is taken
    n_seq, H = 2, 2
    S_final = torch.full((n_seq, H, 128, 128), float("nan"), device="cuda")
    snaps = torch.full((2 * 1024, H, 128, 128), float("nan"), device="cuda")
    o = kda.chunk_fwd(x["q"], x["k"], x["v"], x["z"], x["beta"], x["A"], n_seq=n_seq,
                      S0=x["S0"], S_final=S_final, snaps=snaps)
    torch.cuda.synchronize()
    assert kda.device_status() == 0
    ref = oracle_subset(x, [0, 1], [0, 1])
    assert o_err(f64(o), ref["o"]) <= O_TOL
    assert s_err(f64(S_final), ref["S_final"]) <= S_TOL
    assert s_err(f64(snaps), ref["snaps"]) <= S_TOL


@pytest.mark.parametrize("d", [64, 128])
def test_decode_tokens_multi_token(kda, d):
    """Multi-token decode / speculative verify on resident states: runs of 1 to
    70 tokens per sequence from state slots; commit=False leaves the pool
    untouched, commit=True stores the final states; both match the oracle."""
    lengths = [1, 2, 5, 16, 17, 40, 64, 70]
    n, H = len(lengths), 2
    x = kda_inputs.make_prefill(H, d, d, lengths, seed=23, device="cuda", S0_std=0.02)
    perm = torch.tensor([5, 2, 7, 0, 3, 6, 1, 4], dtype=torch.int32, device="cuda")
    pool = torch.zeros((8, H, d, d), device="cuda")
    pool[perm.long()] = x["S0"]
    before = pool.clone()
    args = [x[nm] for nm in ("q", "k", "v", "z", "beta")] + [x["A"]]
    o_v = kda.decode_tokens(*args, pool, perm, x["cu_seqlens"], commit=False)
    torch.cuda.synchronize()
    assert torch.equal(pool, before)
    o_c = kda.decode_tokens(*args, pool, perm, x["cu_seqlens"], commit=True)
    torch.cuda.synchronize()
    assert torch.equal(o_v, o_c)
    ref = oracle_subset(x, list(range(n)), [0, 1], snapshots=False)
    assert o_err(f64(o_c), ref["o"]) <= O_TOL
    assert s_err(f64(pool[perm.long()]), ref["S_final"]) <= S_TOL


@pytest.mark.parametrize("dk,dv", [(128, 128), (64, 64), (128, 64), (64, 128)])
def test_decode_tokens_short_runs(kda, dk, dv):
    """Short runs (at most 16 tokens per sequence on average) take the
    token-by-token kernel on the state held on chip: empty runs, single
    tokens, a run of 16 tokens (two 8-token blocks) and one of 50 tokens
    (seven blocks, the later ones loaded directly); verify (commit=False)
    leaves the pool untouched, commit=True stores the final states; both
    against the oracle."""
    lengths = [1, 0, 3, 16, 2, 50, 1, 5, 0, 7]
    n, H = len(lengths), 2
    assert sum(lengths) <= 16 * n
    x = kda_inputs.make_prefill(H, dk, dv, lengths, seed=29, device="cuda", S0_std=0.02)
    perm = torch.tensor([3, 9, 0, 7, 5, 1, 8, 2, 6, 4], dtype=torch.int32, device="cuda")
    pool = torch.zeros((n, H, dk, dv), device="cuda")
    pool[perm.long()] = x["S0"]
    before = pool.clone()
    args = [x[nm] for nm in ("q", "k", "v", "z", "beta")] + [x["A"]]
    o_v = kda.decode_tokens(*args, pool, perm, x["cu_seqlens"], commit=False)
    torch.cuda.synchronize()
    assert kda.device_status() == 0
    assert torch.equal(pool, before)
    o_c = kda.decode_tokens(*args, pool, perm, x["cu_seqlens"], commit=True)
    torch.cuda.synchronize()
    assert kda.device_status() == 0
    assert torch.equal(o_v, o_c)
    ref = oracle_subset(x, list(range(n)), [0, 1], snapshots=False)
    assert o_err(f64(o_c), ref["o"]) <= O_TOL
    assert s_err(f64(pool[perm.long()]), ref["S_final"]) <= S_TOL
    # empty runs keep their states exactly
    for b in (1, 8):
        assert torch.equal(pool[int(perm[b])], before[int(perm[b])])


@pytest.mark.parametrize("dk,dv", [(128, 128), (64, 64), (128, 64), (64, 128)])
def test_decode_tokens_many_rows_per_cta(kda, dk, dv):
    """More (sequence, head) rows than the token kernel's persistent CTAs (two
    per SM): each CTA takes several rows in turn, the next row's state and
    tokens prefetched while the current row's tokens run.  Runs of 0 to 20
    tokens (a run's later 8-token blocks loaded directly), permuted slots;
    verify and commit against the oracle, empty runs untouched."""
    rng = np.random.default_rng(37)
    n, H = 200, 4  # 800 rows
    lengths = rng.choice([0, 1, 2, 4, 7, 8, 9, 12, 16, 20], size=n).tolist()
    assert sum(lengths) <= 16 * n
    x = kda_inputs.make_prefill(H, dk, dv, lengths, seed=41, device="cuda", S0_std=0.02)
    perm = torch.from_numpy(rng.permutation(n).astype(np.int32)).to("cuda")
    pool = torch.zeros((n, H, dk, dv), device="cuda")
    pool[perm.long()] = x["S0"]
    before = pool.clone()
    args = [x[nm] for nm in ("q", "k", "v", "z", "beta")] + [x["A"]]
    o_v = kda.decode_tokens(*args, pool, perm, x["cu_seqlens"], commit=False)
    torch.cuda.synchronize()
    assert kda.device_status() == 0
    assert torch.equal(pool, before)
    o_c = kda.decode_tokens(*args, pool, perm, x["cu_seqlens"], commit=True)
    torch.cuda.synchronize()
    assert kda.device_status() == 0
    assert torch.equal(o_v, o_c)
    ref = oracle_subset(x, list(range(n)), list(range(H)), snapshots=False)
    assert o_err(f64(o_c), ref["o"]) <= O_TOL
    assert s_err(f64(pool[perm.long()]), ref["S_final"]) <= S_TOL
    for b in range(n):
        if lengths[b] == 0:
            assert torch.equal(pool[int(perm[b])], before[int(perm[b])])


def test_decode_tokens_bad_slots_among_many_rows(kda):
    """Rejected rows (slots out of range) between valid ones of the same
    persistent CTA: they are skipped and reported, the prefetching of the rows
    around them is unaffected, and pool slots nobody names stay as they were."""
    rng = np.random.default_rng(43)
    n, H, d = 160, 4, 128  # 640 rows
    lengths = rng.integers(1, 13, size=n).tolist()
    x = kda_inputs.make_prefill(H, d, d, lengths, seed=47, device="cuda", S0_std=0.02)
    perm = rng.permutation(n).astype(np.int32)
    bad = [5, 77, 151]
    slots_np = perm.copy()
    slots_np[bad] = [-1, n, 10 ** 6]
    slots = torch.from_numpy(slots_np).to("cuda")
    pool = torch.zeros((n, H, d, d), device="cuda")
    pool[torch.from_numpy(perm).long().to("cuda")] = x["S0"]
    before = pool.clone()
    args = [x[nm] for nm in ("q", "k", "v", "z", "beta")] + [x["A"]]
    kda.decode_tokens(*args, pool, slots, x["cu_seqlens"], commit=True)
    torch.cuda.synchronize()
    assert kda.device_status() == kda.KDA_ERR_SHAPE
    good = [b for b in range(n) if b not in bad]
    ref = oracle_subset(x, good, list(range(H)), snapshots=False)
    got = f64(pool[torch.from_numpy(perm[good]).long().to("cuda")])
    assert s_err(got, ref["S_final"]) <= S_TOL
    for b in bad:  # the slots the rejected sequences would have used are untouched
        assert torch.equal(pool[int(perm[b])], before[int(perm[b])])


def test_decode_tokens_short_runs_match_single_steps(kda):
    """The token-by-token kernel does each token's step as kda_decode_step
    does it: the same pool, run by run or token by token (the k.q sums are
    added in another order, so equal to float rounding)."""
    lengths = [4, 4, 4, 4]
    n, H, d = 4, 2, 128
    x = kda_inputs.make_prefill(H, d, d, lengths, seed=31, device="cuda", S0_std=0.02)
    pool_a = x["S0"].clone()
    pool_b = x["S0"].clone()
    slots = torch.arange(n, dtype=torch.int32, device="cuda")
    o_a = kda.decode_tokens(x["q"], x["k"], x["v"], x["z"], x["beta"], x["A"], pool_a, slots,
                            x["cu_seqlens"], commit=True)
    o_b = torch.empty_like(o_a)
    for t in range(4):
        rows = torch.arange(n, device="cuda") * 4 + t
        ob = kda.decode_step(x["q"][rows], x["k"][rows], x["v"][rows], x["z"][rows],
                             x["beta"][rows], x["A"], pool_b)
        o_b[rows] = ob
    torch.cuda.synchronize()
    assert s_err(f64(pool_a), f64(pool_b)) <= 1e-6
    assert np.max(np.abs(f64(o_a) - f64(o_b))) <= 2.0 ** -7 * max(np.max(np.abs(f64(o_b))), 1e-30)


def test_decode_1000_steps(kda):
    """512 x 32 resident states, 1000 chained steps with fresh inputs: all
    states are checked after steps 1 and 10, 256 seeded (sequence, head)
    pairs after steps 1, 10, 100 and 1000, 16 of them after every step."""
    w = kda_inputs.WORKLOADS["decode"]
    B, H, dk, dv = w["batch"], w["H"], w["dk"], w["dv"]
    pool, A = kda_inputs.make_decode_state(B, H, dk, dv, w["seed"], device="cuda",
                                           std=w["state_std"])
    rng = np.random.default_rng(77)
    pairs = rng.choice(B * H, size=256, replace=False)
    every = pairs[:16]
    pb, ph = torch.tensor(pairs // H, device="cuda"), torch.tensor(pairs % H, device="cuda")
    eb, eh = torch.tensor(every // H, device="cuda"), torch.tensor(every % H, device="cuda")
    Af = f64(A)
    full = np.ascontiguousarray(f64(pool))
    sub = np.ascontiguousarray(f64(pool[pb, ph]))[:, None]  # [256, 1, dk, dv]
    worst_every, worst_o = 0.0, 0.0
    for step in range(w["steps"]):
        t = kda_inputs.make_decode_token(B, H, dk, dv, w["seed"], step, device="cuda")
        o = kda.decode_step(t["q"], t["k"], t["v"], t["z"], t["beta"], A, pool)
        # oracle on the 256-pair subset (one sequence per pair, its own head's A)
        ins = {n: f64(t[n][pb, ph])[:, None] for n in ("q", "k", "v", "z", "beta")}
        o_ref = np.empty((256, dv))
        for hh in np.unique(pairs % H):
            m = (pairs % H) == hh
            st = np.ascontiguousarray(sub[m])
            o_ref[m] = oracle.decode_step(ins["q"][m], ins["k"][m], ins["v"][m], ins["z"][m],
                                          ins["beta"][m], Af[hh:hh + 1], st)[:, 0]
            sub[m] = st
        worst_o = max(worst_o, o_err(f64(o[pb, ph]), o_ref))
        if step < 10:
            oracle.decode_step(f64(t["q"]), f64(t["k"]), f64(t["v"]), f64(t["z"]),
                               f64(t["beta"]), Af, full)
        n = step + 1
        g_every = f64(pool[eb, eh])
        for a, i in enumerate(range(16)):
            worst_every = max(worst_every, s_err(g_every[a], sub[i, 0]))
        if n in (1, 10, 100, 1000):
            g_sub = f64(pool[pb, ph])
            e = max(s_err(g_sub[i], sub[i, 0]) for i in range(256))
            assert e <= DECODE_TOL, f"step {n}: subset state error {e:.3e}"
        if n in (1, 10):
            g_full = f64(pool).reshape(B * H, dk, dv)
            e = max(s_err(g_full[i], full.reshape(B * H, dk, dv)[i]) for i in range(B * H))
            assert e <= DECODE_TOL, f"step {n}: state error {e:.3e}"
    assert worst_every <= DECODE_TOL, f"per-step trajectory error {worst_every:.3e}"
    assert worst_o <= O_TOL, f"decode output error {worst_o:.3e}"


# --- edge cases --------------------------------------------------------------------------------

@pytest.mark.parametrize("dk,dv", [(64, 64), (128, 128), (128, 64), (64, 128)])
def test_ragged_lengths(kda, dk, dv):
    """Empty, single-token, sub-chunk, exact-chunk and ragged sequences."""
    lengths = [0, 1, 63, 64, 65, 127, 128, 200, 331]
    x = kda_inputs.make_prefill(3, dk, dv, lengths, seed=11, device="cuda", S0_std=0.02)
    o, S_final, snaps, offs, ref = check_all(x, kda)
    # the empty sequence keeps its initial state exactly
    assert torch.equal(S_final[0], x["S0"][0])


@pytest.mark.parametrize("n", [512, 600])
def test_many_sequences_and_the_state_pass_order(kda, n):
    """The chunk table ranks up to 512 sequences longest first for the state
    pass (ties in batch order) and leaves more in batch order.  Lengths with
    many ties, empty and exact-chunk sequences: every sequence must be taken
    exactly once (a missed one leaves NaN outputs, a doubled one races)."""
    rng = np.random.default_rng(77 + n)
    lengths = rng.choice([0, 1, 63, 64, 65, 130, 257, 700], size=n).tolist()
    x = kda_inputs.make_prefill(2, 128, 128, lengths, seed=12 + n, device="cuda", S0_std=0.02)
    check_all(x, kda)


def test_zero_initial_state_and_no_optional_outputs(kda):
    x = kda_inputs.make_prefill(2, 64, 64, [150, 77], seed=12, device="cuda")
    o = kda.chunk_fwd(x["q"], x["k"], x["v"], x["z"], x["beta"], x["A"],
                      cu_seqlens=x["cu_seqlens"])
    ref = oracle_subset(x, [0, 1], [0, 1], snapshots=False)
    assert o_err(f64(o), ref["o"]) <= O_TOL


def test_equal_length_batch_without_cu_seqlens(kda):
    x = kda_inputs.make_prefill(2, 128, 128, [192, 192, 192], seed=13, device="cuda",
                                S0_std=0.02)
    n_seq = 3
    S_final = torch.empty((n_seq, 2, 128, 128), device="cuda")
    snaps = torch.empty((9, 2, 128, 128), device="cuda")
    o = kda.chunk_fwd(x["q"], x["k"], x["v"], x["z"], x["beta"], x["A"], n_seq=n_seq, S0=x["S0"],
                      S_final=S_final, snaps=snaps)
    ref = oracle_subset(x, [0, 1, 2], [0, 1])
    assert o_err(f64(o), ref["o"]) <= O_TOL
    assert s_err(f64(S_final), ref["S_final"]) <= S_TOL
    assert s_err(f64(snaps), ref["snaps"]) <= S_TOL


@pytest.mark.parametrize("zval", [float("inf"), float("-inf"), 40.0])
def test_extreme_gates(kda, zval):
    """z = +inf gives g = -5 in every channel (the strongest decay the bound
    allows: a rescaling factor of e^80 per 16-token sub-tile); the output must
    stay finite and match.  z = -inf gives no decay at all."""
    x = kda_inputs.make_prefill(2, 128, 128, [256, 100], seed=14, device="cuda", S0_std=0.02)
    x["z"].fill_(zval)
    o, S_final, snaps, offs, ref = check_all(x, kda)
    assert torch.isfinite(o.float()).all() and torch.isfinite(S_final).all()


def test_prefix_cache_roundtrip(kda):
    """Prefill a sequence, restore the snapshot after 3 chunks into a state
    slot, prefill the suffix from that slot and decode one token from another
    restored slot: both match the oracle run on the whole sequence."""
    L, H, d = 300, 2, 128
    x = kda_inputs.make_prefill(H, d, d, [L], seed=15, device="cuda", S0_std=0.02)
    o, S_final, snaps, offs = run_prefill(kda, x)
    pool = torch.zeros((4, H, d, d), device="cuda")
    kda.state_snapshot(snaps, torch.tensor([2, 1], dtype=torch.int64, device="cuda"), pool,
                       torch.tensor([3, 0], dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert torch.equal(pool[3], snaps[2]) and torch.equal(pool[0], snaps[1])
    cut = 192
    o_suf = kda.chunk_fwd(*(x[n][cut:].contiguous() for n in ("q", "k", "v", "z", "beta")), x["A"],
                          S0=pool[3:4].contiguous())
    ref = oracle_subset(x, [0], [0, 1])
    assert o_err(f64(o_suf), ref["o"][cut:]) <= O_TOL
    # decode the token at position 128 from the snapshot after 2 chunks (slot 0)
    t = {n: x[n][128:129].contiguous() for n in ("q", "k", "v", "z", "beta")}
    od = kda.decode_step(t["q"], t["k"], t["v"], t["z"], t["beta"], x["A"], pool,
                         slots=torch.tensor([0], dtype=torch.int32, device="cuda"))
    assert o_err(f64(od)[0], ref["o"][128]) <= O_TOL


def test_decode_slots_and_prefill_agreement(kda):
    """Decode through a slot permutation equals decode in place; n decode
    steps reproduce the oracle's n-token prefill."""
    n, H, d, steps = 6, 2, 64, 20
    x = kda_inputs.make_prefill(H, d, d, [steps] * n, seed=16, device="cuda", S0_std=0.02)
    perm = torch.tensor([3, 0, 5, 1, 4, 2], dtype=torch.int32, device="cuda")
    pool_a = x["S0"].clone()
    pool_b = torch.empty_like(pool_a)
    pool_b[perm.long()] = x["S0"]
    for t in range(steps):
        rows = torch.arange(n, device="cuda") * steps + t
        tok = {nm: x[nm][rows].contiguous() for nm in ("q", "k", "v", "z", "beta")}
        oa = kda.decode_step(tok["q"], tok["k"], tok["v"], tok["z"], tok["beta"], x["A"], pool_a)
        ob = kda.decode_step(tok["q"], tok["k"], tok["v"], tok["z"], tok["beta"], x["A"], pool_b,
                             slots=perm)
        assert torch.equal(oa, ob)
    assert torch.equal(pool_b[perm.long()], pool_a)
    ref = oracle_subset(x, list(range(n)), [0, 1], snapshots=False)
    assert s_err(f64(pool_a), ref["S_final"]) <= DECODE_TOL


def test_runs_on_a_side_stream(kda):
    x = kda_inputs.make_prefill(2, 64, 64, [130], seed=17, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        o = kda.chunk_fwd(x["q"], x["k"], x["v"], x["z"], x["beta"], x["A"])
    s.synchronize()
    ref = oracle_subset(x, [0], [0, 1], snapshots=False)
    assert o_err(f64(o), ref["o"]) <= O_TOL


# --- fused input pre-ops (L2 norm of q, k rows; sigmoid of beta) -------------------------

@pytest.mark.parametrize("d,pre", [(128, 3), (64, 3), (128, 1), (128, 2)])
def test_preops_prefill(kda, d, pre):
    """Raw projections (q, k rows of norm 0.25..4 x sqrt(d), beta logits): the
    kernels' fused pre-ops against the oracle's pre-ops followed by the
    oracle, ragged varlen batch with S0 (both head sizes on the tensor-core
    kernels)."""
    x = kda_inputs.make_raw_prefill(3, d, d, [200, 64, 1, 130], seed=41 + pre, device="cuda",
                                    S0_std=0.02)
    if not pre & 1:  # norm pre-op off: hand in unit rows, as the plain entry point expects
        for nm in ("q", "k"):
            t = x[nm].float()
            x[nm] = (t / torch.linalg.vector_norm(t, dim=-1, keepdim=True)).to(torch.bfloat16)
    if not pre & 2:
        x["beta"] = torch.sigmoid(x["beta"].float()).to(torch.bfloat16)
    check_all(x, kda, pre=pre)


def test_preops_segment_scan(kda):
    """The scan's three prefill passes all apply the pre-ops (2 x 16,384
    tokens, H = 2: 4 segments of 4096 per chain)."""
    x = kda_inputs.make_raw_prefill(2, 128, 128, [16384, 16384], seed=45, device="cuda",
                                    S0_std=0.02)
    assert kda.workspace_bytes(2, 2 * 16384, 2, 128, 128) > 0
    S_final = torch.full((2, 2, 128, 128), float("nan"), device="cuda")
    o = kda.chunk_fwd(x["q"], x["k"], x["v"], x["z"], x["beta"], x["A"], n_seq=2, S0=x["S0"],
                      S_final=S_final, pre=kda.PRE_L2NORM_QK | kda.PRE_SIGMOID_BETA)
    torch.cuda.synchronize()
    assert kda.device_status() == 0
    ref = oracle_subset(x, [0, 1], [0, 1], snapshots=False, pre=3)
    assert o_err(f64(o), ref["o"]) <= O_TOL
    assert s_err(f64(S_final), ref["S_final"]) <= S_TOL


@pytest.mark.parametrize("d", [64, 128])
def test_preops_decode(kda, d):
    """kda_decode_step_ex and kda_decode_tokens with the pre-ops: 20 chained
    single-token steps, then a 2..33-token run per sequence."""
    n, H = 6, 2
    pool = kda_inputs.make_prefill(H, d, d, [1] * n, seed=46, device="cuda",
                                   S0_std=0.02)["S0"].contiguous()
    state = np.ascontiguousarray(f64(pool))
    A = None
    for step in range(20):
        t = kda_inputs.make_raw_prefill(H, d, d, [1] * n, seed=1000 + step, device="cuda")
        A = t["A"] if A is None else A
        o = kda.decode_step(t["q"], t["k"], t["v"], t["z"], t["beta"], A, pool, pre=3)
        qf, kf, bf = preops.apply(f64(t["q"]), f64(t["k"]), f64(t["beta"]), True, True)
        o_ref = oracle.decode_step(qf, kf, f64(t["v"]), f64(t["z"]), bf, f64(A), state)
        assert o_err(f64(o), o_ref) <= O_TOL
    torch.cuda.synchronize()
    assert s_err(f64(pool), state) <= DECODE_TOL
    lengths = [2, 3, 9, 16, 33, 5]
    x = kda_inputs.make_raw_prefill(H, d, d, lengths, seed=47, device="cuda")
    x["A"] = A
    x["S0"] = pool.clone()
    slots = torch.arange(n, dtype=torch.int32, device="cuda")
    o = kda.decode_tokens(x["q"], x["k"], x["v"], x["z"], x["beta"], A, pool, slots,
                          x["cu_seqlens"], commit=True, pre=3)
    torch.cuda.synchronize()
    ref = oracle_subset(x, list(range(n)), [0, 1], snapshots=False, pre=3)
    assert o_err(f64(o), ref["o"]) <= O_TOL
    assert s_err(f64(pool), ref["S_final"]) <= S_TOL


def test_split_phase_calls_match_one_call(kda):
    """chunk_fwd with PASS_PREPARE then PASS_STATE (the bench's step) gives
    exactly the one-call result, and a state pass can be repeated from the
    same records; both match the oracle."""
    x = kda_inputs.make_prefill(4, 128, 128, [300, 64, 129, 1000], seed=51, device="cuda",
                                S0_std=0.02)
    n = len(x["lengths"])
    total = x["k"].shape[0]
    ws = torch.empty(kda.workspace_bytes(n, total, 4, 128, 128), dtype=torch.uint8,
                     device="cuda")
    offs = kda.snapshot_offsets(x["lengths"])
    args = [x[nm] for nm in ("q", "k", "v", "z", "beta", "A")]
    outs = []
    for passes in ((0,), (kda.PASS_PREPARE, kda.PASS_STATE, kda.PASS_STATE)):
        S_final = torch.full((n, 4, 128, 128), float("nan"), device="cuda")
        snaps = torch.full((int(offs[-1]), 4, 128, 128), float("nan"), device="cuda")
        o = torch.full((total, 4, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
        for ps in passes:
            kda.chunk_fwd(*args, cu_seqlens=x["cu_seqlens"], S0=x["S0"], o=o, S_final=S_final,
                          snaps=snaps, snap_offsets=offs, workspace=ws, pre=ps)
        torch.cuda.synchronize()
        assert kda.device_status() == 0
        outs.append((o, S_final, snaps))
    for a, b in zip(*outs):
        assert torch.equal(a, b)
    ref = oracle_subset(x, list(range(n)), [0, 1, 2, 3])
    assert o_err(f64(outs[1][0]), ref["o"]) <= O_TOL
    assert s_err(f64(outs[1][1]), ref["S_final"]) <= S_TOL
    assert s_err(f64(outs[1][2]), ref["snaps"]) <= S_TOL


def test_single_pass_kernel_ragged_batch(kda):
    """With a workspace too small for any records the prefill runs the
    single-pass tensor-core kernel: ragged varlen batch with S0, every output,
    final state and snapshot against the oracle."""
    lengths = [0, 1, 63, 64, 65, 127, 128, 200, 331]
    x = kda_inputs.make_prefill(3, 128, 128, lengths, seed=52, device="cuda", S0_std=0.02)
    total = x["k"].shape[0]
    n = len(lengths)
    offs = kda.snapshot_offsets(lengths)
    S_final = torch.full((n, 3, 128, 128), float("nan"), device="cuda")
    snaps = torch.full((int(offs[-1]), 3, 128, 128), float("nan"), device="cuda")
    o = torch.full((total, 3, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    tiny = torch.empty(16, dtype=torch.uint8, device="cuda")
    kda.chunk_fwd(x["q"], x["k"], x["v"], x["z"], x["beta"], x["A"], cu_seqlens=x["cu_seqlens"],
                  S0=x["S0"], o=o, S_final=S_final, snaps=snaps, snap_offsets=offs,
                  workspace=tiny)
    torch.cuda.synchronize()
    assert kda.device_status() == 0
    ref = oracle_subset(x, list(range(n)), [0, 1, 2])
    assert np.all(np.isfinite(f64(o)))
    assert o_err(f64(o), ref["o"]) <= O_TOL
    assert s_err(f64(S_final), ref["S_final"]) <= S_TOL
    assert s_err(f64(snaps), ref["snaps"]) <= S_TOL
    assert torch.equal(S_final[0], x["S0"][0])


@pytest.mark.parametrize("d", [64, 128])
def test_all_empty_batch(kda, d):
    """A batch of empty sequences: nothing to write in o, every final state is
    its initial state."""
    x = kda_inputs.make_prefill(2, d, d, [0, 0, 0], seed=53, device="cuda", S0_std=0.02)
    S_final = torch.full((3, 2, d, d), float("nan"), device="cuda")
    o = kda.chunk_fwd(x["q"], x["k"], x["v"], x["z"], x["beta"], x["A"],
                      cu_seqlens=x["cu_seqlens"], S0=x["S0"], S_final=S_final)
    torch.cuda.synchronize()
    assert kda.device_status() == 0
    assert o.shape[0] == 0
    assert torch.equal(S_final, x["S0"])


@pytest.mark.parametrize("heads_per_group", [1, 3])
def test_two_pass_in_head_groups(kda, heads_per_group):
    """A workspace holding the records of only some heads makes the two-pass
    prefill run the heads in groups (here 4 heads as 4 x 1 or 3 + 1): same
    results as the oracle, ragged varlen batch with S0 and snapshots."""
    H = 4
    lengths = [300, 130, 64, 1]
    x = kda_inputs.make_prefill(H, 128, 128, lengths, seed=54, device="cuda", S0_std=0.02)
    n, total = len(lengths), x["k"].shape[0]
    kib = lambda b: (b + 1023) // 1024 * 1024
    table = kib((n + 1) * 4) + kib(((total + 63) // 64 + n) * 8) + kib(n * 4)  # starts, chunks, order
    per_head = ((total + 63) // 64 + n) * 73 * 1024
    assert kda.workspace_bytes(n, total, H, 128, 128) == table + H * per_head
    ws = torch.empty(table + heads_per_group * per_head, dtype=torch.uint8, device="cuda")
    offs = kda.snapshot_offsets(lengths)
    S_final = torch.full((n, H, 128, 128), float("nan"), device="cuda")
    snaps = torch.full((int(offs[-1]), H, 128, 128), float("nan"), device="cuda")
    o = kda.chunk_fwd(x["q"], x["k"], x["v"], x["z"], x["beta"], x["A"], cu_seqlens=x["cu_seqlens"],
                      S0=x["S0"], S_final=S_final, snaps=snaps, snap_offsets=offs, workspace=ws)
    torch.cuda.synchronize()
    assert kda.device_status() == 0
    ref = oracle_subset(x, list(range(n)), list(range(H)))
    assert o_err(f64(o), ref["o"]) <= O_TOL
    assert s_err(f64(S_final), ref["S_final"]) <= S_TOL
    assert s_err(f64(snaps), ref["snaps"]) <= S_TOL


# --- errors only the GPU can see -----------------------------------------------------------

def test_stalled_wait_times_out_and_the_next_call_is_clean(kda):
    """The KDA_TEST_STALL hook makes the tensor-core kernel wait on an mbarrier
    that nothing arms, with a small poll limit and nothing in flight: the wait
    gives up, KDA_ERR_TIMEOUT is in the status word, no output is written, and
    an ordinary call right after it on the same context matches the oracle."""
    assert kda.device_status() == 0
    x = kda_inputs.make_prefill(2, 128, 128, [130, 64], seed=61, device="cuda", S0_std=0.02)
    o = torch.full((194, 2, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    kda.chunk_fwd(x["q"], x["k"], x["v"], x["z"], x["beta"], x["A"], cu_seqlens=x["cu_seqlens"],
                  S0=x["S0"], o=o, pre=kda.TEST_STALL)
    torch.cuda.synchronize()
    assert kda.device_status() == kda.KDA_ERR_TIMEOUT
    assert torch.isnan(o.float()).all()  # the CTAs returned before writing anything
    assert kda.device_status() == 0      # read-and-reset cleared it
    o, S_final, snaps, offs, _ = check_all(x, kda)


def test_bad_slot_and_row_indices_are_skipped_and_reported(kda):
    """Out-of-range slot / snapshot-row indices are checked on the device: the
    row is skipped (no access outside the pool), KDA_ERR_SHAPE is recorded,
    and every in-range row is still computed correctly."""
    n, H, d = 4, 2, 64
    x = kda_inputs.make_prefill(H, d, d, [1] * n, seed=62, device="cuda", S0_std=0.02)
    pool = x["S0"].clone()
    slots = torch.tensor([2, 7, -1, 0], dtype=torch.int32, device="cuda")  # 7, -1 are bad
    before = pool.clone()
    o = torch.full((n, H, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    kda.decode_step(x["q"], x["k"], x["v"], x["z"], x["beta"], x["A"], pool, slots=slots, o=o)
    torch.cuda.synchronize()
    assert kda.device_status() == kda.KDA_ERR_SHAPE
    assert torch.isnan(o[1].float()).all() and torch.isnan(o[2].float()).all()
    assert torch.equal(pool[1], before[1]) and torch.equal(pool[3], before[3])
    st = np.ascontiguousarray(f64(before[[2, 0]]))
    o_ref = oracle.decode_step(*(f64(x[nm][[0, 3]]) for nm in ("q", "k", "v", "z", "beta")),
                               f64(x["A"]), st)
    assert o_err(f64(o[[0, 3]]), o_ref) <= O_TOL
    assert s_err(f64(pool[[2, 0]]), st) <= DECODE_TOL
    # snapshot restore: a row past the snapshots and a slot past the pool
    snaps = torch.randn((3, H, d, d), device="cuda")
    pool2 = torch.zeros((2, H, d, d), device="cuda")
    kda.state_snapshot(snaps, torch.tensor([1, 3, 0], dtype=torch.int64, device="cuda"), pool2,
                       torch.tensor([0, 1, 5], dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert kda.device_status() == kda.KDA_ERR_SHAPE
    assert torch.equal(pool2[0], snaps[1]) and torch.equal(pool2[1], torch.zeros_like(pool2[1]))
    # multi-token decode through a bad slot: that sequence is skipped
    y = kda_inputs.make_prefill(H, d, d, [3, 5], seed=63, device="cuda", S0_std=0.02)
    pool3 = y["S0"].clone()
    before3 = pool3.clone()
    kda.decode_tokens(y["q"], y["k"], y["v"], y["z"], y["beta"], y["A"], pool3,
                      torch.tensor([1, 9], dtype=torch.int32, device="cuda"), y["cu_seqlens"])
    torch.cuda.synchronize()
    assert kda.device_status() == kda.KDA_ERR_SHAPE
    assert torch.equal(pool3[0], before3[0])
    ref = oracle_subset(dict(y, S0=before3[[1, 0]].contiguous()), [0], [0, 1], snapshots=False)
    assert s_err(f64(pool3[1]), ref["S_final"][0]) <= S_TOL


def test_stream_status_words_tell_streams_apart(kda):
    """Two streams with a status word each (kda_stream_status_bind): a bad slot
    in a call on one stream and a timed-out wait in a call on the other are
    recorded in their own words; the device word and the other stream's word
    stay clear; after unbinding, the device word takes the codes again."""
    assert kda.device_status() == 0
    n, H, d = 4, 2, 64
    x = kda_inputs.make_prefill(H, d, d, [1] * n, seed=64, device="cuda", S0_std=0.02)
    y = kda_inputs.make_prefill(2, 128, 128, [130, 64], seed=61, device="cuda", S0_std=0.02)
    s_a, s_b = torch.cuda.Stream(), torch.cuda.Stream()
    w_a = torch.zeros(1, dtype=torch.int32, device="cuda")
    w_b = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    kda.stream_status_bind(w_a, s_a)
    kda.stream_status_bind(w_b, s_b)
    try:
        pool = x["S0"].clone()
        before = pool.clone()
        slots = torch.tensor([2, 7, -1, 0], dtype=torch.int32, device="cuda")  # 7, -1 are bad
        o_b = torch.full((194, 2, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
        torch.cuda.synchronize()
        kda.decode_step(x["q"], x["k"], x["v"], x["z"], x["beta"], x["A"], pool, slots=slots,
                        stream=s_a)
        kda.chunk_fwd(y["q"], y["k"], y["v"], y["z"], y["beta"], y["A"],
                      cu_seqlens=y["cu_seqlens"], S0=y["S0"], o=o_b, pre=kda.TEST_STALL,
                      stream=s_b)
        assert kda.stream_status(s_a) == kda.KDA_ERR_SHAPE
        assert kda.stream_status(s_b) == kda.KDA_ERR_TIMEOUT
        assert kda.stream_status(s_a) == 0 and kda.stream_status(s_b) == 0  # read and reset
        assert torch.isnan(o_b.float()).all()
        assert torch.equal(pool[1], before[1]) and torch.equal(pool[3], before[3])
        assert kda.device_status() == 0  # nothing reached the device word
    finally:
        kda.stream_status_bind(None, s_a)
        kda.stream_status_bind(None, s_b)
    with pytest.raises(kda.KDAError):
        kda.stream_status(s_a)  # no word is bound any more
    pool = x["S0"].clone()
    slots = torch.tensor([2, 7, -1, 0], dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    kda.decode_step(x["q"], x["k"], x["v"], x["z"], x["beta"], x["A"], pool, slots=slots,
                    stream=s_a)
    s_a.synchronize()
    assert kda.device_status() == kda.KDA_ERR_SHAPE
    assert int(w_a.item()) == 0


def test_stream_status_word_is_kept_by_a_captured_graph(kda):
    """A call captured into a CUDA graph on a stream with its own status word
    records into that word at every replay, also after the stream was unbound
    (the word bound at capture time is part of the graph)."""
    assert kda.device_status() == 0
    n, H, d = 4, 2, 64
    x = kda_inputs.make_prefill(H, d, d, [1] * n, seed=65, device="cuda", S0_std=0.02)
    pool = x["S0"].clone()
    slots = torch.tensor([2, 7, -1, 0], dtype=torch.int32, device="cuda")  # 7, -1 are bad
    o = torch.empty((n, H, d), dtype=torch.bfloat16, device="cuda")
    word = torch.zeros(1, dtype=torch.int32, device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # one uncaptured call first, on the same stream
        kda.decode_step(x["q"], x["k"], x["v"], x["z"], x["beta"], x["A"], pool, slots=slots,
                        o=o, stream=side)
    side.synchronize()
    assert kda.device_status() == kda.KDA_ERR_SHAPE
    kda.stream_status_bind(word, side)
    try:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            kda.decode_step(x["q"], x["k"], x["v"], x["z"], x["beta"], x["A"], pool,
                            slots=slots, o=o, stream=side)
    finally:
        kda.stream_status_bind(None, side)
    torch.cuda.synchronize()
    assert int(word.item()) == 0  # capturing runs nothing
    g.replay()
    torch.cuda.synchronize()
    assert int(word.item()) == kda.KDA_ERR_SHAPE
    assert kda.device_status() == 0
    del g


@pytest.mark.parametrize("workspace", [True, False])
def test_malformed_cu_seqlens_and_snap_offsets_are_reported(kda, workspace):
    """A decreasing cu_seqlens, or snap_offsets that do not match the lengths,
    are caught on the device (two-pass and single-pass kernels alike): the
    call touches nothing outside its arrays and records KDA_ERR_SHAPE; the
    same call with the correct arrays then matches the oracle."""
    lengths = [130, 64, 70]
    x = kda_inputs.make_prefill(2, 128, 128, lengths, seed=64, device="cuda", S0_std=0.02)
    total = x["k"].shape[0]
    ws = (torch.empty(kda.workspace_bytes(3, total, 2, 128, 128), dtype=torch.uint8,
                      device="cuda") if workspace else torch.empty(16, dtype=torch.uint8,
                                                                   device="cuda"))
    offs = kda.snapshot_offsets(lengths)
    snaps = torch.zeros((int(offs[-1]), 2, 128, 128), device="cuda")
    S_final = torch.zeros((3, 2, 128, 128), device="cuda")
    args = [x[nm] for nm in ("q", "k", "v", "z", "beta", "A")]
    bad_cu = torch.tensor([0, 150, 100, total], dtype=torch.int32, device="cuda")
    kda.chunk_fwd(*args, cu_seqlens=bad_cu, S0=x["S0"], S_final=S_final, snaps=snaps,
                  snap_offsets=offs, workspace=ws)
    torch.cuda.synchronize()
    assert kda.device_status() == kda.KDA_ERR_SHAPE
    bad_offs = torch.tensor([0, 2, 2, 5], dtype=torch.int64, device="cuda")  # seq 1 needs 1 row
    kda.chunk_fwd(*args, cu_seqlens=x["cu_seqlens"], S0=x["S0"], S_final=S_final, snaps=snaps,
                  snap_offsets=bad_offs, workspace=ws)
    torch.cuda.synchronize()
    assert kda.device_status() == kda.KDA_ERR_SHAPE
    o = kda.chunk_fwd(*args, cu_seqlens=x["cu_seqlens"], S0=x["S0"], S_final=S_final,
                      snaps=snaps, snap_offsets=offs, workspace=ws)
    torch.cuda.synchronize()
    assert kda.device_status() == 0
    ref = oracle_subset(x, [0, 1, 2], [0, 1])
    assert o_err(f64(o), ref["o"]) <= O_TOL
    assert s_err(f64(S_final), ref["S_final"]) <= S_TOL
    assert s_err(f64(snaps), ref["snaps"]) <= S_TOL


def test_fp16_range_is_reported_not_silent(kda):
    """The state and the chunk terms U, W pass through fp16 tensor-core
    operands.  Values of |v| ~ 3e4 overflow that range: the call records
    KDA_ERR_RANGE instead of returning silent infinities.  |v| ~ 300 (and S0
    to match) stays inside it and matches the oracle."""
    x = kda_inputs.make_prefill(2, 128, 128, [200, 64], seed=65, device="cuda", S0_std=0.02)
    big = dict(x, v=(x["v"].float() * 3e4).to(torch.bfloat16))
    n_seq = 2
    S_final = torch.empty((n_seq, 2, 128, 128), device="cuda")
    kda.chunk_fwd(big["q"], big["k"], big["v"], big["z"], big["beta"], big["A"],
                  cu_seqlens=big["cu_seqlens"], S0=big["S0"], S_final=S_final)
    torch.cuda.synchronize()
    assert kda.device_status() & kda.KDA_ERR_RANGE
    ok = dict(x, v=(x["v"].float() * 300).to(torch.bfloat16), S0=x["S0"] * 1.5e4)
    check_all(ok, kda)
