"""Seeded synthetic inputs for KDA prefill and decode.

This module is shared by the tests, the smoke check and the benchmark.  It
only draws random numbers in the shapes and distributions of the workloads;
it holds none of the attention method's arithmetic (no gate, no decay, no
recurrence).  The preconditions of the inputs - unit-norm q and k per token
and head, beta already passed through a sigmoid - are part of the recipe.

Recipe (all workloads): q, k ~ N(0, 1) drawn in fp32, L2-normalised over the
key dimension per (token, head), then rounded to bf16; v ~ N(0, 1) -> bf16;
z ~ N(0, 1) -> bf16; beta = sigmoid(N(0, 1)) -> bf16; A ~ U(-1, 1) fp32, one
per head; initial states S0 ~ N(0, std^2) fp32 where the workload has them.
Draw order is q, k, v, z, beta, A, S0 from one torch.Generator seeded with
the workload's seed.  Variable sequence lengths come from NumPy's
default_rng(seed) so that they do not depend on the device.
"""
from __future__ import annotations

import math

import numpy as np
import torch

# Workloads.  Sizes follow the 1M-token context and the 3:1 KDA/MLA layer
# shapes that "Kimi K3 Technical Report - Open Frontier Intelligence" describes
# (Key claims; sec. 2.1); head count and head size are this library's choice.
WORKLOADS = {
    "tiny": dict(kind="prefill", B=1, H=2, T=256, dk=64, dv=64, chunk=64, seed=1000,
                 snapshots=True),
    "mid": dict(kind="prefill", B=4, H=16, T=8192, dk=128, dv=128, chunk=64, seed=1001,
                snapshots=True),
    "varlen": dict(kind="varlen", n_seq=64, len_lo=512, len_hi=32768, H=32, dk=128, dv=128,
                   chunk=64, seed=1002, S0_std=0.02, snapshots=True),
    "decode": dict(kind="decode", batch=512, H=32, dk=128, dv=128, steps=1000, seed=1003,
                   state_std=0.02),
    "long": dict(kind="prefill", B=1, H=16, T=1048576, dk=128, dv=128, chunk=64, seed=1004,
                 snapshots=True),
}

_PIECE = 1 << 24  # elements drawn per call, bounds temporary memory


def _randn(shape, gen, device, std=1.0):
    """N(0, std^2) fp32 tensor drawn in fixed-size pieces (deterministic)."""
    n = math.prod(shape)
    out = torch.empty(n, dtype=torch.float32, device=device)
    for s in range(0, n, _PIECE):
        e = min(n, s + _PIECE)
        out[s:e] = torch.randn(e - s, generator=gen, device=device, dtype=torch.float32)
    if std != 1.0:
        out.mul_(std)
    return out.view(*shape)


def _unit_rows_bf16(shape, gen, device):
    """N(0,1) rows normalised to unit L2 norm over the last dim, then bf16."""
    x = _randn(shape, gen, device)
    rows = x.view(-1, shape[-1])
    for s in range(0, rows.shape[0], 1 << 16):
        r = rows[s:s + (1 << 16)]
        r.div_(torch.linalg.vector_norm(r, dim=-1, keepdim=True).clamp_min(1e-30))
    return x.to(torch.bfloat16)


def varlen_lengths(n_seq, lo, hi, seed):
    """Sequence lengths ~ uniform integers in [lo, hi] (inclusive)."""
    return [int(x) for x in np.random.default_rng(seed).integers(lo, hi + 1, size=n_seq)]


def make_prefill(H, dk, dv, lengths, seed, device="cpu", S0_std=None):
    """Packed inputs for a batch of sequences with the given lengths.

    Returns dict(q, k, z [total, H, dk] bf16; v [total, H, dv] bf16;
    beta [total, H] bf16; A [H] fp32; S0 [n_seq, H, dk, dv] fp32 or None;
    cu_seqlens [n_seq + 1] int32 on ``device``; lengths list).
    """
    total = int(sum(lengths))
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    q = _unit_rows_bf16((total, H, dk), gen, device)
    k = _unit_rows_bf16((total, H, dk), gen, device)
    v = _randn((total, H, dv), gen, device).to(torch.bfloat16)
    z = _randn((total, H, dk), gen, device).to(torch.bfloat16)
    beta = torch.sigmoid(_randn((total, H), gen, device)).to(torch.bfloat16)
    A = (torch.rand(H, generator=gen, device=device, dtype=torch.float32) * 2.0 - 1.0)
    S0 = None
    if S0_std is not None:
        S0 = _randn((len(lengths), H, dk, dv), gen, device, std=float(S0_std))
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32), device=device)
    return dict(q=q, k=k, v=v, z=z, beta=beta, A=A, S0=S0, cu_seqlens=cu,
                lengths=[int(x) for x in lengths])


def make_raw_prefill(H, dk, dv, lengths, seed, device="cpu", S0_std=None):
    """Inputs as a model's projections give them, before the pre-ops: q, k rows
    N(0, 1) times a per-row scale U[0.25, 4] (not unit length), beta the raw
    N(0, 1) logit.  Everything else as make_prefill.  bf16 like the others."""
    total = int(sum(lengths))
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    q = _randn((total, H, dk), gen, device)
    k = _randn((total, H, dk), gen, device)
    q.mul_(torch.rand((total, H, 1), generator=gen, device=device) * 3.75 + 0.25)
    k.mul_(torch.rand((total, H, 1), generator=gen, device=device) * 3.75 + 0.25)
    v = _randn((total, H, dv), gen, device).to(torch.bfloat16)
    z = _randn((total, H, dk), gen, device).to(torch.bfloat16)
    beta = _randn((total, H), gen, device).to(torch.bfloat16)
    A = (torch.rand(H, generator=gen, device=device, dtype=torch.float32) * 2.0 - 1.0)
    S0 = None
    if S0_std is not None:
        S0 = _randn((len(lengths), H, dk, dv), gen, device, std=float(S0_std))
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32), device=device)
    return dict(q=q.to(torch.bfloat16), k=k.to(torch.bfloat16), v=v, z=z, beta=beta, A=A, S0=S0,
                cu_seqlens=cu, lengths=[int(x) for x in lengths])


def make_workload_prefill(name, device="cpu", **override):
    """Inputs of a named prefill workload ('tiny', 'mid', 'varlen', 'long')."""
    w = dict(WORKLOADS[name])
    w.update(override)
    if w["kind"] == "varlen":
        lengths = varlen_lengths(w["n_seq"], w["len_lo"], w["len_hi"], w["seed"])
        return make_prefill(w["H"], w["dk"], w["dv"], lengths, w["seed"], device,
                            S0_std=w.get("S0_std"))
    return make_prefill(w["H"], w["dk"], w["dv"], [w["T"]] * w["B"], w["seed"], device,
                        S0_std=w.get("S0_std"))


def make_decode_state(batch, H, dk, dv, seed, device="cpu", std=0.02):
    """Resident states ~ N(0, std^2) fp32 [batch, H, dk, dv] and A [H]."""
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    state = _randn((batch, H, dk, dv), gen, device, std=std)
    A = (torch.rand(H, generator=gen, device=device, dtype=torch.float32) * 2.0 - 1.0)
    return state, A


def make_decode_token(batch, H, dk, dv, seed, step, device="cpu"):
    """Fresh one-token inputs of decode step ``step`` (0-based)."""
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed) * 1_000_003 + 7919 * (int(step) + 1))
    q = _unit_rows_bf16((batch, H, dk), gen, device)
    k = _unit_rows_bf16((batch, H, dk), gen, device)
    v = _randn((batch, H, dv), gen, device).to(torch.bfloat16)
    z = _randn((batch, H, dk), gen, device).to(torch.bfloat16)
    beta = torch.sigmoid(_randn((batch, H), gen, device)).to(torch.bfloat16)
    return dict(q=q, k=k, v=v, z=z, beta=beta)


def to_f64(t):
    """Exact upcast of a (bf16 / fp32) tensor to a NumPy float64 array."""
    return t.detach().to("cpu").to(torch.float64).numpy()
