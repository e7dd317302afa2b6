"""GB300-native Kimi Delta Attention (KDA): chunkwise prefill and recurrent decode.

A thin Python binding over the C ABI in ``include/kda.h`` (the CUDA library
``libkda_gb300.so`` built from ``csrc/``).  The functions here only check and
marshal arguments - every step of the computation runs in the library's CUDA
kernels.  PyTorch supplies device memory and the current stream.

The library must be built first (``build()``); without it every call raises,
there is no CPU or PyTorch fallback.
"""
from __future__ import annotations

import ctypes
import os

import torch

from .build import LIB_PATH, build  # noqa: F401  (re-exported)

GMIN = -5.0   # "Kimi K3 Technical Report - Open Frontier Intelligence", sec. 2.1.1
CHUNK = 64
# Arithmetic of the prefill: bf16 in/out with tf32 / bf16 / fp16 tensor-core
# operands, fp32 accumulation and fp32 state.
PREFILL_COMPUTE_DTYPE = "bf16"

# Input pre-ops (KDA_PRE_* in kda.h): L2-normalise q, k rows; sigmoid of beta.
PRE_L2NORM_QK = 1
PRE_SIGMOID_BETA = 2
# Split-phase calls of chunk_fwd (KDA_PASS_* in kda.h): only the chunk
# preparation, or only the state pass from the records it left in `workspace`.
PASS_PREPARE = 0x100
PASS_STATE = 0x200
# Test hook (KDA_TEST_STALL in kda.h): the kernel gives up on a wait nothing
# arms and records KDA_ERR_TIMEOUT in the device status word.
TEST_STALL = 0x10000

KDA_OK = 0
STATUS_NAMES = {0: "KDA_OK", 1: "KDA_ERR_NULL", 2: "KDA_ERR_SHAPE", 3: "KDA_ERR_ALIGN",
                4: "KDA_ERR_UNSUPPORTED", 5: "KDA_ERR_WORKSPACE", 6: "KDA_ERR_CUDA",
                7: "KDA_ERR_TIMEOUT", 8: "KDA_ERR_RANGE"}
KDA_ERR_NULL = 1
KDA_ERR_SHAPE = 2
KDA_ERR_TIMEOUT = 7
KDA_ERR_RANGE = 8

EXPORTED = ("kda_status_string", "kda_version", "kda_chunk_fwd_workspace_bytes",
            "kda_chunk_fwd", "kda_decode_step", "kda_state_snapshot", "kda_device_status",
            "kda_chunk_fwd_noalloc", "kda_decode_tokens", "kda_chunk_fwd_ex",
            "kda_decode_step_ex", "kda_stream_status_bind", "kda_stream_status")

_lib = None


class KDAError(RuntimeError):
    """A non-zero kda_status returned by the library."""

    def __init__(self, fn, status):
        self.status = int(status)
        super().__init__(f"{fn} failed: {STATUS_NAMES.get(self.status, self.status)}")


def lib():
    """The loaded CUDA library (ctypes handle).  Raises if it was not built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: run "
                              "linear_attention_serving_chunk_gb300.build() first")
        L = ctypes.CDLL(LIB_PATH)
        P, I, I64, F, SZ, U = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float,
                               ctypes.c_size_t, ctypes.c_uint)
        L.kda_status_string.restype = ctypes.c_char_p
        L.kda_status_string.argtypes = [I]
        L.kda_version.restype = I
        L.kda_version.argtypes = []
        L.kda_chunk_fwd_workspace_bytes.restype = SZ
        L.kda_chunk_fwd_workspace_bytes.argtypes = [I, I64, I, I, I, I]
        L.kda_chunk_fwd.restype = I
        L.kda_chunk_fwd.argtypes = [P, P, P, P, P, P, F, P, I, I64, I, I, I, I, P, P, P, P, P,
                                    P, SZ, P]
        L.kda_chunk_fwd_ex.restype = I
        L.kda_chunk_fwd_ex.argtypes = [P, P, P, P, P, P, F, P, I, I64, I, I, I, I, U, P, P, P,
                                       P, P, P, SZ, P]
        L.kda_chunk_fwd_noalloc.restype = I
        L.kda_chunk_fwd_noalloc.argtypes = [P, P, P, P, P, P, F, P, I, I64, I, I, I, I, P, P, P,
                                            P, P, P]
        L.kda_decode_tokens.restype = I
        L.kda_decode_tokens.argtypes = [P, P, P, P, P, P, F, P, I, I64, I, I, I, U, P, I, P, I,
                                        P, P]
        L.kda_decode_step.restype = I
        L.kda_decode_step.argtypes = [P, P, P, P, P, P, F, P, I, P, I, I, I, I, P, P]
        L.kda_decode_step_ex.restype = I
        L.kda_decode_step_ex.argtypes = [P, P, P, P, P, P, F, P, I, P, I, I, I, I, U, P, P]
        L.kda_state_snapshot.restype = I
        L.kda_state_snapshot.argtypes = [P, I64, P, P, I, P, I, I, I, I, P]
        L.kda_device_status.restype = I
        L.kda_device_status.argtypes = [I]
        L.kda_stream_status_bind.restype = I
        L.kda_stream_status_bind.argtypes = [P, P]
        L.kda_stream_status.restype = I
        L.kda_stream_status.argtypes = [P, I]
        _lib = L
    return _lib


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _check(t, name, dtype, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def _raise_on(fn, status):
    if status != KDA_OK:
        raise KDAError(fn, status)


def snapshot_offsets(lengths, chunk=CHUNK, device="cuda"):
    """Snapshot row offsets [n_seq + 1] (int64): prefix sums of floor(L / chunk)."""
    offs = [0]
    for L in lengths:
        offs.append(offs[-1] + int(L) // chunk)
    return torch.tensor(offs, dtype=torch.int64, device=device)


def workspace_bytes(n_seq, total_tokens, H, dk, dv, chunk=CHUNK):
    return int(lib().kda_chunk_fwd_workspace_bytes(n_seq, total_tokens, H, dk, dv, chunk))


def chunk_fwd(q, k, v, z, beta, A, gmin=GMIN, cu_seqlens=None, n_seq=None, S0=None, o=None,
              S_final=None, snaps=None, snap_offsets=None, workspace=None, chunk=CHUNK,
              pre=0, stream=None):
    """KDA prefill (kda_chunk_fwd).  Shapes: q, k, z [total, H, dk] bf16;
    v [total, H, dv] bf16; beta [total, H] bf16; A [H] fp32; cu_seqlens int32
    [n_seq + 1] or None (then n_seq equal sequences, default 1); S0, S_final
    [n_seq, H, dk, dv] fp32; snaps [rows, H, dk, dv] fp32 with snap_offsets
    int64 [n_seq + 1].  Outputs that are None are allocated (o) or skipped
    (S_final, snaps).  pre: PRE_* flags (raw q, k and beta logits; calls
    kda_chunk_fwd_ex when non-zero).  Returns o."""
    total, H, dk = k.shape
    dv = v.shape[2]
    for t, nm in ((q, "q"), (k, "k"), (z, "z")):
        _check(t, nm, torch.bfloat16, (total, H, dk))
    _check(v, "v", torch.bfloat16, (total, H, dv))
    _check(beta, "beta", torch.bfloat16, (total, H))
    _check(A, "A", torch.float32, (H,))
    if cu_seqlens is not None:
        _check(cu_seqlens, "cu_seqlens", torch.int32)
        n_seq = cu_seqlens.numel() - 1
    elif n_seq is None:
        n_seq = 1
    if S0 is not None:
        _check(S0, "S0", torch.float32, (n_seq, H, dk, dv))
    if S_final is not None:
        _check(S_final, "S_final", torch.float32, (n_seq, H, dk, dv))
    if snaps is not None:
        _check(snaps, "snaps", torch.float32)
        if snap_offsets is not None:
            _check(snap_offsets, "snap_offsets", torch.int64, (n_seq + 1,))
    if o is None:
        o = torch.empty((total, H, dv), dtype=torch.bfloat16, device=k.device)
    _check(o, "o", torch.bfloat16, (total, H, dv))
    need = workspace_bytes(n_seq, total, H, dk, dv, chunk)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=k.device)
        if stream is not None and isinstance(stream, torch.cuda.Stream):
            # allocated on the current stream, used on `stream`: keep the
            # block out of the allocator until the call's kernels are done
            workspace.record_stream(stream)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    if pre:
        st = lib().kda_chunk_fwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(z), _ptr(beta), _ptr(A),
                                    float(gmin), _ptr(cu_seqlens), int(n_seq), int(total),
                                    int(H), int(dk), int(dv), int(chunk), int(pre), _ptr(S0),
                                    _ptr(o), _ptr(S_final), _ptr(snaps), _ptr(snap_offsets),
                                    _ptr(workspace), ws_bytes, _stream(stream))
        _raise_on("kda_chunk_fwd_ex", st)
        return o
    st = lib().kda_chunk_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(z), _ptr(beta), _ptr(A),
                             float(gmin), _ptr(cu_seqlens), int(n_seq), int(total), int(H),
                             int(dk), int(dv), int(chunk), _ptr(S0), _ptr(o), _ptr(S_final),
                             _ptr(snaps), _ptr(snap_offsets), _ptr(workspace), ws_bytes,
                             _stream(stream))
    _raise_on("kda_chunk_fwd", st)
    return o


def decode_step(q, k, v, z, beta, A, state_pool, slots=None, gmin=GMIN, o=None, pre=0,
                stream=None):
    """One decode step (kda_decode_step), in place on state_pool
    [n_slots, H, dk, dv] fp32.  q, k, z [n, H, dk]; v [n, H, dv]; beta [n, H]
    bf16; slots int32 [n] or None; pre: PRE_* flags (kda_decode_step_ex when
    non-zero).  Returns o [n, H, dv] bf16."""
    n, H, dk = k.shape
    dv = v.shape[2]
    for t, nm in ((q, "q"), (k, "k"), (z, "z")):
        _check(t, nm, torch.bfloat16, (n, H, dk))
    _check(v, "v", torch.bfloat16, (n, H, dv))
    _check(beta, "beta", torch.bfloat16, (n, H))
    _check(A, "A", torch.float32, (H,))
    _check(state_pool, "state_pool", torch.float32)
    if state_pool.dim() != 4 or tuple(state_pool.shape[1:]) != (H, dk, dv):
        raise ValueError("state_pool must be [n_slots, H, dk, dv]")
    if slots is None:
        if state_pool.shape[0] < n:
            raise ValueError("state_pool has fewer slots than rows")
    else:
        _check(slots, "slots", torch.int32, (n,))
    if o is None:
        o = torch.empty((n, H, dv), dtype=torch.bfloat16, device=k.device)
    _check(o, "o", torch.bfloat16, (n, H, dv))
    n_slots = int(state_pool.shape[0])
    if pre:
        st = lib().kda_decode_step_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(z), _ptr(beta), _ptr(A),
                                      float(gmin), _ptr(state_pool), n_slots, _ptr(slots), int(n),
                                      int(H), int(dk), int(dv), int(pre), _ptr(o),
                                      _stream(stream))
        _raise_on("kda_decode_step_ex", st)
        return o
    st = lib().kda_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(z), _ptr(beta), _ptr(A),
                               float(gmin), _ptr(state_pool), n_slots, _ptr(slots), int(n),
                               int(H), int(dk), int(dv), _ptr(o), _stream(stream))
    _raise_on("kda_decode_step", st)
    return o


def decode_tokens(q, k, v, z, beta, A, state_pool, slots, cu_seqlens, commit=True, gmin=GMIN,
                  o=None, pre=0, stream=None):
    """Several tokens per sequence on resident states (kda_decode_tokens):
    sequence b's tokens are rows cu_seqlens[b]:cu_seqlens[b+1] of q, k, v, z,
    beta; its state is state_pool[slots[b]], updated in place when commit.
    pre: PRE_* flags.  Returns o [total, H, dv] bf16."""
    total, H, dk = k.shape
    dv = v.shape[2]
    for t, nm in ((q, "q"), (k, "k"), (z, "z")):
        _check(t, nm, torch.bfloat16, (total, H, dk))
    _check(v, "v", torch.bfloat16, (total, H, dv))
    _check(beta, "beta", torch.bfloat16, (total, H))
    _check(A, "A", torch.float32, (H,))
    _check(cu_seqlens, "cu_seqlens", torch.int32)
    n = cu_seqlens.numel() - 1
    _check(slots, "slots", torch.int32, (n,))
    _check(state_pool, "state_pool", torch.float32)
    if state_pool.dim() != 4 or tuple(state_pool.shape[1:]) != (H, dk, dv):
        raise ValueError("state_pool must be [n_slots, H, dk, dv]")
    if o is None:
        o = torch.empty((total, H, dv), dtype=torch.bfloat16, device=k.device)
    _check(o, "o", torch.bfloat16, (total, H, dv))
    st = lib().kda_decode_tokens(_ptr(q), _ptr(k), _ptr(v), _ptr(z), _ptr(beta), _ptr(A),
                                 float(gmin), _ptr(cu_seqlens), int(n), int(total), int(H),
                                 int(dk), int(dv), int(pre), _ptr(state_pool),
                                 int(state_pool.shape[0]), _ptr(slots), 1 if commit else 0,
                                 _ptr(o), _stream(stream))
    _raise_on("kda_decode_tokens", st)
    return o


def state_snapshot(snaps, src_idx, state_pool, dst_slots, stream=None):
    """Copy snapshot rows src_idx (int64 [n]) into state slots dst_slots
    (int32 [n]) (kda_state_snapshot)."""
    _check(snaps, "snaps", torch.float32)
    _check(state_pool, "state_pool", torch.float32)
    n = src_idx.numel()
    _check(src_idx, "src_idx", torch.int64, (n,))
    _check(dst_slots, "dst_slots", torch.int32, (n,))
    _, H, dk, dv = state_pool.shape
    if tuple(snaps.shape[1:]) != (H, dk, dv):
        raise ValueError("snaps and state_pool disagree on (H, dk, dv)")
    st = lib().kda_state_snapshot(_ptr(snaps), int(snaps.shape[0]), _ptr(src_idx),
                                  _ptr(state_pool), int(state_pool.shape[0]), _ptr(dst_slots),
                                  int(n), int(H), int(dk), int(dv), _stream(stream))
    _raise_on("kda_state_snapshot", st)


def device_status(reset=True):
    """Read (and clear) the device status word; synchronises the device."""
    return int(lib().kda_device_status(1 if reset else 0))


def stream_status_bind(word, stream=None):
    """Give `stream` (default: the current stream) a status word of its own:
    `word`, a zeroed one-element int32 CUDA tensor that the caller keeps
    alive while it is bound, or None to remove the binding."""
    if word is not None:
        _check(word, "word", torch.int32, (1,))
    _raise_on("kda_stream_status_bind", lib().kda_stream_status_bind(_stream(stream), _ptr(word)))


def stream_status(stream=None, reset=True):
    """Read (and clear) the word bound to `stream`; synchronises that stream only."""
    st = int(lib().kda_stream_status(_stream(stream), 1 if reset else 0))
    if st == KDA_ERR_NULL:
        raise KDAError("kda_stream_status", st)
    return st
