"""Host-side checks of the C ABI: the library loads, exports every function
declared in include/kda.h, and rejects bad arguments before launching
anything (no GPU needed)."""
import ctypes
import os
import re

import pytest

import linear_attention_serving_chunk_gb300 as kda

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kda.h")


@pytest.fixture(scope="module")
def L():
    kda.build()
    return kda.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kda_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_expected_entry_points():
    names = declared_functions()
    for fn in ("kda_chunk_fwd", "kda_decode_step", "kda_state_snapshot"):
        assert fn in names
    assert set(names) == set(kda.EXPORTED)


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), f"{name} is declared in kda.h but not exported"


def test_status_strings_and_version(L):
    assert L.kda_version() >= 100
    for s in range(9):
        assert L.kda_status_string(s)
    assert L.kda_status_string(8) != b"unknown status"
    assert L.kda_status_string(99) == b"unknown status"


def test_stream_status_binding_table(L):
    """kda_stream_status_bind is host-side bookkeeping (nothing is enqueued, so
    the pointers below are never dereferenced): a misaligned word is refused,
    64 streams can be bound and a 65th cannot, binding again replaces the word,
    unbinding frees a place and is a no-op for an unbound stream, and reading
    an unbound stream's word is KDA_ERR_NULL."""
    word = ctypes.c_void_p(0x20000)
    streams = [ctypes.c_void_p(0x1000 + 16 * i) for i in range(65)]
    try:
        assert L.kda_stream_status_bind(streams[0], ctypes.c_void_p(0x20002)) == 3
        for s in streams[:64]:
            assert L.kda_stream_status_bind(s, word) == 0
        assert L.kda_stream_status_bind(streams[64], word) == 2
        assert L.kda_stream_status_bind(streams[3], ctypes.c_void_p(0x20004)) == 0
        assert L.kda_stream_status_bind(streams[3], None) == 0
        assert L.kda_stream_status_bind(streams[64], word) == 0
        assert L.kda_stream_status_bind(streams[3], None) == 0
        assert L.kda_stream_status(streams[3], 0) == 1
    finally:
        for s in streams:
            L.kda_stream_status_bind(s, None)


def _chunk_args(**kw):
    fake = ctypes.c_void_p(0x10000)  # never dereferenced: every call below is rejected first
    args = dict(q=fake, k=fake, v=fake, z=fake, beta=fake, A=fake, gmin=-5.0, cu=None, n_seq=1,
                total=128, H=2, dk=64, dv=64, chunk=64, S0=None, o=fake, S_final=None,
                snaps=None, snap_offsets=None, ws=None, ws_bytes=0, stream=None)
    args.update(kw)
    return list(args.values())


@pytest.mark.parametrize("kw,status", [
    (dict(dk=96), 4), (dict(dv=32), 4), (dict(chunk=32), 4), (dict(gmin=-8.0), 4),
    (dict(gmin=0.5), 4), (dict(gmin=float("nan")), 4), (dict(H=0), 2), (dict(n_seq=-1), 2),
    (dict(total=-5), 2), (dict(n_seq=3, total=128), 2), (dict(q=None), 1), (dict(A=None), 1),
    (dict(o=None), 1), (dict(q=ctypes.c_void_p(0x10008)), 3),
    (dict(snaps=ctypes.c_void_p(0x20000), cu=ctypes.c_void_p(0x30000)), 1),
    (dict(n_seq=0, total=0), 0),
])
def test_chunk_fwd_rejects_before_launch(L, kw, status):
    assert L.kda_chunk_fwd(*_chunk_args(**kw)) == status


@pytest.mark.parametrize("kw,status", [
    (dict(dk=48), 4), (dict(gmin=-7.0), 4), (dict(n=-1), 2), (dict(H=0), 2), (dict(q=None), 1),
    (dict(pool=None), 1), (dict(o=ctypes.c_void_p(0x10004)), 3), (dict(n=0), 0),
    # rows without a slot array need that many slots; a negative pool size is malformed
    (dict(n_slots=3), 2), (dict(n_slots=-1), 2),
])
def test_decode_step_rejects_before_launch(L, kw, status):
    fake = ctypes.c_void_p(0x10000)
    a = dict(q=fake, k=fake, v=fake, z=fake, beta=fake, A=fake, gmin=-5.0, pool=fake, n_slots=4,
             slots=None, n=4, H=2, dk=64, dv=64, o=fake, stream=None)
    a.update(kw)
    assert L.kda_decode_step(*a.values()) == status


@pytest.mark.parametrize("kw,status", [
    (dict(dk=32), 4), (dict(n=-2), 2), (dict(snaps=None), 1), (dict(dst=None), 1),
    (dict(src=ctypes.c_void_p(0x10002)), 3), (dict(n=0), 0), (dict(n_rows=-1), 2),
    (dict(n_slots=-3), 2),
])
def test_state_snapshot_rejects_before_launch(L, kw, status):
    fake = ctypes.c_void_p(0x10000)
    a = dict(snaps=fake, n_rows=8, src=fake, pool=fake, n_slots=4, dst=fake, n=2, H=2, dk=64,
             dv=64, stream=None)
    a.update(kw)
    assert L.kda_state_snapshot(*a.values()) == status


@pytest.mark.parametrize("kw,status", [
    (dict(dk=80), 4), (dict(n=-1), 2), (dict(slots=None), 1), (dict(cu=None), 1),
    (dict(pool=None), 1), (dict(o=ctypes.c_void_p(0x10008)), 3), (dict(n=0, total=0), 0),
    (dict(n_slots=-1), 2), (dict(total=0), 0),
])
def test_decode_tokens_rejects_before_launch(L, kw, status):
    fake = ctypes.c_void_p(0x10000)
    a = dict(q=fake, k=fake, v=fake, z=fake, beta=fake, A=fake, gmin=-5.0, cu=fake, n=4,
             total=20, H=2, dk=64, dv=64, pre=0, pool=fake, n_slots=4, slots=fake, commit=1,
             o=fake, stream=None)
    a.update(kw)
    assert L.kda_decode_tokens(*a.values()) == status


def _ex_args(**kw):
    """kda_chunk_fwd_ex arguments: kda_chunk_fwd's with `pre` after chunk."""
    args = _chunk_args(**{k: v for k, v in kw.items() if k != "pre"})
    if "ws_bytes" in kw:  # a (fake, never touched) workspace pointer of that size
        args[19] = ctypes.c_void_p(0x40000)
    return args[:14] + [kw.get("pre", 0)] + args[14:]


@pytest.mark.parametrize("kw,status", [
    (dict(pre=0x300, dk=128, dv=128), 4), (dict(pre=0x100), 5),
    # the stall test hook does not combine with a split-phase flag
    (dict(pre=0x10100, dk=128, dv=128), 4), (dict(pre=0x10000, total=0, n_seq=1), 4),
    (dict(pre=0x100, dk=128, dv=128), 5), (dict(pre=0x200, dk=128, dv=128, ws_bytes=4096), 5),
    (dict(pre=4), 4), (dict(pre=0x80000000), 4), (dict(pre=3, dk=96), 4),
    (dict(pre=3, q=None), 1), (dict(pre=1, H=0), 2), (dict(pre=3, n_seq=0, total=0), 0),
    (dict(pre=2, q=ctypes.c_void_p(0x10008)), 3),
])
def test_chunk_fwd_ex_rejects_before_launch(L, kw, status):
    assert L.kda_chunk_fwd_ex(*_ex_args(**kw)) == status


@pytest.mark.parametrize("kw,status", [
    (dict(pre=8), 4), (dict(pre=3, dk=48), 4), (dict(pre=3, q=None), 1), (dict(pre=1, n=0), 0),
])
def test_decode_step_ex_rejects_before_launch(L, kw, status):
    fake = ctypes.c_void_p(0x10000)
    a = dict(q=fake, k=fake, v=fake, z=fake, beta=fake, A=fake, gmin=-5.0, pool=fake, n_slots=4,
             slots=None, n=4, H=2, dk=64, dv=64, pre=0, o=fake, stream=None)
    a.update(kw)
    assert L.kda_decode_step_ex(*a.values()) == status


def test_decode_tokens_rejects_unknown_pre_flags(L):
    fake = ctypes.c_void_p(0x10000)
    assert L.kda_decode_tokens(fake, fake, fake, fake, fake, fake, -5.0, fake, 4, 20, 2, 64, 64,
                               16, fake, 4, fake, 1, fake, None) == 4


def test_workspace_query_is_pure_host(L):
    assert L.kda_chunk_fwd_workspace_bytes(4, 4 * 8192, 16, 128, 128, 64) >= 0


REC = 73 * 1024  # one (chunk, head) record of the two-pass prefill


def table(n_seq, total):
    """The varlen tables ahead of the records: the chunk start of every
    sequence (int32 [n_seq + 1]), the first token and length of every chunk
    (int32 x 2 per chunk, for up to ceil(T/64) + n_seq chunks) and the state
    pass's order of the sequences (int32 [n_seq]), each rounded up to 1 KiB."""
    kib = lambda b: (b + 1023) // 1024 * 1024
    return kib((n_seq + 1) * 4) + kib(((total + 63) // 64 + n_seq) * 8) + kib(n_seq * 4)


@pytest.mark.parametrize("n_seq,total,H,dk,dv,chunk,expect", [
    # the bench workload: two passes, records of every head for ceil(T/64) + n_seq
    # chunks after the tables
    (4, 4 * 8192, 16, 128, 128, 64, table(4, 4 * 8192) + (512 + 4) * 16 * REC),
    # one 2^20-token sequence, 16 heads: the segment scan (64 segments of 16,384
    # tokens: three [64, 16, 128, 128] fp32 arrays) plus every chunk's record
    (1, 1 << 20, 16, 128, 128, 64, 3 * 64 * 16 * 128 * 128 * 4 + (1 << 14) * 16 * REC),
    # too short for four segments of at least 4096 tokens: two passes
    (1, 8192, 4, 128, 128, 64, table(1, 8192) + (128 + 1) * 4 * REC),
    # 64-channel heads run the same two passes (records keep the 128-channel tiles)
    (1, 256, 2, 64, 64, 64, table(1, 256) + (4 + 1) * 2 * REC),
    (3, 300, 2, 128, 64, 64, table(3, 300) + (5 + 3) * 2 * REC),
    # only chunk = 64 exists
    (4, 4 * 8192, 16, 128, 128, 32, 0),
])
def test_workspace_bytes_formula(L, n_seq, total, H, dk, dv, chunk, expect):
    """The sizes include/kda.h documents for kda_chunk_fwd_workspace_bytes."""
    L.kda_chunk_fwd_workspace_bytes.restype = ctypes.c_size_t
    L.kda_chunk_fwd_workspace_bytes.argtypes = [ctypes.c_int, ctypes.c_int64, ctypes.c_int,
                                                ctypes.c_int, ctypes.c_int, ctypes.c_int]
    assert L.kda_chunk_fwd_workspace_bytes(n_seq, total, H, dk, dv, chunk) == expect


def test_python_binding_fails_loudly_without_cuda_tensors(L):
    import torch
    x = torch.zeros(64, 1, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        kda.chunk_fwd(x, x, x, x, torch.zeros(64, 1, dtype=torch.bfloat16),
                      torch.zeros(1, dtype=torch.float32))


def test_noalloc_scratch_decision_matches_chunk_fwd(L):
    """kda_chunk_fwd_noalloc needs its fixed scratch only where kda_chunk_fwd
    would take the segment scan, and a scan beyond that scratch falls back to
    the single-pass kernel instead of being refused.  One 2^20-token sequence
    with 16 heads and snapshots: without snap_offsets the scan would need
    192 MiB; with snap_offsets kda_chunk_fwd takes no scan.  Either way the call
    passes the scratch decision and stops at the next host check here (a
    misaligned o: KDA_ERR_ALIGN), launching nothing."""
    fake = ctypes.c_void_p(0x10000)
    bad_o = ctypes.c_void_p(0x10008)
    common = [fake] * 6 + [-5.0, None, 1, 1 << 20, 16, 128, 128, 64, None]
    assert L.kda_chunk_fwd_noalloc(*common, bad_o, None, fake, None, None) == 3
    assert L.kda_chunk_fwd_noalloc(*common, bad_o, None, fake, fake, None) == 3
