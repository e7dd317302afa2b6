"""KDA oracle: TEST INFRASTRUCTURE ONLY.

Plain fp64 CPU implementations of Kimi Delta Attention used to check the CUDA
library.  Only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU
baseline leg may import this package; the product path never does, and this
package imports nothing from it.

* ``kda_ref.c`` - the sequential token-by-token recurrence (the definition),
  built into ``libkda_ref.so`` by :func:`build` and called through ctypes.
* ``chunk_np`` - an independent NumPy chunkwise form, used to pin the C code.

Functions take and return NumPy float64 arrays in the layouts described in
``kda_ref.c`` ([tokens, heads, dim] for per-token tensors, [n, heads, dk, dv]
for states).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_ref.c")
_LIB_PATH = os.path.join(_HERE, "libkda_ref.so")

GMIN = -5.0  # "Kimi K3 Technical Report - Open Frontier Intelligence", sec. 2.1.1


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile kda_ref.c (gcc, -O2, OpenMP when available) into a shared library."""
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src)):
        return out
    tmp = out + ".tmp%d" % os.getpid()
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", src, "-o", tmp, "-lm"]
    res = subprocess.run(base[:1] + ["-fopenmp"] + base[1:], capture_output=True, text=True)
    if res.returncode != 0:  # no OpenMP runtime: build single-threaded
        res = subprocess.run(base, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("oracle build failed:\n" + res.stderr)
    os.replace(tmp, out)
    return out


def _bind(path):
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    lib.kda_ref_prefill.restype = ctypes.c_int
    lib.kda_ref_prefill.argtypes = [P, P, P, P, P, P, ctypes.c_double, P, ctypes.c_int,
                                    ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                    P, P, P, P, P, ctypes.c_int]
    lib.kda_ref_decode_step.restype = ctypes.c_int
    lib.kda_ref_decode_step.argtypes = [P, P, P, P, P, P, ctypes.c_double, P, ctypes.c_int,
                                        ctypes.c_int, ctypes.c_int, ctypes.c_int, P]
    lib.kda_ref_gate.restype = None
    lib.kda_ref_gate.argtypes = [P, P, ctypes.c_double, ctypes.c_int64, ctypes.c_int,
                                 ctypes.c_int, P]
    lib.kda_ref_num_threads.restype = ctypes.c_int
    lib.kda_ref_num_threads.argtypes = []
    return lib


def _f64(x):
    return np.ascontiguousarray(x, dtype=np.float64)


def _ptr(a):
    return None if a is None else a.ctypes.data


def snapshot_offsets(lengths, chunk: int = 64):
    """Row offsets of each sequence's snapshots: prefix sums of floor(L/chunk)."""
    counts = [int(L) // chunk for L in lengths]
    return np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)


class Oracle:
    """The oracle's Python API bound to one compiled copy of kda_ref.c.

    The module-level functions use the copy built by :func:`build`; the
    oracle's own mutation tests bind deliberately broken copies the same way.
    """

    def __init__(self, lib_path=None):
        self._lib = _bind(lib_path or build())

    def num_threads(self) -> int:
        """OpenMP threads the oracle runs with (OMP_NUM_THREADS or all cores)."""
        return int(self._lib.kda_ref_num_threads())

    def gate(self, z, A, gmin: float = GMIN):
        """g = gmin * sigmoid(exp(A_h) * z) for z [T, H, dk] and A [H]."""
        z = _f64(z)
        A = _f64(A)
        T, H, dk = z.shape
        g = np.empty_like(z)
        self._lib.kda_ref_gate(_ptr(z), _ptr(A), float(gmin), T, H, dk, _ptr(g))
        return g

    def prefill(self, q, k, v, z, beta, A, gmin: float = GMIN, cu_seqlens=None, S0=None,
                chunk: int = 64, snapshots: bool = False, erase: bool = True):
        """Sequential KDA over packed sequences.

        q, k, z: [total, H, dk]; v: [total, H, dv]; beta: [total, H]; A: [H];
        cu_seqlens: [n_seq + 1] token offsets (None = one sequence);
        S0: [n_seq, H, dk, dv] or None (zero state).
        Returns dict(o, S_final, snaps, snap_offsets).
        """
        q, k, v, z, beta, A = (_f64(x) for x in (q, k, v, z, beta, A))
        total, H, dk = k.shape
        dv = v.shape[2]
        if cu_seqlens is None:
            cu_seqlens = np.array([0, total], np.int64)
        cu = np.ascontiguousarray(cu_seqlens, dtype=np.int64)
        n_seq = len(cu) - 1
        S0a = None if S0 is None else _f64(S0).reshape(n_seq, H, dk, dv)
        o = np.zeros((total, H, dv))
        S_final = np.zeros((n_seq, H, dk, dv))
        offs = snapshot_offsets(np.diff(cu), chunk)
        snaps = np.zeros((int(offs[-1]), H, dk, dv)) if snapshots else None
        rc = self._lib.kda_ref_prefill(_ptr(q), _ptr(k), _ptr(v), _ptr(z), _ptr(beta), _ptr(A),
                                       float(gmin), _ptr(cu), n_seq, H, dk, dv, int(chunk),
                                       _ptr(S0a), _ptr(o), _ptr(S_final), _ptr(snaps),
                                       _ptr(offs), 1 if erase else 0)
        if rc != 0:
            raise ValueError("kda_ref_prefill rejected its arguments")
        return {"o": o, "S_final": S_final, "snaps": snaps, "snap_offsets": offs}

    def decode_step(self, q, k, v, z, beta, A, state, gmin: float = GMIN):
        """One decode step; ``state`` [n, H, dk, dv] (float64, C order) is
        updated in place.  q, k, z: [n, H, dk]; v: [n, H, dv]; beta: [n, H].
        Returns o [n, H, dv]."""
        q, k, v, z, beta, A = (_f64(x) for x in (q, k, v, z, beta, A))
        if state.dtype != np.float64 or not state.flags["C_CONTIGUOUS"]:
            raise TypeError("state must be a C-contiguous float64 array")
        n, H, dk = k.shape
        dv = v.shape[2]
        o = np.zeros((n, H, dv))
        rc = self._lib.kda_ref_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(z), _ptr(beta),
                                           _ptr(A), float(gmin), _ptr(state), n, H, dk, dv,
                                           _ptr(o))
        if rc != 0:
            raise ValueError("kda_ref_decode_step rejected its arguments")
        return o


_default = None


def _oracle():
    global _default
    if _default is None:
        _default = Oracle()
    return _default


def num_threads() -> int:
    return _oracle().num_threads()


def gate(z, A, gmin: float = GMIN):
    return _oracle().gate(z, A, gmin)


def prefill(*args, **kw):
    return _oracle().prefill(*args, **kw)


def decode_step(*args, **kw):
    return _oracle().decode_step(*args, **kw)


num_threads.__doc__ = Oracle.num_threads.__doc__
gate.__doc__ = Oracle.gate.__doc__
prefill.__doc__ = Oracle.prefill.__doc__
decode_step.__doc__ = Oracle.decode_step.__doc__


if __name__ == "__main__":  # python -m oracle  -> build only
    print(build(force="--force" in sys.argv))
