"""Oracle for chunk-oriented collective schedules.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this package.  It
shares no code with ``collective_communication_schedule_gb300`` and imports
nothing from it; the only module both sides use is ``datagen`` (seeded
inputs, none of the method's arithmetic).

Contents
--------
* ``ccl_oracle.c`` -- a plain program-order interpreter of copy/reduce chunk
  operations with its own bf16/f16 round-to-nearest-even (MSCCLang report,
  §III.1 "system design": chunk-oriented programs over input/output/scratch
  buffers with copy and reduce operations).
* ``schedules`` -- the oracle's own generators of the collective programs
  (ring AllReduce / AllGather / ReduceScatter, hierarchical AllReduce,
  two-phase AllToAll, AllToNext), written from the readings recorded in the
  design notes.
* ``explore`` -- an exhaustive interleaving explorer for tiny programs
  (determinism and absence of deadlock with bounded link FIFOs).

Parity status: every function here is pinned by ``tests/test_oracle_*.py``
(closed forms, library special cases, exhaustive rounding checks, brute
force on tiny inputs).  Special values follow IEEE 754 addition in the
buffer type (pinned against numpy / torch on every pair of special values);
the payload of a NaN result is not pinned.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

from . import schedules  # noqa: F401  (re-exported)

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ccl_oracle.c")
_SO = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

# codes shared with the op layout (restated, not imported)
F32, BF16, F16, I32 = 0, 1, 2, 3
IN, OUT, SCR = 0, 1, 2
COPY, REDUCE = 0, 1

NP_STORAGE = {F32: np.float32, BF16: np.uint16, F16: np.uint16, I32: np.int32}
ESIZE = {F32: 4, BF16: 2, F16: 2, I32: 4}
DTYPE_NAMES = {"f32": F32, "bf16": BF16, "f16": F16, "i32": I32}


def build(force: bool = False) -> str:
    """Compile the C interpreter into ``oracle/liboracle.so`` with gcc."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        cmd = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
               "-std=c11", "-Wall", "-o", _SO + ".tmp", _SRC]
        subprocess.run(cmd, check=True)
        os.replace(_SO + ".tmp", _SO)
    return _SO


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_SO)
            c_u16p = ctypes.POINTER(ctypes.c_uint16)
            c_f32p = ctypes.POINTER(ctypes.c_float)
            L.oracle_run.restype = ctypes.c_int
            L.oracle_run.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                     ctypes.c_int64, ctypes.c_int, ctypes.c_void_p,
                                     ctypes.POINTER(ctypes.c_int)]
            for name in ("oracle_f32_to_bf16_array", "oracle_f32_to_f16_array"):
                getattr(L, name).argtypes = [c_f32p, c_u16p, ctypes.c_int64]
            L.oracle_f16_to_f32_array.argtypes = [c_u16p, c_f32p, ctypes.c_int64]
            for name in ("oracle_add_bf16_array", "oracle_add_f16_array"):
                getattr(L, name).argtypes = [c_u16p, c_u16p, c_u16p, ctypes.c_int64]
            _lib = L
    return _lib


def _p(a, t):
    return a.ctypes.data_as(ctypes.POINTER(t))


def f32_to_bf16(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    y = np.empty(x.shape, np.uint16)
    lib().oracle_f32_to_bf16_array(_p(x, ctypes.c_float), _p(y, ctypes.c_uint16), x.size)
    return y


def f32_to_f16(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    y = np.empty(x.shape, np.uint16)
    lib().oracle_f32_to_f16_array(_p(x, ctypes.c_float), _p(y, ctypes.c_uint16), x.size)
    return y


def f16_to_f32(h: np.ndarray) -> np.ndarray:
    h = np.ascontiguousarray(h, dtype=np.uint16)
    y = np.empty(h.shape, np.float32)
    lib().oracle_f16_to_f32_array(_p(h, ctypes.c_uint16), _p(y, ctypes.c_float), h.size)
    return y


def bf16_to_f32(h: np.ndarray) -> np.ndarray:
    """bf16 is the upper half of a binary32 pattern: widening is a shift."""
    return (np.ascontiguousarray(h, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def add_bf16(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=np.uint16)
    b = np.ascontiguousarray(b, dtype=np.uint16)
    y = np.empty(a.shape, np.uint16)
    lib().oracle_add_bf16_array(_p(a, ctypes.c_uint16), _p(b, ctypes.c_uint16),
                                _p(y, ctypes.c_uint16), a.size)
    return y


def add_f16(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=np.uint16)
    b = np.ascontiguousarray(b, dtype=np.uint16)
    y = np.empty(a.shape, np.uint16)
    lib().oracle_add_f16_array(_p(a, ctypes.c_uint16), _p(b, ctypes.c_uint16),
                               _p(y, ctypes.c_uint16), a.size)
    return y


class OracleError(RuntimeError):
    pass


def run(ops: np.ndarray, nranks: int, nchunks, chunk_elems: int, dtype: int,
        inputs, sentinel: int = 0xA5):
    """Interpret ``ops`` in program order.

    ``inputs[r]`` is rank r's input buffer (storage dtype of ``dtype``) with
    ``nchunks[0] * chunk_elems`` elements.  Output and scratch buffers start
    filled with the ``sentinel`` byte.  Returns ``(outs, scratch)`` lists of
    numpy arrays.

    Because every operation maps chunk k' onto chunk k element by element
    (in-chunk offset preserved), running with ``chunk_elems = s`` on
    gathered columns of the inputs computes exactly those columns of the
    full result; ``run_sampled`` uses that.
    """
    ops = np.ascontiguousarray(np.asarray(ops, dtype=np.int32).reshape(-1, 8))
    st = NP_STORAGE[dtype]
    nchunks = [int(c) for c in nchunks]
    ins = []
    for r in range(nranks):
        a = np.ascontiguousarray(inputs[r], dtype=st).copy()
        if a.size != nchunks[IN] * chunk_elems:
            raise OracleError(f"rank {r} input has {a.size} elements, "
                              f"expected {nchunks[IN] * chunk_elems}")
        ins.append(a)
    outs = [np.full(nchunks[OUT] * chunk_elems * ESIZE[dtype], sentinel, np.uint8).view(st)
            for _ in range(nranks)]
    scr = [np.full(max(nchunks[SCR], 0) * chunk_elems * ESIZE[dtype], sentinel, np.uint8).view(st)
           for _ in range(nranks)]
    ptrs = (ctypes.c_void_p * (3 * nranks))()
    for r in range(nranks):
        ptrs[0 * nranks + r] = ins[r].ctypes.data
        ptrs[1 * nranks + r] = outs[r].ctypes.data
        ptrs[2 * nranks + r] = scr[r].ctypes.data if scr[r].size else None
    nch = (ctypes.c_int64 * 3)(*nchunks)
    bad = ctypes.c_int(-1)
    rc = lib().oracle_run(ops.ctypes.data, ops.shape[0], nranks, nch, chunk_elems, dtype,
                          ptrs, ctypes.byref(bad))
    if rc != 0:
        raise OracleError(f"oracle_run failed with status {rc} at op {bad.value}")
    # in-place writes into input buffers (allowed by the program model) are
    # visible to the caller through the returned copies
    return outs, scr, ins


def run_sampled(ops, nranks, nchunks, chunk_elems, dtype, inputs, offsets):
    """Exact result restricted to the in-chunk ``offsets`` of every chunk.

    Returns per-rank output arrays of shape ``(nchunks[OUT], len(offsets))``.
    """
    offsets = np.asarray(offsets, dtype=np.int64)
    cols = []
    for r in range(nranks):
        a = np.asarray(inputs[r]).reshape(nchunks[IN], chunk_elems)
        cols.append(np.ascontiguousarray(a[:, offsets]).reshape(-1))
    outs, _, _ = run(ops, nranks, nchunks, len(offsets), dtype, cols)
    return [o.reshape(nchunks[OUT], len(offsets)) for o in outs]
