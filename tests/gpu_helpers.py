"""Shared helpers of the GPU tests: inputs from ``datagen``, expected values
from ``oracle`` only, device results from the C ABI through the binding."""
import numpy as np

import datagen
import oracle
from oracle import schedules as OS

KIND_TO_ORACLE = {
    0: ("ring_allreduce", lambda R, G, wrap: (R,)),
    1: ("ring_allgather", lambda R, G, wrap: (R,)),
    2: ("ring_reducescatter", lambda R, G, wrap: (R,)),
    3: ("hier_allreduce", lambda R, G, wrap: (G, R // G)),
    4: ("alltoall_two_phase", lambda R, G, wrap: (G, R // G)),
    5: ("alltonext", lambda R, G, wrap: (G, R // G, wrap)),
}

TORCH_STORAGE = {0: "float32", 1: "int16", 2: "int16", 3: "int32"}


def oracle_program(kind, R, G=0, wrap=False):
    name, args = KIND_TO_ORACLE[kind]
    return OS.BUILTINS[name](*args(R, G, wrap))


def to_device(arrs, dtype):
    import torch
    out = []
    for a in arrs:
        if dtype in (1, 2):
            t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16))
        else:
            t = torch.from_numpy(np.ascontiguousarray(a))
        out.append(t.cuda())
    return out


def empty_outputs(n_ranks, n_elems, dtype, fill=0xA5):
    import torch
    dt = getattr(torch, TORCH_STORAGE[dtype])
    outs = []
    for _ in range(n_ranks):
        t = torch.empty(n_elems, dtype=dt, device="cuda")
        t.view(torch.uint8).fill_(fill)
        outs.append(t)
    return outs


def to_host(ts, dtype):
    res = []
    for t in ts:
        a = t.cpu().numpy()
        if dtype in (1, 2):
            a = a.view(np.uint16)
        res.append(a)
    return res


def run_case(ccl, kind, R, G, ce, dtype, dist, seed, wrap=False, fuse=True, sampled=None, **opts):
    """Run the built-in collective on the GPU and the oracle on the CPU
    (``fuse``: True, False or "nochain" for copy receives left unchained).
    Returns (gpu_outputs, oracle_outputs, plan); with ``sampled`` (array of
    in-chunk offsets) the oracle computes only those columns and the GPU
    outputs are reduced to the same columns."""
    import torch
    flags = ccl.FLAG_WRAP if wrap else 0
    if fuse == "nochain":
        flags |= ccl.FLAG_NOCHAIN_COPIES
    elif not fuse:
        flags |= ccl.FLAG_NOFUSE
    sched = ccl.Schedule.builtin(kind, R, G, flags)
    plan = ccl.Plan(sched, ce, dtype, **opts)
    ops, nch = oracle_program(kind, R, G, wrap)
    assert tuple(nch[:2]) == tuple(plan.nchunks[:2])
    ins = datagen.rank_inputs(seed, dist, R, nch[0] * ce, dtype)
    d_in = to_device(ins, dtype)
    d_out = empty_outputs(R, nch[1] * ce, dtype)
    plan.execute(d_in, d_out)
    torch.cuda.synchronize()
    plan.status()
    got = to_host(d_out, dtype)
    if sampled is None:
        want, _, _ = oracle.run(ops, R, nch, ce, dtype, ins)
    else:
        want = oracle.run_sampled(ops, R, nch, ce, dtype, ins, sampled)
        got = [g.reshape(nch[1], ce)[:, sampled] for g in got]
    return got, want, plan


def assert_bitexact(got, want):
    for r, (g, w) in enumerate(zip(got, want)):
        g8 = np.ascontiguousarray(g).view(np.uint8)
        w8 = np.ascontiguousarray(w).view(np.uint8)
        if not np.array_equal(g8, w8):
            bad = np.nonzero(np.ascontiguousarray(g).reshape(-1) != np.ascontiguousarray(w).reshape(-1))[0]
            raise AssertionError(f"rank {r}: {bad.size} elements differ, first at {bad[:8]}: "
                                 f"got {np.ascontiguousarray(g).reshape(-1)[bad[:4]]} "
                                 f"want {np.ascontiguousarray(w).reshape(-1)[bad[:4]]}")


def nan_mask(a, dtype):
    """Elements of a host array (storage form of ``dtype``) that are NaN."""
    a = np.ascontiguousarray(a)
    if dtype == 0:
        return np.isnan(a.view(np.float32))
    if dtype == 1:
        u = a.view(np.uint16)
        return ((u & 0x7F80) == 0x7F80) & ((u & 0x7F) != 0)
    if dtype == 2:
        return np.isnan(a.view(np.float16))
    return np.zeros(a.shape, bool)


def assert_bitexact_but_nan(got, want, dtype):
    """Bit-exact, except that a NaN matches any NaN (payload and sign of a
    NaN are not pinned)."""
    for r, (g, w) in enumerate(zip(got, want)):
        gn, wn = nan_mask(g, dtype), nan_mask(w, dtype)
        if not np.array_equal(gn, wn):
            bad = np.nonzero(gn != wn)[0]
            raise AssertionError(f"rank {r}: NaN at different places, first at {bad[:8]}")
        g8 = np.ascontiguousarray(g)[~gn]
        w8 = np.ascontiguousarray(w)[~wn]
        if not np.array_equal(g8.view(np.uint8), w8.view(np.uint8)):
            bad = np.nonzero(g8 != w8)[0]
            raise AssertionError(f"rank {r}: {bad.size} non-NaN elements differ, first at {bad[:8]}")
