"""Uneven AllToAll (per-pair block sizes): oracle pins and the compiled
program on the host (no GPU).

* the oracle's program against the closed form written here with numpy
  slicing: out[d] = blocks from s = 0, 1, ... of in[s]'s block for d;
* every interleaving of tiny cases gives one result and never sticks;
* the compiled (fused and unfused) instruction lists, interpreted kind by
  kind, equal the oracle; byte count closed form; argument validation.
"""
import numpy as np
import pytest

import datagen
import oracle
from oracle import explore as E
from oracle import schedules as OS

ccl = pytest.importorskip("collective_communication_schedule_gb300")
from test_compiler_planner import interpret_fused  # noqa: E402

F32, BF16, I32 = 0, 1, 3


def closed_form(counts, ins, ce, nout):
    """out[d] = concat over s of in[s][block for d]; unwritten tail = 0xA5."""
    c = np.asarray(counts)
    R = c.shape[0]
    outs = []
    for d in range(R):
        o = np.full(nout * ce * ins[0].itemsize, 0xA5, np.uint8).view(ins[0].dtype)
        pos = 0
        for s in range(R):
            start = int(c[s, :d].sum()) * ce
            n = int(c[s, d]) * ce
            o[pos:pos + n] = ins[s][start:start + n]
            pos += n
        outs.append(o)
    return outs


COUNTS = [
    [[1]],
    [[0, 2], [3, 0]],
    [[1, 2, 0], [0, 1, 3], [2, 0, 1]],
    [[0, 0, 5, 0], [1, 1, 1, 1], [0, 4, 0, 0], [2, 0, 0, 3]],
]


@pytest.mark.parametrize("counts", COUNTS + ["skewed"])
@pytest.mark.parametrize("dtype", [F32, BF16, I32])
def test_oracle_equals_closed_form(counts, dtype):
    if counts == "skewed":
        counts = datagen.alltoallv_counts(5, 8, 24)
    ops, nch = OS.alltoallv(counts)
    R = len(counts)
    ce = 3
    dist = "int" if dtype == I32 else "normal"
    ins = datagen.rank_inputs(11, dist, R, nch[0] * ce, dtype)
    want = closed_form(counts, ins, ce, nch[1])
    got, _, _ = oracle.run(ops, R, nch, ce, dtype, ins)
    for r in range(R):
        assert np.array_equal(got[r].view(np.uint8), want[r].view(np.uint8)), f"rank {r}"


@pytest.mark.parametrize("counts", COUNTS[1:])
@pytest.mark.parametrize("K", [1, 2])
def test_every_interleaving_gives_one_result(counts, K):
    ops, nch = OS.alltoallv(counts)
    res = E.explore(ops, len(counts), nch, K=K)
    assert res["deadlocks"] == 0
    assert len(res["outputs"]) == 1


@pytest.mark.parametrize("counts", COUNTS + ["skewed"])
@pytest.mark.parametrize("fuse", [True, False])
def test_compiled_program_equals_oracle(counts, fuse):
    if counts == "skewed":
        counts = datagen.alltoallv_counts(6, 8, 16)
    s = ccl.Schedule.alltoallv(counts, 0 if fuse else ccl.FLAG_NOFUSE)
    ops, nch = OS.alltoallv(counts)
    assert tuple(s.info().nchunks) == tuple(nch)
    # same pairs, whatever the program order
    assert sorted(tuple(o) for o in s.ops()) == sorted(tuple(int(v) for v in o) for o in ops)
    R, ce = len(counts), 4
    ins = datagen.rank_inputs(2, "normal", R, nch[0] * ce, BF16)
    got = interpret_fused(s.instrs(), R, nch, ce, BF16, ins)
    want, _, _ = oracle.run(ops, R, nch, ce, BF16, ins)
    for r in range(R):
        assert np.array_equal(got[r].view(np.uint8), want[r].view(np.uint8)), f"rank {r}"


def test_bytes_closed_form():
    """A local block is one copy (2 bytes per element byte); a block between
    ranks is a send and a receive (4), or one direct copy (2)."""
    counts = datagen.alltoallv_counts(7, 8, 40)
    s = ccl.Schedule.alltoallv(counts)
    local = int(np.trace(counts))
    remote = int(np.sum(counts)) - local
    assert s.info().bytes_per_chunk_elem_x_esize == 2 * local + 4 * remote
    ce = 256
    st = s.check(ce, F32, link_mode=ccl.LINK_DIRECT)
    assert st.schedule_bytes == 2 * (local + remote) * ce * 4
    assert st.nlinks == 0
    # collective minimum: every input chunk read once, every output chunk written once
    assert st.min_bytes == 2 * int(np.sum(counts)) * ce * 4


@pytest.mark.parametrize("bad", [[[0, 0], [0, 0]], [[1, -1], [0, 1]], [[1, 2], [3]]])
def test_invalid_counts_are_rejected(bad):
    with pytest.raises((ccl.CclError, ValueError)):
        ccl.Schedule.alltoallv(bad)
