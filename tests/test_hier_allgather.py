"""Hierarchical AllGather (in-group, cross-group, in-group; HetCCL summary,
"hierarchical algorithm design and pipelined execution") on the host.

* the oracle's program against the AllGather closed form (concatenation),
  for several group shapes and dtypes;
* every interleaving of a tiny case gives one result and never sticks;
* the benchmark's own user program, written independently of the oracle's,
  compiled (fused, unfused, no copy chaining) and interpreted kind by kind,
  equals the oracle; every block crosses into each other group exactly once.
"""
import numpy as np
import pytest

import datagen
import oracle
from oracle import explore as E
from oracle import schedules as OS

ccl = pytest.importorskip("collective_communication_schedule_gb300")
bench = pytest.importorskip("bench")
from test_compiler_planner import interpret_fused  # noqa: E402

F32, BF16, F16, I32 = 0, 1, 2, 3
SHAPES = [(2, 2), (4, 2), (3, 3), (8, 2), (2, 4)]


@pytest.mark.parametrize("G,ng", SHAPES)
@pytest.mark.parametrize("dtype", [F32, BF16, I32])
def test_oracle_equals_concatenation(G, ng, dtype):
    ops, nch = OS.hier_allgather(G, ng)
    R, ce = G * ng, 7
    ins = datagen.rank_inputs(3, "int" if dtype == I32 else "normal", R, nch[0] * ce, dtype)
    got, _, _ = oracle.run(ops, R, nch, ce, dtype, ins)
    want = np.concatenate(ins)
    for r in range(R):
        assert np.array_equal(got[r].view(np.uint8), want.view(np.uint8)), f"rank {r}"


@pytest.mark.parametrize("K", [1, 2])
def test_every_interleaving_gives_one_result(K):
    ops, nch = OS.hier_allgather(2, 2)
    res = E.explore(ops, 4, nch, K=K)
    assert res["deadlocks"] == 0
    assert len(res["outputs"]) == 1


@pytest.mark.parametrize("G,ng", SHAPES)
@pytest.mark.parametrize("fuse", [ccl.FUSE_FULL, ccl.FUSE_NONE, ccl.FUSE_NOCHAIN])
def test_user_program_compiles_to_the_oracle_result(G, ng, fuse):
    ops, nch = bench.hier_allgather_program(G, ng)
    R, ce = G * ng, 5
    s = ccl.Schedule.compile(ops, R, nch, fuse=fuse)
    ref_ops, ref_nch = OS.hier_allgather(G, ng)
    assert tuple(ref_nch) == tuple(nch)
    ins = datagen.rank_inputs(9, "normal", R, nch[0] * ce, F16)
    got = interpret_fused(s.instrs(), R, nch, ce, F16, ins)
    want, _, _ = oracle.run(ref_ops, R, nch, ce, F16, ins)
    for r in range(R):
        assert np.array_equal(got[r].view(np.uint8), want[r].view(np.uint8)), f"rank {r}"


@pytest.mark.parametrize("G,ng", SHAPES)
def test_each_block_enters_every_other_group_once(G, ng):
    ops, _ = bench.hier_allgather_program(G, ng)
    cross = [o for o in ops if o[1] // G != o[4] // G]
    assert len(cross) == G * ng * (ng - 1)
    assert len({(o[6], o[4] // G) for o in cross}) == len(cross)   # (block, group) pairs distinct
    assert len(ops) == G * ng + G * ng * (ng - 1) + G * ng * ng * (G - 1)
