"""Property test of the compiler (hypothesis, host only): random chunk
programs over 2-5 ranks, any mix of copies and reductions between any
buffers (inputs written too), compiled in each fusion mode and run by the
kind-by-kind interpreter of the fused instructions, equal the oracle's
program-order interpretation bit for bit, in integer and half precision;
and every one of them plans (timeline, threadblocks, FIFO simulation) in
every fusion mode and both transports."""
import numpy as np
import pytest

hyp = pytest.importorskip("hypothesis")
st = pytest.importorskip("hypothesis.strategies")

import datagen  # noqa: E402
import oracle  # noqa: E402

ccl = pytest.importorskip("collective_communication_schedule_gb300")
from test_compiler_planner import interpret_fused  # noqa: E402

F32, I32, F16 = 0, 3, 2


@st.composite
def programs(draw):
    R = draw(st.integers(2, 5))
    C = draw(st.integers(1, 5))
    n = draw(st.integers(1, 30))
    ops = []
    for _ in range(n):
        cnt = draw(st.integers(1, C))
        op = draw(st.integers(0, 1))
        sr, dr = draw(st.integers(0, R - 1)), draw(st.integers(0, R - 1))
        sb, db = draw(st.integers(0, 2)), draw(st.integers(0, 2))
        so, do = draw(st.integers(0, C - cnt)), draw(st.integers(0, C - cnt))
        if sr == dr and sb == db and so < do + cnt and do < so + cnt:
            continue                     # a range may not overlap itself
        ops.append((op, sr, sb, so, dr, db, do, cnt))
    hyp.assume(ops)
    return R, C, ops


@hyp.settings(max_examples=150, deadline=None)
@hyp.given(programs(), st.sampled_from([ccl.FUSE_NONE, ccl.FUSE_FULL, ccl.FUSE_NOCHAIN]), st.integers(0, 2**31))
def test_compiled_programs_equal_the_oracle(prog, fuse, seed):
    R, C, ops = prog
    nch = (C, C, C)
    s = ccl.Schedule.compile(ops, R, nch, fuse=fuse)
    # the unfused form always plans; the fused form does too (from a less
    # fused compilation of the same program when its own cannot be planned)
    for link_mode in (ccl.LINK_FIFO, ccl.LINK_DIRECT):
        ccl.Schedule.compile(ops, R, nch, fuse=ccl.FUSE_NONE).check(64, F32, link_mode=link_mode)
        s.check(64, F32, link_mode=link_mode)
    ce = 3
    for dtype, dist in ((I32, "int"), (F16, "normal")):
        ins = datagen.rank_inputs(seed % 1000, dist, R, C * ce, dtype)
        got = interpret_fused(s.instrs(), R, nch, ce, dtype, ins)
        want, _, _ = oracle.run(np.array(ops, dtype=np.int32), R, nch, ce, dtype, ins)
        for r in range(R):
            assert np.array_equal(got[r].view(np.uint8), want[r].view(np.uint8)), (r, dtype)
