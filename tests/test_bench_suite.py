"""The benchmark suite's plans, checked on the host (no GPU).

Every row of the suite plans with its own options; the ring rows' schedule
bytes equal the closed form of a ring AllReduce whose all-gather hops are
direct copies; every plan fits the co-residency limit of the executor's
cooperative launch; the kernel each row launches is the one named in the
benchmark line.
"""
import pytest

ccl = pytest.importorskip("collective_communication_schedule_gb300")
bench = pytest.importorskip("bench")

MiB = 1 << 20


def _plan(row):
    name, kind, R, G, dt, cb, dist, seed, opts = row
    s, po = bench.schedule_and_opts(ccl, kind, R, G, opts)
    return s, s.check(cb // bench.ESIZE[dt], dt, **po), po


@pytest.mark.parametrize("row", bench.SUITE, ids=[r[0] for r in bench.SUITE])
def test_every_row_plans_within_two_ctas_per_sm(row):
    s, st, po = _plan(row)
    assert 0 < st.nthreadblocks <= 2 * 152
    assert st.schedule_bytes >= st.min_bytes > 0
    assert st.engine == po.get("engine", 0)
    maxt = 512 if st.nthreads <= 512 else 1024
    assert bench.kernel_name(st) == (f"ccl_exec_seq_kernel<{maxt}>" if st.engine == 1
                                     else f"ccl_exec_kernel<simple, {maxt}>")


@pytest.mark.parametrize("name", ["ring_bf16", "ring_f32", "ar_1m"])
def test_ring_rows_match_the_closed_form(name):
    """Ring AllReduce over R ranks of N bytes each: R N (6 - 4/R) schedule
    bytes fully fused through FIFOs; leaving the R - 2 middle all-gather hops
    of every chunk unchained and direct saves one byte per element byte on
    each of them, N (R - 2) in all; and the first all-gather hop of every
    chunk -- the recv-reduce-copy-send that completes it and the plain
    receive it feeds -- writes the next rank's output directly, saving the
    receive's 2 bytes per element byte: 2 N in all.  With every fold
    (7), per rank and chunk of cb bytes: the reduce-scatter's R steps (3R
    units) pair up into floor(R/2) steps that read the next rank's input
    themselves (2 units less each); the receive the completing step feeds
    is folded into it; the R - 2 middle all-gather hops run two at a time (3
    per pair, 2 for an odd one out), or three (4 per triple) with fold bit
    3."""
    row = [r for r in bench.SUITE if r[0] == name][0]
    _, kind, R, G, dt, cb, dist, seed, opts = row
    assert opts.get("fuse") == "nochain" and opts.get("link_mode") == 1
    N = R * cb                       # R chunks of cb bytes per rank
    _, st, _ = _plan(row)
    fold = opts.get("fold", bench.DEFAULT_FOLD)
    assert fold & 7 == 7
    k = R - 2    # all-gather copies: pairs (3 each), or triples (4 each) with bit 3
    chain = 4 * (k // 3) + (0, 2, 3)[k % 3] if fold & 8 else 3 * (k // 2) + 2 * (k % 2)
    units = 3 * R - 2 * (R // 2) + chain
    assert st.schedule_bytes == R * units * cb
    assert st.min_bytes == 2 * R * N


def test_small_rows_run_sequential_and_large_rows_pipelined():
    engines = {r[0]: r[8].get("engine", 0) for r in bench.SUITE}
    assert {n for n, e in engines.items() if e == 1} == {"ag_3m", "rs_3m", "ar_1m"}


def test_hier_allgather_benchmark_plans_fit():
    """The --hier-allgather runs: the hierarchical program and the flat ring,
    unfused with direct copies, plan within the co-residency limit at the
    benchmark's size and move the same bytes: every one of the R x R output
    chunks is written once by one copy that reads one chunk (2 R^2 chunks),
    against the collective minimum of R input and R^2 output chunks (copy
    chains not folded).  With copy chains folded both move fewer bytes, as
    many as the oracle counts for their programs."""
    from oracle import bytes as OB
    from oracle import schedules as OS
    G, ng = 8, 2
    R, ce = G * ng, 2 * MiB
    ops, nch = bench.hier_allgather_program(G, ng)
    hier = ccl.Schedule.compile(ops, R, nch, fuse=False)
    flat = ccl.Schedule.builtin(ccl.RING_ALLGATHER, R, 0, ccl.FLAG_NOFUSE)
    for s, prog in ((hier, ops), (flat, OS.ring_allgather(R)[0])):
        for o in (dict(channels=8, link_mode=1), dict(channels=8, link_mode=1, tb_alloc=2, tb_budget=304)):
            st = s.check(ce, 1, fold=1, **o)
            assert st.nthreadblocks <= 2 * 152
            assert st.schedule_bytes == 2 * R * R * ce * 2
            assert st.min_bytes == (R + R * R) * ce * 2
            folded = s.check(ce, 1, fold=3, **o)
            assert folded.nthreadblocks <= 2 * 152
            assert folded.schedule_bytes < st.schedule_bytes
            assert folded.schedule_bytes == OB.schedule_bytes(prog, R, nch, ce, 1, "none", True, 3)


@pytest.mark.parametrize("kind", [1, 2])
def test_committed_sweep_tables_plan_on_their_schedules(kind):
    """Every row of a committed tuning table plans, at its size and at
    channels 1-4, on the schedule the sweep runs it with (the AllGather's
    copy receives unchained), and the tables cover every sweep size."""
    import os
    name = {1: "ring_allgather", 2: "ring_reducescatter"}[kind]
    rows, dt = ccl.read_tune_table(os.path.join(bench.TABLE_DIR, f"{name}_r8_bf16.json"))
    R = 8
    sizes = [kib * 1024 // 2 // R for kib in bench.SWEEP_KIB]
    assert sorted(r.chunk_elems for r in rows) == sizes and dt == 1
    s = bench.sweep_schedule(ccl, kind, R)
    for ce in sizes:
        base = ccl.lookup_tune_table(rows, ce)
        for ch in (1, 2, 3, 4):
            o = ccl.PlanOpts.from_buffer_copy(base)
            o.channels = ch
            st = s.check(ce, 1, opts=o)
            assert st.nthreadblocks <= 2 * 152
