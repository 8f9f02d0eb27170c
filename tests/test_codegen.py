"""Kernels generated for single plans, on the host: the generator expresses
every built-in collective and every benchmark row as code (its replay of the
planner's steps passes), refuses what it cannot express, and the source
compiles for sm_103a with the run-time compiler (no GPU needed)."""
import pytest

ccl = pytest.importorskip("collective_communication_schedule_gb300")

F32, BF16, F16, I32 = 0, 1, 2, 3


@pytest.mark.parametrize("kind,R,G", [(0, 8, 0), (1, 8, 0), (2, 5, 0), (3, 16, 8), (4, 8, 4), (5, 6, 3)])
@pytest.mark.parametrize("opts", [dict(), dict(engine=1), dict(channels=3, microbatches=4, mb_window=2, fifo_slots=8),
                                  dict(link_mode=0, tb_alloc=1, microbatches=3), dict(mb_order=2, microbatches=5),
                                  dict(tb_alloc=2, channels=2, tb_budget=8)])
def test_every_builtin_has_a_generated_kernel(kind, R, G, opts):
    s = ccl.Schedule.builtin(kind, R, G)
    src, _ = s.codegen_source(1003, F32, **opts)
    assert "ccl_gen_kernel" in src and "gtb0" in src
    # nothing is read from the step, link or dependency tables
    assert "P.recs" not in src and "P.links" not in src and "P.deps" not in src


def test_every_benchmark_row_has_a_generated_kernel():
    import bench

    class A:
        only, scale = "", 1.0
    for name, kind, R, G, dt, cb, dist, seed, opts in bench.selected_suite(A):
        sched, popts = bench.schedule_and_opts(ccl, kind, R, G, opts)
        src, _ = sched.codegen_source(cb // bench.ESIZE[dt], dt, **popts)
        assert src.count("static __device__ __noinline__ void gtb") == sched.check(
            cb // bench.ESIZE[dt], dt, **popts).nthreadblocks, name


def test_generated_source_compiles_for_sm103a():
    s = ccl.Schedule.builtin(ccl.RING_ALLREDUCE, 4)
    for dtype in (F32, BF16):
        for engine in (0, 1):
            src, cubin = s.codegen_source(4096, dtype, compile=True, engine=engine, channels=2)
            assert cubin > 0
            # the kernel is built for the 512-thread limit unless asked otherwise
            assert "__launch_bounds__(512, 1)" in src
    src, cubin = s.codegen_source(4096, F32, compile=True, nthreads=1024)
    assert "__launch_bounds__(1024, 1)" in src and cubin > 0


def test_the_ll_protocol_is_refused():
    s = ccl.Schedule.builtin(ccl.RING_ALLREDUCE, 4)
    with pytest.raises(ccl.CclError) as e:
        s.codegen_source(4096, F32, protocol=1)
    assert e.value.code == 5


def test_codegen_option_round_trips_through_a_tune_table(tmp_path):
    r = ccl.TuneRow()
    r.chunk_elems = 64
    r.best = ccl.default_opts()
    r.best.codegen = 1
    ccl.write_tune_table([r], F32, tmp_path / "t.json")
    rows, _ = ccl.read_tune_table(tmp_path / "t.json")
    assert rows[0].best.codegen == 1
