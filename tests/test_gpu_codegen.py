"""Generated kernels on the GPU: plans with codegen = 1 run their own
NVRTC-compiled kernel (stats.codegen) and equal the oracle bit for bit, on
both engines, ragged chunks, several channels, micro-batches and windows,
FIFO and direct transport, repeated executions and in-place calls; the step
timeline of an instrumented generated plan is filled like the library's."""
import numpy as np
import pytest

from gpu_helpers import assert_bitexact, empty_outputs, oracle_program, run_case, to_device, to_host

pytestmark = pytest.mark.gpu

F32, BF16, F16, I32 = 0, 1, 2, 3
DIST = {F32: "normal", BF16: "normal", F16: "uniform", I32: "int"}


@pytest.fixture(scope="module")
def ccl():
    import collective_communication_schedule_gb300 as m
    return m


CASES = [
    # kind, R, G, chunk elements, dtype, fuse, plan options
    (0, 8, 0, 3001, F32, True, dict(engine=1)),
    (0, 8, 0, 4096, BF16, "nochain", dict(engine=1, channels=2, slot_bytes=4096)),
    (0, 8, 0, 2053, F32, True, dict(channels=2, microbatches=3, slot_bytes=4096)),
    (3, 4, 2, 1000, F32, "nochain", dict(channels=2, microbatches=4, mb_window=2, fifo_slots=8, slot_bytes=2048,
                                          tb_alloc=1)),
    (2, 5, 0, 777, BF16, True, dict(engine=1, link_mode=0)),
    (1, 8, 0, 999, F16, False, dict(engine=1, channels=2)),
    (4, 8, 4, 500, I32, True, dict(link_mode=1, tb_alloc=2, tb_budget=8, channels=2)),
    (5, 6, 3, 640, F32, False, dict(microbatches=2, link_mode=1)),
    (0, 5, 0, 1500, I32, True, dict(mb_order=2, microbatches=3, link_mode=0)),
    (3, 4, 2, 2048, F32, True, dict(bulk=1, tile_bytes=4096, slot_bytes=8192)),
    # receives folded into their senders (two-destination steps)
    (1, 8, 0, 999, BF16, "nochain", dict(engine=1, link_mode=1, cluster=4)),
    (0, 8, 0, 2053, F32, "nochain", dict(link_mode=1, channels=2)),
    # copy chains folded too (two remote destinations in one step)
    (1, 8, 0, 999, BF16, "nochain", dict(engine=1, link_mode=1, cluster=4, fold=3)),
    (0, 8, 0, 2053, F32, "nochain", dict(link_mode=1, channels=2, fold=3)),
    (3, 8, 4, 1024, F32, "nochain", dict(link_mode=1, microbatches=4, mb_window=2, tb_alloc=1, fold=3)),
    (5, 6, 3, 640, F32, False, dict(microbatches=2, link_mode=1, fold=2)),
    # reduction chains folded (third operand, steps two ranks apart)
    (2, 8, 0, 1001, BF16, True, dict(engine=1, link_mode=1, cluster=4, fold=7)),
    (0, 8, 0, 2053, F16, "nochain", dict(link_mode=1, channels=2, fold=7)),
    (3, 8, 4, 1024, F32, "nochain", dict(link_mode=1, microbatches=4, mb_window=2, tb_alloc=1, fold=7)),
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_generated_kernel_bitexact(ccl, case):
    kind, R, G, ce, dtype, fuse, opts = CASES[case]
    got, want, plan = run_case(ccl, kind, R, G, ce, dtype, DIST[dtype], 50 + case, fuse=fuse, codegen=1, **opts)
    assert plan.stats().codegen == 1
    assert_bitexact(got, want)


@pytest.mark.parametrize("engine", [0, 1])
def test_generated_kernel_repeated_and_in_place(ccl, engine):
    """Five executions of one generated plan (sequence numbers continue
    across executions), then in place."""
    import torch
    import datagen
    import oracle
    R, ce = 8, 2000
    plan = ccl.Plan(ccl.Schedule.builtin(ccl.RING_ALLREDUCE, R), ce, F32, codegen=1, engine=engine,
                    slot_bytes=2048, fifo_slots=3, microbatches=2)
    ops, nch = oracle_program(0, R)
    for rep in range(5):
        host = datagen.rank_inputs(70 + rep, "normal", R, R * ce, F32)
        outs = empty_outputs(R, R * ce, F32)
        plan.execute(to_device(host, F32), outs)
        torch.cuda.synchronize()
        plan.status()
        want, _, _ = oracle.run(ops, R, nch, ce, F32, host)
        assert_bitexact(to_host(outs, F32), want)
    d = to_device(host, F32)
    plan.execute(d, d)
    torch.cuda.synchronize()
    plan.status()
    assert_bitexact(to_host(d, F32), want)


def test_generated_and_interpreted_kernels_have_the_same_timeline_shape(ccl):
    import torch
    import datagen
    R, ce = 8, 4096
    s = ccl.Schedule.builtin(ccl.RING_ALLREDUCE, R)
    ins = to_device(datagen.rank_inputs(1, "normal", R, R * ce, F32), F32)
    outs = empty_outputs(R, R * ce, F32)
    for codegen in (0, 1):
        plan = ccl.Plan(s, ce, F32, channels=2, instrument=1, codegen=codegen)
        plan.execute(ins, outs)
        torch.cuda.synchronize()
        plan.status()
        raw, tb = plan.timeline_raw()
        assert raw.shape[0] == plan.stats().nsteps
        assert np.all(raw[:, 4] >= raw[:, 0]) and np.all(raw[:, 0] > 0)


def test_debug_hook_is_refused_on_a_generated_plan(ccl):
    plan = ccl.Plan(ccl.Schedule.builtin(ccl.RING_ALLREDUCE, 4), 1024, F32, codegen=1)
    with pytest.raises(ccl.CclError) as e:
        plan.debug_drop_signal(0, 0)
    assert e.value.code == 5


def test_generated_sequential_kernel_on_clusters(ccl):
    got, want, plan = run_case(ccl, 0, 8, 0, 3001, F32, "normal", 77, codegen=1, engine=1, cluster=4, channels=2,
                               slot_bytes=4096)
    st = plan.stats()
    assert st.codegen == 1 and st.cluster == 4
    assert_bitexact(got, want)
