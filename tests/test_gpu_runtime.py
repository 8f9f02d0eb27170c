"""GPU runtime behaviour: bounded waits, instrumentation, tuner, host-buffer
path, and full-size parity in the benchmark's launch configurations."""
import numpy as np
import pytest

from gpu_helpers import assert_bitexact, empty_outputs, oracle_program, run_case, to_device, to_host

pytestmark = pytest.mark.gpu

F32, BF16, F16, I32 = 0, 1, 2, 3


@pytest.fixture(scope="module")
def ccl():
    import collective_communication_schedule_gb300 as m
    return m


def test_lost_signal_times_out_and_device_stays_usable(ccl):
    """A plan patched to skip one flag post: the waiting threadblock gives up
    after 50 ms, the status reads CCL_ERR_TIMEOUT, and the GPU then runs a
    fresh plan correctly (host-made fault, no device fault)."""
    import torch
    import datagen
    s = ccl.Schedule.builtin(ccl.RING_ALLREDUCE, 4)
    plan = ccl.Plan(s, 1024, F32, timeout_ms=50)
    plan.debug_drop_signal(0, 0)
    ins = to_device(datagen.rank_inputs(0, "normal", 4, 4 * 1024, F32), F32)
    outs = empty_outputs(4, 4 * 1024, F32)
    plan.execute(ins, outs)
    torch.cuda.synchronize()
    with pytest.raises(ccl.CclError) as ei:
        plan.status()
    assert ei.value.code == 8
    assert "gave up waiting" in ei.value.detail
    got, want, _ = run_case(ccl, 0, 4, 0, 1024, F32, "normal", 0)
    assert_bitexact(got, want)


@pytest.mark.parametrize("engine", [0, 1])
def test_lost_counter_times_out_and_device_stays_usable(ccl, engine):
    """Direct copies signal dependency counters instead of FIFO flags: a
    threadblock of link-free copies that posts none of its counters makes its
    dependents give up after 50 ms (on the sequential engine the wait for a
    single counter is a loop of acquire loads); the GPU then runs a fresh
    plan.  Copy chains stay unfolded, so that the first all-gather copy has
    a dependent (the copy that forwards its chunk)."""
    import torch
    import datagen
    s = ccl.Schedule.builtin(ccl.RING_ALLREDUCE, 4, 0, ccl.FLAG_NOCHAIN_COPIES)
    plan = ccl.Plan(s, 1024, F32, timeout_ms=50, link_mode=ccl.LINK_DIRECT, tb_alloc=ccl.TB_CONNECTION,
                    engine=engine, fold=1)
    steps = plan.steps()
    by_tb = {}
    for k, st in enumerate(steps):
        by_tb.setdefault(int(st["tb"]), []).append(st)
    free = [tb for tb, lst in by_tb.items() if all(x["link_in"] < 0 and x["link_out"] < 0 for x in lst)]
    assert free, "the plan has a threadblock of direct copies"
    for i in range(len(by_tb[free[0]])):
        plan.debug_drop_signal(free[0], i)
    ins = to_device(datagen.rank_inputs(1, "normal", 4, 4 * 1024, F32), F32)
    outs = empty_outputs(4, 4 * 1024, F32)
    plan.execute(ins, outs)
    torch.cuda.synchronize()
    with pytest.raises(ccl.CclError) as ei:
        plan.status()
    assert ei.value.code == 8
    assert "gave up waiting" in ei.value.detail
    got, want, _ = run_case(ccl, 0, 4, 0, 1024, F32, "normal", 1, fuse="nochain", link_mode=ccl.LINK_DIRECT,
                            engine=engine)
    assert_bitexact(got, want)


def test_timeline_reports_idle_fractions(ccl):
    import torch
    import datagen
    s = ccl.Schedule.builtin(ccl.HIER_ALLREDUCE, 16, 8)
    plan = ccl.Plan(s, 65536, F32, channels=2, microbatches=4, instrument=1)
    ins = to_device(datagen.rank_inputs(2, "normal", 16, 16 * 65536, F32), F32)
    outs = empty_outputs(16, 16 * 65536, F32)
    plan.execute(ins, outs)
    torch.cuda.synchronize()
    plan.status()
    tl = plan.timeline()
    st = plan.stats()
    assert len(tl["idle"]) == st.nthreadblocks
    assert all(0.0 <= x <= 1.0 for x in tl["idle"])
    assert tl["mean_idle"] <= tl["max_idle"] + 1e-12 and tl["span_us"] > 0


def test_tuner_returns_a_configuration_that_runs(ccl):
    import torch
    import datagen
    import oracle
    R, ce = 8, 32768
    s = ccl.Schedule.builtin(ccl.RING_ALLREDUCE, R)
    host = datagen.rank_inputs(0, "uniform", R, R * ce, F32)
    ins = to_device(host, F32)
    outs = empty_outputs(R, R * ce, F32)
    best, rep = ccl.tune(s, ce, F32, ins, outs, max_rounds=1, reps=3)
    assert rep.probes >= 2 and rep.best_us > 0
    assert rep.best_us <= rep.default_us * 1.10 + 5.0
    plan = ccl.Plan(s, ce, F32, opts=best)
    outs = empty_outputs(R, R * ce, F32)
    plan.execute(ins, outs)
    torch.cuda.synchronize()
    plan.status()
    ops, nch = oracle_program(0, R)
    want, _, _ = oracle.run(ops, R, nch, ce, F32, host)
    assert_bitexact(to_host(outs, F32), want)


def test_execute_host_round_trip(ccl):
    import torch
    import datagen
    import oracle
    R, G, ce = 8, 4, 5000
    s = ccl.Schedule.builtin(ccl.ALLTOALL_2PHASE, R, G)
    plan = ccl.Plan(s, ce, F16, channels=2)
    host = datagen.rank_inputs(3, "uniform", R, R * ce, F16)
    h_in = [torch.from_numpy(a.view(np.int16)).pin_memory() for a in host]
    h_out = [torch.empty(R * ce, dtype=torch.int16).pin_memory() for _ in range(R)]
    d_in = [torch.empty(R * ce, dtype=torch.int16, device="cuda") for _ in range(R)]
    d_out = [torch.empty(R * ce, dtype=torch.int16, device="cuda") for _ in range(R)]
    plan.execute_host(h_in, h_out, d_in, d_out)
    torch.cuda.synchronize()
    plan.status()
    ops, nch = oracle_program(4, R, G)
    want, _, _ = oracle.run(ops, R, nch, ce, F16, host)
    assert_bitexact([t.numpy().view(np.uint16) for t in h_out], want)


def _bench_rows():
    import bench
    return bench.SUITE


@pytest.mark.parametrize("row", range(8))
def test_full_size_benchmark_configurations(ccl, row):
    """Every collective of the benchmark at its full size and plan options;
    the oracle computes 64 sampled in-chunk columns exactly, and the
    copy collectives are also compared in full."""
    import torch
    name, kind, R, G, dt, chunk_bytes, dist, seed, opts = _bench_rows()[row]
    ce = chunk_bytes // {0: 4, 1: 2, 2: 2, 3: 4}[dt]
    rng = np.random.default_rng(12345 + row)
    cols = np.unique(np.concatenate([[0, ce - 1], rng.integers(0, ce, 62)]))
    got, want, plan = run_case(ccl, kind, R, G, ce, dt, dist, seed, sampled=cols, **opts)
    assert_bitexact(got, want)
    del got, want, plan
    torch.cuda.empty_cache()


def test_plan_steps_match_the_timeline(ccl):
    """Step introspection lines up with the raw stamps: same count, threadblock
    boundaries, and every step posted no earlier than it started."""
    import torch
    import datagen
    s = ccl.Schedule.builtin(ccl.ALLTONEXT, 6, 3)
    plan = ccl.Plan(s, 4096, F32, channels=2, instrument=1)
    ins = to_device(datagen.rank_inputs(1, "normal", 6, 6 * 4096, F32), F32)
    outs = empty_outputs(6, 6 * 4096, F32)
    plan.execute(ins, outs)
    torch.cuda.synchronize()
    plan.status()
    steps = plan.steps()
    stamps, tb = plan.timeline_raw()
    assert len(steps) == plan.stats().nsteps == stamps.shape[0]
    for b in range(len(tb) - 1):
        assert all(st["tb"] == b for st in steps[tb[b]:tb[b + 1]])
    assert np.all(stamps[:, 4] >= stamps[:, 0])
    assert all(st["nelem"] >= 0 and st["kind"] in range(len(ccl.KIND_NAMES)) for st in steps)


def test_execute_host_async_pipelines_two_plans_and_reuses_buffers(ccl):
    """Two plans share copy-in / compute / copy-out streams; each runs twice
    on the same device buffers with new host inputs (the plan's events order
    the second round after the first)."""
    import torch
    import datagen
    import oracle
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    s_comp = torch.cuda.current_stream()
    cases = []
    for kind, R, G, dt, ce in [(0, 8, 0, F32, 8192), (4, 8, 4, F16, 4096)]:
        plan = ccl.Plan(ccl.Schedule.builtin(kind, R, G), ce, dt, channels=2)
        tdt = torch.float32 if dt == F32 else torch.int16
        d_in = [torch.empty(plan.in_elems, dtype=tdt, device="cuda") for _ in range(R)]
        d_out = [torch.empty(plan.out_elems, dtype=tdt, device="cuda") for _ in range(R)]
        cases.append((kind, R, G, dt, ce, plan, tdt, d_in, d_out))
    for rnd in range(2):
        results = []
        for kind, R, G, dt, ce, plan, tdt, d_in, d_out in cases:
            host = datagen.rank_inputs(40 + rnd, "uniform", R, plan.in_elems, dt)
            h_in = [torch.from_numpy(a.view(np.int16) if dt != F32 else a).pin_memory() for a in host]
            h_out = [torch.empty(plan.out_elems, dtype=tdt).pin_memory() for _ in range(R)]
            plan.execute_host_async(h_in, h_out, d_in, d_out, s_in, s_comp, s_out)
            # the pinned host tensors must outlive the copies torch cannot see
            results.append((kind, R, G, dt, ce, plan, host, h_out, h_in))
        s_out.synchronize()
        torch.cuda.synchronize()
        for kind, R, G, dt, ce, plan, host, h_out, _ in results:
            plan.status()
            ops, nch = oracle_program(kind, R, G)
            want, _, _ = oracle.run(ops, R, nch, ce, dt, host)
            got = [t.numpy().view(np.uint16) if dt != F32 else t.numpy() for t in h_out]
            assert_bitexact(got, want)


def test_lost_signal_on_a_cluster_times_out_and_device_stays_usable(ccl):
    """The same host-made fault on the sequential engine with clusters of
    four CTAs: every CTA of the waiting cluster gives up, the others skip
    their data through the same barriers once the status is recorded, the
    kernel ends and the status reads CCL_ERR_TIMEOUT."""
    import torch
    import datagen
    s = ccl.Schedule.builtin(ccl.RING_ALLREDUCE, 4)
    plan = ccl.Plan(s, 1024, F32, timeout_ms=50, engine=ccl.ENGINE_SEQUENTIAL, cluster=4)
    plan.debug_drop_signal(0, 0)
    ins = to_device(datagen.rank_inputs(0, "normal", 4, 4 * 1024, F32), F32)
    outs = empty_outputs(4, 4 * 1024, F32)
    plan.execute(ins, outs)
    torch.cuda.synchronize()
    with pytest.raises(ccl.CclError) as ei:
        plan.status()
    assert ei.value.code == 8
    got, want, _ = run_case(ccl, 0, 4, 0, 1024, F32, "normal", 0, engine=ccl.ENGINE_SEQUENTIAL, cluster=4)
    assert_bitexact(got, want)


def test_lost_consumed_flags_on_ll_sequential_time_out(ccl):
    """LL slots on the sequential engine carry their data flags in the
    lines, but a consumer still posts that it has read a slot: a threadblock
    that posts nothing leaves its producer waiting for a slot to come free
    (two-slot FIFOs, four slots per step), which gives up after 50 ms."""
    import torch
    import datagen
    s = ccl.Schedule.builtin(ccl.RING_ALLREDUCE, 4)
    plan = ccl.Plan(s, 4096, F32, timeout_ms=50, engine=ccl.ENGINE_SEQUENTIAL, protocol=ccl.PROTO_LL, cluster=2,
                    fifo_slots=2, slot_bytes=4096)
    n0 = sum(1 for st in plan.steps() if int(st["tb"]) == 0)
    for i in range(n0):
        plan.debug_drop_signal(0, i)
    ins = to_device(datagen.rank_inputs(2, "normal", 4, 4 * 4096, F32), F32)
    outs = empty_outputs(4, 4 * 4096, F32)
    plan.execute(ins, outs)
    torch.cuda.synchronize()
    with pytest.raises(ccl.CclError) as ei:
        plan.status()
    assert ei.value.code == 8
    got, want, _ = run_case(ccl, 0, 4, 0, 4096, F32, "normal", 2, engine=ccl.ENGINE_SEQUENTIAL, protocol=ccl.PROTO_LL,
                            cluster=2, fifo_slots=2, slot_bytes=4096)
    assert_bitexact(got, want)
