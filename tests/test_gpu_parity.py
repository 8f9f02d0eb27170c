"""GPU executor vs the oracle, bit for bit (fixed reduction order).

Sizes span several slots, channels and micro-batches, with ragged element
counts (unaligned chunk starts, element tails) as well as the aligned
workload shapes.  Every expected value comes from ``oracle``.
"""
import numpy as np
import pytest

from gpu_helpers import assert_bitexact, run_case

pytestmark = pytest.mark.gpu

F32, BF16, F16, I32 = 0, 1, 2, 3
DIST = {F32: "normal", BF16: "normal", F16: "uniform", I32: "int"}


@pytest.fixture(scope="module")
def ccl():
    import collective_communication_schedule_gb300 as m
    return m


# (kind, R, G)
BUILTINS = [(0, 8, 0), (1, 8, 0), (2, 8, 0), (3, 16, 8), (4, 32, 8), (5, 24, 8),
            (0, 3, 0), (2, 5, 0), (3, 4, 2), (4, 4, 2), (5, 6, 3)]


@pytest.mark.parametrize("kind,R,G", BUILTINS)
@pytest.mark.parametrize("dtype", [F32, BF16, F16, I32])
def test_builtin_small_bitexact(ccl, kind, R, G, dtype):
    got, want, _ = run_case(ccl, kind, R, G, 1000, dtype, DIST[dtype], 7)
    assert_bitexact(got, want)


@pytest.mark.parametrize("ce", [1, 7, 33, 4093])
@pytest.mark.parametrize("dtype", [BF16, F32])
def test_ragged_sizes(ccl, ce, dtype):
    """Chunk sizes that leave element tails and unaligned chunk starts."""
    for kind, R, G in [(0, 8, 0), (3, 4, 2), (5, 6, 3)]:
        got, want, _ = run_case(ccl, kind, R, G, ce, dtype, DIST[dtype], 11, channels=2)
        assert_bitexact(got, want)


@pytest.mark.parametrize("channels", [1, 2, 3, 4])
@pytest.mark.parametrize("mb", [0, 1, 5])
def test_channels_and_microbatches_do_not_change_bits(ccl, channels, mb):
    # many slots per piece: 64 KiB chunks, 16 KiB slots
    got, want, plan = run_case(ccl, 0, 8, 0, 16384, BF16, "normal", 1, channels=channels, microbatches=mb,
                               slot_bytes=16384, fifo_slots=4)
    assert_bitexact(got, want)
    assert plan.stats().channels == channels


@pytest.mark.parametrize("sched", [0, 1])
@pytest.mark.parametrize("alloc", [0, 1])
@pytest.mark.parametrize("order", [0, 1, 3])
def test_scheduler_allocation_order(ccl, sched, alloc, order):
    for kind, R, G in [(3, 16, 8), (4, 8, 4), (5, 12, 4)]:
        got, want, _ = run_case(ccl, kind, R, G, 2048, F32, "normal", 2, scheduler=sched, tb_alloc=alloc,
                                mb_order=order, microbatches=4, slot_bytes=4096)
        assert_bitexact(got, want)


def test_unfused_equals_fused(ccl):
    for kind, R, G in [(0, 8, 0), (2, 8, 0), (3, 16, 8), (5, 24, 8)]:
        got, want, _ = run_case(ccl, kind, R, G, 512, BF16, "normal", 3, fuse=False)
        assert_bitexact(got, want)


# fused through FIFOs the program needs round-robin task order with 4 slots
# (the HPDS order deadlocks below 16 slots; the planner rejects it)
@pytest.mark.parametrize("fuse,opts", [(True, dict(channels=2, scheduler=0)), (False, dict(channels=2, link_mode=1)),
                                       (False, dict(channels=3, link_mode=1, tb_alloc=2, tb_budget=24)),
                                       (True, dict(channels=2, engine=1, microbatches=2, scheduler=0))])
def test_hier_allgather_program_bitexact(ccl, fuse, opts):
    """The benchmark's hierarchical AllGather user program (16 ranks as 2
    groups of 8), compiled through ccl_schedule_compile, against the oracle's
    own program: ragged chunk (unaligned starts, element tail)."""
    import torch
    import bench
    import datagen
    import oracle
    from oracle import schedules as OS
    from gpu_helpers import to_device, empty_outputs, to_host
    G, ng, ce = 8, 2, 5001
    R = G * ng
    ops, nch = bench.hier_allgather_program(G, ng)
    plan = ccl.Plan(ccl.Schedule.compile(ops, R, nch, fuse=fuse), ce, BF16, slot_bytes=16384, **opts)
    ins = datagen.rank_inputs(5, "normal", R, ce, BF16)
    d_out = empty_outputs(R, R * ce, BF16)
    plan.execute(to_device(ins, BF16), d_out)
    torch.cuda.synchronize()
    plan.status()
    ref_ops, _ = OS.hier_allgather(G, ng)
    want, _, _ = oracle.run(ref_ops, R, nch, ce, BF16, ins)
    assert_bitexact(to_host(d_out, BF16), want)


@pytest.mark.parametrize("link_mode", [0, 1])
def test_sequential_engine_bitexact(ccl, link_mode):
    """The sequential engine (one step at a time, every thread moving data)
    on every built-in: ragged chunks, several slots per piece, micro-batches
    and windows, FIFO and direct transport, fused and unfused programs."""
    cases = [(0, 8, 0, 4099, F32, True), (0, 5, 0, 1000, BF16, "nochain"), (1, 8, 0, 3001, F16, True),
             (2, 8, 0, 777, BF16, True), (3, 16, 8, 2048, F32, "nochain"), (4, 8, 4, 1000, F16, True),
             (5, 24, 8, 1500, F32, False), (0, 8, 0, 1000, I32, True)]
    for kind, R, G, ce, dtype, fuse in cases:
        got, want, plan = run_case(ccl, kind, R, G, ce, dtype, DIST[dtype], 21, fuse=fuse, link_mode=link_mode,
                                   engine=ccl.ENGINE_SEQUENTIAL, channels=2, microbatches=3, slot_bytes=4096)
        assert plan.stats().engine == ccl.ENGINE_SEQUENTIAL
        assert_bitexact(got, want)


def test_sequential_engine_repeated_executions(ccl):
    """Flags and counters carry the execution number: five executions of one
    plan (slot indices wrap differently each time) stay bit-exact."""
    import torch
    import datagen
    import oracle
    from gpu_helpers import oracle_program, to_device, empty_outputs, to_host
    s = ccl.Schedule.builtin(0, 8, 0)
    plan = ccl.Plan(s, 3000, BF16, engine=ccl.ENGINE_SEQUENTIAL, slot_bytes=2048, fifo_slots=3, microbatches=2)
    ops, nch = oracle_program(0, 8, 0, False)
    for rep in range(5):
        ins = datagen.rank_inputs(30 + rep, "normal", 8, nch[0] * 3000, BF16)
        d_out = empty_outputs(8, nch[1] * 3000, BF16)
        plan.execute(to_device(ins, BF16), d_out)
        torch.cuda.synchronize()
        plan.status()
        want, _, _ = oracle.run(ops, 8, nch, 3000, BF16, ins)
        assert_bitexact(to_host(d_out, BF16), want)


@pytest.mark.parametrize("link_mode", [0, 1])
def test_nochain_copies_bitexact(ccl, link_mode):
    """Reductions fused, copy receives unchained: under direct transport every
    all-gather hop is a plain copy into the next rank's buffer."""
    for kind, R, G, dtype in [(0, 8, 0, BF16), (3, 16, 8, F32), (1, 8, 0, BF16), (5, 24, 8, F32), (0, 3, 0, F16)]:
        got, want, _ = run_case(ccl, kind, R, G, 1000, dtype, DIST[dtype], 8, fuse="nochain", link_mode=link_mode,
                                channels=2, microbatches=3, slot_bytes=4096, tb_alloc=2 if link_mode else 0)
        assert_bitexact(got, want)


def test_config0_ring_allreduce_fp32_and_int32(ccl):
    """R = 8, 262144 elements per rank (8 chunks of 32768), seed 0."""
    got, want, _ = run_case(ccl, 0, 8, 0, 32768, F32, "uniform", 0)
    assert_bitexact(got, want)
    got, want, _ = run_case(ccl, 0, 8, 0, 32768, I32, "int", 0)
    assert_bitexact(got, want)


@pytest.mark.parametrize("kbytes", [32, 64, 128, 256, 512, 1024, 2048, 3072])
@pytest.mark.parametrize("channels", [1, 2, 3, 4])
def test_config1_allgather_reducescatter_sweep(ccl, kbytes, channels):
    R = 8
    ce = kbytes * 1024 // 2 // R          # bf16 elements per chunk
    for kind in (1, 2):
        got, want, _ = run_case(ccl, kind, R, 0, ce, BF16, "normal", 1, channels=channels)
        assert_bitexact(got, want)


def test_alltonext_wrap_and_untouched_rank0(ccl):
    got, want, _ = run_case(ccl, 5, 12, 4, 300, F32, "normal", 4, wrap=True)
    assert_bitexact(got, want)
    got, want, _ = run_case(ccl, 5, 12, 4, 300, F32, "normal", 4, wrap=False)
    assert_bitexact(got, want)
    assert np.all(np.ascontiguousarray(got[0]).view(np.uint8) == 0xA5)


def test_repeated_executions_reuse_flags(ccl):
    """Sequence numbers continue across executions without a reset."""
    import torch
    import datagen
    import oracle
    from gpu_helpers import oracle_program, to_device, empty_outputs, to_host
    s = ccl.Schedule.builtin(0, 8, 0)
    plan = ccl.Plan(s, 4096, BF16, slot_bytes=2048, fifo_slots=3, channels=2)
    ops, nch = oracle_program(0, 8)
    for it in range(5):
        ins = datagen.rank_inputs(100 + it, "normal", 8, 8 * 4096, BF16)
        d_in = to_device(ins, BF16)
        d_out = empty_outputs(8, 8 * 4096, BF16)
        plan.execute(d_in, d_out)
        torch.cuda.synchronize()
        plan.status()
        want, _, _ = oracle.run(ops, 8, nch, 4096, BF16, ins)
        assert_bitexact(to_host(d_out, BF16), want)


@pytest.mark.parametrize("link_mode", [0, 1])
@pytest.mark.parametrize("bulk", [0, 1])
@pytest.mark.parametrize("kind,R,G", [(0, 8, 0), (1, 8, 0), (2, 5, 0), (3, 16, 8), (4, 32, 8), (5, 24, 8), (5, 6, 3)])
def test_transport_and_data_path_do_not_change_bits(ccl, kind, R, G, link_mode, bulk):
    """FIFO vs direct transport, register vs bulk (TMA) tiles, with a ragged
    chunk so unaligned tiles take the register path inside the same plan."""
    for ce, dtype in ((4096, BF16), (1003, F32)):
        got, want, _ = run_case(ccl, kind, R, G, ce, dtype, DIST[dtype], 21, link_mode=link_mode, bulk=bulk,
                                tile_bytes=4096, slot_bytes=8192)
        assert_bitexact(got, want)


@pytest.mark.parametrize("window", [1, 2, 3, 8])
@pytest.mark.parametrize("order", [1, 3])
def test_microbatch_windows_do_not_change_bits(ccl, window, order):
    """Micro-batches interleaved per instruction in windows of 1..8, with
    FIFOs deep enough for the window (pieces of one slot)."""
    for kind, R, G in [(3, 16, 8), (0, 8, 0), (5, 12, 4), (2, 5, 0)]:
        got, want, plan = run_case(ccl, kind, R, G, 4096, F32, "normal", 5, microbatches=8, mb_order=order,
                                   mb_window=window, fifo_slots=window + 1 if window > 1 else 4, slot_bytes=4096,
                                   tb_alloc=1, link_mode=0)
        assert_bitexact(got, want)
        assert plan.stats().mb_window in (window, 1)


@pytest.mark.parametrize("kind,R,G", BUILTINS)
@pytest.mark.parametrize("dtype", [F32, BF16, F16, I32])
def test_ll_protocol_bitexact(ccl, kind, R, G, dtype):
    """Inline-flag slots: chunks of a multiple of 16 bytes, several slots and
    channels, FIFO and direct transport."""
    for lm in (0, 1):
        got, want, plan = run_case(ccl, kind, R, G, 1024, dtype, DIST[dtype], 9, protocol=1, channels=2,
                                   slot_bytes=2048, link_mode=lm)
        assert_bitexact(got, want)
        assert plan.stats().protocol == 1


def test_ll_protocol_repeated_executions_and_windows(ccl):
    """Line flags follow the slot sequence numbers across executions; windows
    and micro-batches keep the bits."""
    import torch
    import datagen
    import oracle
    from gpu_helpers import oracle_program, to_device, empty_outputs, to_host
    s = ccl.Schedule.builtin(3, 16, 8)
    plan = ccl.Plan(s, 4096, F32, protocol=1, slot_bytes=4096, fifo_slots=8, microbatches=4, mb_window=2,
                    tb_alloc=1)
    ops, nch = oracle_program(3, 16, 8)
    for it in range(4):
        ins = datagen.rank_inputs(200 + it, "normal", 16, 16 * 4096, F32)
        d_out = empty_outputs(16, 16 * 4096, F32)
        plan.execute(to_device(ins, F32), d_out)
        torch.cuda.synchronize()
        plan.status()
        want, _, _ = oracle.run(ops, 16, nch, 4096, F32, ins)
        assert_bitexact(to_host(d_out, F32), want)


@pytest.mark.parametrize("kind,R,G", BUILTINS)
@pytest.mark.parametrize("dtype", [F32, BF16, F16, I32])
def test_ll_protocol_on_the_sequential_engine_bitexact(ccl, kind, R, G, dtype):
    """LL slots on the sequential engine (every thread polls the lines of its
    part of a slot): one CTA per program and clusters of 2 and 4, several
    slots per piece, two channels, FIFO and direct transport."""
    # the 32-rank AllToAll's 416 FIFO threadblocks fit on the device only
    # one CTA each: its clustered cases run direct copies, balanced
    big = R >= 32
    for lm, cluster in ((0, 0), (1, 2), (1, 4) if big else (0, 4)):
        extra = dict(tb_alloc=2, tb_budget=64) if big and cluster else {}
        got, want, plan = run_case(ccl, kind, R, G, 1024, dtype, DIST[dtype], 19, protocol=1, engine=1, channels=2,
                                   slot_bytes=2048, link_mode=lm, cluster=cluster, nthreads=128, **extra)
        assert_bitexact(got, want)
        st = plan.stats()
        assert (st.protocol, st.engine, st.cluster) == (1, 1, max(1, cluster))


@pytest.mark.parametrize("cluster", [0, 8])
def test_ll_sequential_repeated_executions_and_windows(ccl, cluster):
    """Line flags of the sequential engine follow the slot sequence numbers
    across executions, with micro-batch windows and FIFOs shorter than a
    link's slots per execution."""
    import torch
    import datagen
    import oracle
    from gpu_helpers import oracle_program, to_device, empty_outputs, to_host
    s = ccl.Schedule.builtin(0, 8)
    plan = ccl.Plan(s, 4096, BF16, protocol=1, engine=1, cluster=cluster, nthreads=256, slot_bytes=2048,
                    fifo_slots=3, microbatches=4, mb_window=2)
    ops, nch = oracle_program(0, 8)
    for it in range(5):
        ins = datagen.rank_inputs(300 + it, "normal", 8, 8 * 4096, BF16)
        d_out = empty_outputs(8, 8 * 4096, BF16)
        plan.execute(to_device(ins, BF16), d_out)
        torch.cuda.synchronize()
        plan.status()
        want, _, _ = oracle.run(ops, 8, nch, 4096, BF16, ins)
        assert_bitexact(to_host(d_out, BF16), want)


@pytest.mark.parametrize("engine,protocol,cluster", [(0, 0, 0), (0, 1, 0), (1, 0, 0), (1, 1, 0), (1, 1, 4), (1, 0, 8)])
@pytest.mark.parametrize("fifo_slots", [13, 14, 16])
def test_fifo_deeper_than_an_execution_repeated(ccl, engine, protocol, cluster, fifo_slots):
    """A FIFO that holds every slot a link carries in one execution (the
    8-rank fused ring sends 14 one-slot pieces per link at this size): no
    slot is reused inside an execution, so no consumer posts that it has
    read one and no producer waits for that -- the next execution, a later
    kernel, reuses the slots.  At 14 slots the FIFO is exactly one
    execution deep; at 13 the last piece reuses the first slot.  Six
    executions, bit-exact each time, then in place."""
    import torch
    import datagen
    import oracle
    from gpu_helpers import oracle_program, to_device, empty_outputs, to_host
    R, ce = 8, 4096
    plan = ccl.Plan(ccl.Schedule.builtin(0, R), ce, BF16, engine=engine, protocol=protocol, cluster=cluster,
                    nthreads=256, slot_bytes=ce * 2, fifo_slots=fifo_slots, channels=1)
    ops, nch = oracle_program(0, R)
    for it in range(6):
        ins = datagen.rank_inputs(400 + it, "normal", R, R * ce, BF16)
        d_out = empty_outputs(R, R * ce, BF16)
        plan.execute(to_device(ins, BF16), d_out)
        torch.cuda.synchronize()
        plan.status()
        want, _, _ = oracle.run(ops, R, nch, ce, BF16, ins)
        assert_bitexact(to_host(d_out, BF16), want)
    d = to_device(ins, BF16)
    plan.execute(d, d)
    torch.cuda.synchronize()
    plan.status()
    assert_bitexact(to_host(d, BF16), want)


@pytest.mark.parametrize("R,tokens,seed", [(4, 64, 1), (8, 96, 2), (32, 48, 3)])
@pytest.mark.parametrize("dtype", [F32, BF16, I32])
@pytest.mark.parametrize("link_mode", [0, 1])
def test_alltoallv_bitexact(ccl, R, tokens, seed, dtype, link_mode):
    """Skewed token routing (one chunk = one token's vector); outputs shorter
    than the longest keep their untouched tail."""
    import torch
    import datagen
    import oracle
    from oracle import schedules as OS
    from gpu_helpers import to_device, empty_outputs, to_host
    counts = datagen.alltoallv_counts(seed, R, tokens)
    ce = 96 if dtype == BF16 else 80
    s = ccl.Schedule.alltoallv(counts)
    plan = ccl.Plan(s, ce, dtype, channels=2, link_mode=link_mode, tb_alloc=1)
    ops, nch = OS.alltoallv(counts)
    ins = datagen.rank_inputs(seed, DIST[dtype], R, nch[0] * ce, dtype)
    d_out = empty_outputs(R, nch[1] * ce, dtype)
    plan.execute(to_device(ins, dtype), d_out)
    torch.cuda.synchronize()
    plan.status()
    want, _, _ = oracle.run(ops, R, nch, ce, dtype, ins)
    assert_bitexact(to_host(d_out, dtype), want)


@pytest.mark.parametrize("budget", [64, 256])
def test_balanced_allocation_bitexact(ccl, budget):
    """Link-free threadblocks merged by bin packing: uneven and two-phase
    AllToAll, AllToNext with unfused direct relays."""
    import torch
    import datagen
    import oracle
    from oracle import schedules as OS
    from gpu_helpers import to_device, empty_outputs, to_host
    counts = datagen.alltoallv_counts(4, 16, 64)
    s = ccl.Schedule.alltoallv(counts)
    plan = ccl.Plan(s, 128, BF16, channels=4, link_mode=1, tb_alloc=2, tb_budget=budget, channel_scaling=1)
    ops, nch = OS.alltoallv(counts)
    ins = datagen.rank_inputs(4, "normal", 16, nch[0] * 128, BF16)
    d_out = empty_outputs(16, nch[1] * 128, BF16)
    plan.execute(to_device(ins, BF16), d_out)
    torch.cuda.synchronize()
    plan.status()
    want, _, _ = oracle.run(ops, 16, nch, 128, BF16, ins)
    assert_bitexact(to_host(d_out, BF16), want)
    for kind, R, G, fuse in [(4, 32, 8, True), (5, 24, 8, False), (4, 8, 4, True)]:
        got, want, _ = run_case(ccl, kind, R, G, 1000, F32, "normal", 6, fuse=fuse, link_mode=1, tb_alloc=2,
                                tb_budget=budget, channels=2, microbatches=4)
        assert_bitexact(got, want)


@pytest.mark.parametrize("kind,R,G", [(0, 1, 0), (0, 2, 0), (1, 1, 0), (1, 2, 0), (2, 1, 0), (2, 2, 0),
                                      (3, 2, 1), (4, 2, 1), (5, 2, 1), (5, 2, 2)])
@pytest.mark.parametrize("dtype", [F32, BF16])
def test_trivial_rank_counts(ccl, kind, R, G, dtype):
    got, want, _ = run_case(ccl, kind, R, G, 777, dtype, DIST[dtype], 13)
    assert_bitexact(got, want)


@pytest.mark.parametrize("dtype", [F32, BF16, F16])
def test_two_rank_allreduce_equals_torch_add(ccl, dtype):
    """R = 2: every output element is one rounded addition, so the result is
    torch's own elementwise add of the two inputs, bit for bit."""
    import torch
    import datagen
    from gpu_helpers import to_device, empty_outputs
    tdt = {F32: torch.float32, BF16: torch.bfloat16, F16: torch.float16}[dtype]
    ce = 4096
    ins = datagen.rank_inputs(21, DIST[dtype], 2, 2 * ce, dtype)
    d_in = to_device(ins, dtype)
    d_out = empty_outputs(2, 2 * ce, dtype)
    plan = ccl.Plan(ccl.Schedule.builtin(ccl.RING_ALLREDUCE, 2), ce, dtype, channels=2)
    plan.execute(d_in, d_out)
    torch.cuda.synchronize()
    plan.status()
    ref = (d_in[0].view(tdt) + d_in[1].view(tdt)).view(d_in[0].dtype)
    for r in range(2):
        assert torch.equal(d_out[r], ref), f"rank {r}"


# A user program that writes input buffers: rank 0's input chunk 2 is
# written by a copy from rank 1 and a reduction from rank 2 (threadblocks of
# other ranks), then read by rank 0's threadblock for rank 3 and rank 1;
# rank 0 also overwrites its own input chunk 1 and sends it on; rank 3 copies
# its output back into its input and reduces that into rank 2.
WRITES_INPUTS = [(0, 1, 0, 0, 0, 0, 2, 1), (1, 2, 0, 1, 0, 0, 2, 1), (0, 0, 0, 2, 3, 1, 0, 1),
                 (1, 0, 0, 2, 1, 1, 1, 1), (0, 0, 0, 0, 0, 0, 1, 1), (0, 0, 0, 1, 2, 1, 0, 1),
                 (0, 3, 1, 0, 3, 0, 0, 1), (1, 3, 0, 0, 2, 1, 1, 1), (1, 1, 0, 2, 3, 1, 1, 1)]


@pytest.mark.parametrize("fuse", [True, False, 2])
@pytest.mark.parametrize("opts", [dict(link_mode=0), dict(link_mode=1), dict(link_mode=1, bulk=1, tile_bytes=4096),
                                  dict(link_mode=0, engine=1), dict(link_mode=1, tb_alloc=2, channels=3)])
def test_program_that_writes_inputs_bitexact(ccl, fuse, opts):
    """Inputs written during the execution by other ranks' threadblocks and
    read afterwards on third ranks: the reads see the written values (no
    streaming load of a stale line, bulk copies ordered after the writes);
    outputs and the written inputs equal the oracle's."""
    import torch
    import datagen
    import oracle
    from gpu_helpers import to_device, empty_outputs, to_host
    R, nch, ce = 4, (3, 2, 1), 6007
    ops = np.array(WRITES_INPUTS, np.int32)
    plan = ccl.Plan(ccl.Schedule.compile(WRITES_INPUTS, R, nch, fuse=fuse), ce, F32, slot_bytes=8192,
                    **dict(dict(channels=2), **opts))
    for rep in range(2):
        ins = datagen.rank_inputs(40 + rep, "normal", R, nch[0] * ce, F32)
        d_in = to_device(ins, F32)
        d_out = empty_outputs(R, nch[1] * ce, F32)
        plan.execute(d_in, d_out)
        torch.cuda.synchronize()
        plan.status()
        want_out, _, want_in = oracle.run(ops, R, nch, ce, F32, ins)
        assert_bitexact(to_host(d_out, F32), want_out)
        assert_bitexact(to_host(d_in, F32), want_in)


@pytest.mark.parametrize("opts", [dict(), dict(channels=3, microbatches=2), dict(engine=1), dict(engine=1, cluster=4),
                                  dict(tb_alloc=2, channels=2), dict(bulk=1, tile_bytes=4096)])
@pytest.mark.parametrize("dtype", [F32, BF16])
def test_allgather_with_folded_copy_send_bitexact(ccl, opts, dtype):
    """Ring AllGather, copy receives unchained, direct transport: each
    rank's first step writes its block into its own output and the next
    rank's in one pass (a copy-send with its receive folded in); ragged
    chunks."""
    import torch
    import datagen
    import oracle
    from gpu_helpers import oracle_program, to_device, empty_outputs, to_host
    R, ce = 8, 3001
    plan = ccl.Plan(ccl.Schedule.builtin(1, R, 0, ccl.FLAG_NOCHAIN_COPIES), ce, dtype, link_mode=1,
                    slot_bytes=4096, **opts)
    assert plan.stats().nlinks == 0
    assert any(st["kind"] == ccl.KIND_NAMES.index("copy2") for st in plan.steps())
    ops, nch = oracle_program(1, R)
    ins = datagen.rank_inputs(71, DIST[dtype], R, ce, dtype)
    d_out = empty_outputs(R, R * ce, dtype)
    plan.execute(to_device(ins, dtype), d_out)
    torch.cuda.synchronize()
    plan.status()
    want, _, _ = oracle.run(ops, R, nch, ce, dtype, ins)
    assert_bitexact(to_host(d_out, dtype), want)


@pytest.mark.parametrize("R", [2, 5, 8])
@pytest.mark.parametrize("opts", [dict(), dict(channels=3, microbatches=2), dict(engine=1, cluster=4),
                                  dict(protocol=1), dict(engine=1, protocol=1), dict(bulk=1, tile_bytes=4096)])
def test_allreduce_with_folded_reduce_copy_send_bitexact(ccl, R, opts):
    """Ring AllReduce, copy receives unchained, direct transport: the step
    that completes a chunk (receive, reduce, copy to the own output) also
    writes the next rank's output, whose receive is folded away; ragged
    chunks, bf16, then in place."""
    import torch
    import datagen
    import oracle
    from gpu_helpers import oracle_program, to_device, empty_outputs, to_host
    ce = 4096 if opts.get("protocol") else 3001
    plan = ccl.Plan(ccl.Schedule.builtin(0, R, 0, ccl.FLAG_NOCHAIN_COPIES), ce, BF16, link_mode=1,
                    slot_bytes=4096, **opts)
    assert any(st["kind"] == ccl.KIND_NAMES.index("rrc2") for st in plan.steps())
    ops, nch = oracle_program(0, R)
    ins = datagen.rank_inputs(73, "normal", R, R * ce, BF16)
    d_out = empty_outputs(R, R * ce, BF16)
    plan.execute(to_device(ins, BF16), d_out)
    torch.cuda.synchronize()
    plan.status()
    want, _, _ = oracle.run(ops, R, nch, ce, BF16, ins)
    assert_bitexact(to_host(d_out, BF16), want)
    d = to_device(ins, BF16)
    plan.execute(d, d)
    torch.cuda.synchronize()
    plan.status()
    assert_bitexact(to_host(d, BF16), want)


CHAIN_OPTS = [dict(), dict(channels=3, microbatches=2), dict(engine=1), dict(engine=1, cluster=4),
              dict(protocol=1), dict(engine=1, protocol=1), dict(tb_alloc=2, channels=2),
              dict(bulk=1, tile_bytes=4096), dict(microbatches=4, mb_window=2, tb_alloc=1)]


@pytest.mark.parametrize("opts", CHAIN_OPTS)
@pytest.mark.parametrize("kind,R,G,fuse,dtype", [(1, 8, 0, "nochain", BF16), (1, 5, 0, "nochain", F32),
                                                 (0, 8, 0, "nochain", BF16), (0, 4, 0, "nochain", F32),
                                                 (3, 8, 4, "nochain", F32), (5, 6, 3, False, F32)])
@pytest.mark.parametrize("fold", [2, 3, 10, 15])
def test_copy_chains_folded_bitexact(ccl, opts, kind, R, G, fuse, dtype, fold):
    """Direct transport with copy chains folded: a copy that sends on what
    another direct copy delivered is written by that copy's pass (two
    remote destinations in one step) -- ring AllGather and AllReduce
    all-gather hops, the hierarchical AllReduce's in-group all-gather, the
    AllToNext relays; every engine, protocol and allocation; ragged chunks
    (LL: 16-byte multiples); then in place where the collective allows."""
    import torch
    import datagen
    import oracle
    from gpu_helpers import oracle_program, to_device, empty_outputs, to_host
    ll = opts.get("protocol") == 1
    ce = 4096 if ll else 3001
    flags = ccl.FLAG_NOCHAIN_COPIES if fuse == "nochain" else ccl.FLAG_NOFUSE
    sched = ccl.Schedule.builtin(kind, R, G, flags)
    plan = ccl.Plan(sched, ce, dtype, link_mode=1, slot_bytes=4096, fold=fold, **opts)
    multi = {ccl.KIND_NAMES.index("copy2"), ccl.KIND_NAMES.index("copy3")}
    assert any(st["kind"] in multi for st in plan.steps())
    assert plan.stats().schedule_bytes < sched.check(ce, dtype, link_mode=1, slot_bytes=4096, fold=fold & 1,
                                                     **opts).schedule_bytes
    ops, nch = oracle_program(kind, R, G)
    nin, nout = nch[0] * ce, nch[1] * ce
    ins = datagen.rank_inputs(79 + kind, DIST[dtype], R, nin, dtype)
    d_out = empty_outputs(R, nout, dtype)
    plan.execute(to_device(ins, dtype), d_out)
    torch.cuda.synchronize()
    plan.status()
    want, _, _ = oracle.run(ops, R, nch, ce, dtype, ins)
    assert_bitexact(to_host(d_out, dtype), want)
    if kind == 0:
        d = to_device(ins, dtype)
        plan.execute(d, d)
        torch.cuda.synchronize()
        plan.status()
        assert_bitexact(to_host(d, dtype), want)


REDUCE_OPTS = [dict(), dict(channels=3, microbatches=2), dict(engine=1), dict(engine=1, cluster=4),
               dict(tb_alloc=2, channels=2), dict(bulk=1, tile_bytes=4096),
               dict(microbatches=4, mb_window=2, tb_alloc=1), dict(protocol=1)]


@pytest.mark.parametrize("opts", REDUCE_OPTS)
@pytest.mark.parametrize("kind,R,G,fuse", [(2, 8, 0, True), (2, 5, 0, True), (2, 2, 0, True), (0, 8, 0, "nochain"),
                                           (0, 5, 0, "nochain"), (0, 2, 0, "nochain"), (0, 8, 0, True),
                                           (3, 16, 8, "nochain"), (3, 8, 4, True)])
@pytest.mark.parametrize("dtype", [F32, BF16, F16, I32])
def test_reduction_chains_folded_bitexact(ccl, opts, kind, R, G, fuse, dtype):
    """Direct transport with every fold on (7): consecutive steps of a
    reduction chain run as one step that reads the next rank's local
    operand itself and adds it after its own sum -- ReduceScatter, ring
    AllReduce (even and odd R, the completing step in a pair or alone), the
    hierarchical AllReduce -- in every dtype (bf16 / f16 would show any
    change of the summation order), on both engines, clusters, channels and
    micro-batches, packing, the bulk path and windows; with the LL protocol
    nothing folds and the result is the same.  Ragged chunks (LL: 16-byte
    multiples); the AllReduce rows then in place."""
    import torch
    import datagen
    import oracle
    from gpu_helpers import oracle_program, to_device, empty_outputs, to_host
    ll = opts.get("protocol") == 1
    ce = 4096 if ll else 3001
    flags = ccl.FLAG_NOCHAIN_COPIES if fuse == "nochain" else 0
    sched = ccl.Schedule.builtin(kind, R, G, flags)
    plan = ccl.Plan(sched, ce, dtype, link_mode=1, slot_bytes=4096, fold=7, **opts)
    # (a send folded into the recv-reduce-copy it feeds is a reduce)
    three = {ccl.KIND_NAMES.index(k) for k in ("rrs3", "rrc3", "rrcs3", "rsend", "rcsend", "reduce", "rrc3d",
                                                 "reduce2")}
    assert any(st["kind"] in three for st in plan.steps()) == (not ll)
    # (never more bytes; at R = 2 the AllReduce's pair costs what the
    # receive fold it replaces saved)
    assert plan.stats().schedule_bytes <= sched.check(ce, dtype, link_mode=1, slot_bytes=4096, fold=3,
                                                      **opts).schedule_bytes
    ops, nch = oracle_program(kind, R, G)
    ins = datagen.rank_inputs(83 + kind, DIST[dtype], R, nch[0] * ce, dtype)
    d_out = empty_outputs(R, nch[1] * ce, dtype)
    plan.execute(to_device(ins, dtype), d_out)
    torch.cuda.synchronize()
    plan.status()
    want, _, _ = oracle.run(ops, R, nch, ce, dtype, ins)
    assert_bitexact(to_host(d_out, dtype), want)
    if kind in (0, 3):
        d = to_device(ins, dtype)
        plan.execute(d, d)
        torch.cuda.synchronize()
        plan.status()
        assert_bitexact(to_host(d, dtype), want)


CHAIN_PROGRAM_OPTS = [dict(), dict(engine=1), dict(engine=1, cluster=4), dict(channels=2, microbatches=2),
                      dict(protocol=1), dict(bulk=1, tile_bytes=4096), dict(tb_alloc=2, channels=2),
                      dict(microbatches=4, mb_window=2, tb_alloc=1)]


@pytest.mark.parametrize("seed", range(8))
@pytest.mark.parametrize("shape", [(4, 4, 30), (6, 6, 40)])
@pytest.mark.parametrize("fuse", [True, "nochain", False])
@pytest.mark.parametrize("fold", [7, 15])
@pytest.mark.parametrize("opts", CHAIN_PROGRAM_OPTS)
def test_random_chain_programs_folded_bitexact(ccl, seed, shape, fuse, fold, opts):
    """Random chain-rich chunk programs over 4 and 6 ranks (copies and
    reductions handed on from rank to rank, into outputs and scratch),
    planned on direct transport with the copy-chain and reduction-chain
    folds on, run on the GPU on both engines, clusters, channels and
    micro-batches, LL, the bulk path, packing and windows: bit-exact against
    the oracle's program-order run in f32 and bf16 (bf16 shows any change of
    a chain's summation order)."""
    import torch
    import datagen
    import oracle
    from gpu_helpers import to_device, empty_outputs, to_host
    from test_compiler_planner import chain_program
    R, C, nops = shape
    ops, nch = chain_program(seed, R=R, C=C, nops=nops)
    ce = 4096 if opts.get("protocol") == 1 else 3001
    mode = {True: ccl.FUSE_FULL, "nochain": ccl.FUSE_NOCHAIN, False: ccl.FUSE_NONE}[fuse]
    sched = ccl.Schedule.compile(ops, R, nch, fuse=mode)
    for dtype in (F32, BF16):
        plan = ccl.Plan(sched, ce, dtype, link_mode=1, slot_bytes=4096, fold=fold, **opts)
        ins = datagen.rank_inputs(90 + seed, DIST[dtype], R, nch[0] * ce, dtype)
        d_out = empty_outputs(R, nch[1] * ce, dtype)
        plan.execute(to_device(ins, dtype), d_out)
        torch.cuda.synchronize()
        plan.status()
        want, _, _ = oracle.run(np.array(ops, np.int32), R, nch, ce, dtype, ins)
        assert_bitexact(to_host(d_out, dtype), want)


@pytest.mark.parametrize("seed", range(8))
@pytest.mark.parametrize("shape", [(4, 4, 30), (6, 6, 40)])
@pytest.mark.parametrize("fuse", [True, "nochain", False])
@pytest.mark.parametrize("opts", [dict(), dict(fifo_slots=2), dict(engine=1), dict(protocol=1),
                                  dict(channels=2, microbatches=2), dict(tb_alloc=1)])
def test_random_chain_programs_through_fifos_bitexact(ccl, seed, shape, fuse, opts):
    """The same random programs over FIFO links (a fused send holds its
    slot while the receiver works; two slots a link at the least): where
    the fused form's timeline or slot count cannot be met the plan is made
    from a less fused compilation, and the result stays bit-exact."""
    import torch
    import datagen
    import oracle
    from gpu_helpers import to_device, empty_outputs, to_host
    from test_compiler_planner import chain_program
    R, C, nops = shape
    ops, nch = chain_program(seed, R=R, C=C, nops=nops)
    ce = 4096 if opts.get("protocol") == 1 else 3001
    mode = {True: ccl.FUSE_FULL, "nochain": ccl.FUSE_NOCHAIN, False: ccl.FUSE_NONE}[fuse]
    plan = ccl.Plan(ccl.Schedule.compile(ops, R, nch, fuse=mode), ce, BF16, link_mode=0, slot_bytes=4096, **opts)
    ins = datagen.rank_inputs(95 + seed, "normal", R, nch[0] * ce, BF16)
    d_out = empty_outputs(R, nch[1] * ce, BF16)
    plan.execute(to_device(ins, BF16), d_out)
    torch.cuda.synchronize()
    plan.status()
    want, _, _ = oracle.run(np.array(ops, np.int32), R, nch, ce, BF16, ins)
    assert_bitexact(to_host(d_out, BF16), want)


def test_random_chain_programs_take_every_fold(ccl):
    """The random programs above do exercise the folds: across the seeds
    the plans hold two- and three-destination copies and three-operand
    reductions."""
    from test_compiler_planner import chain_program
    seen = set()
    for seed in range(8):
        ops, nch = chain_program(seed)
        for mode in (ccl.FUSE_FULL, ccl.FUSE_NOCHAIN, ccl.FUSE_NONE):
            for fold in (7, 15):
                plan = ccl.Plan(ccl.Schedule.compile(ops, 4, nch, fuse=mode), 3001, F32, link_mode=1,
                                slot_bytes=4096, fold=fold)
                seen |= {ccl.KIND_NAMES[st["kind"]] for st in plan.steps()}
    assert {"copy2", "copy3"} <= seen
    assert seen & {"rrs3", "rrc3", "rrcs3", "rsend", "rcsend", "rrc3d", "reduce2"}


SPECIALS = {0: [np.inf, -np.inf, np.nan, 3.0e38], 1: [0x7F80, 0xFF80, 0x7FC0, 0x7F7F], 2: [0x7C00, 0xFC00, 0x7E00, 0x7BFF]}


@pytest.mark.parametrize("dtype", [F32, BF16, F16])
@pytest.mark.parametrize("kind,R,opts", [(0, 8, dict()), (0, 8, dict(engine=1, cluster=4)), (0, 8, dict(protocol=1)),
                                         (2, 5, dict()), (3, 16, dict(channels=2, microbatches=2))])
def test_special_values_propagate_as_the_oracle_says(ccl, dtype, kind, R, opts):
    """Infinities, NaNs and values that overflow when added, planted in the
    inputs: every output element that is NaN in the oracle's result is NaN
    on the GPU and the rest is bit-exact (IEEE addition in the buffer type;
    a NaN's payload is not pinned)."""
    import torch
    import datagen
    import oracle
    from gpu_helpers import (oracle_program, to_device, empty_outputs, to_host, assert_bitexact_but_nan,
                             nan_mask)
    G = 8 if kind == 3 else 0
    ce = 4096
    ops, nch = oracle_program(kind, R, G)
    ins = datagen.rank_inputs(81, DIST[dtype], R, nch[0] * ce, dtype)
    rng = np.random.default_rng(82)
    for r in range(R):
        pos = rng.choice(nch[0] * ce, 24, replace=False)
        vals = np.array(SPECIALS[dtype] * 6)
        if dtype == F32:
            ins[r][pos] = vals.astype(np.float32)
        else:
            ins[r][pos] = vals.astype(np.uint16)
    plan = ccl.Plan(ccl.Schedule.builtin(kind, R, G), ce, dtype, **opts)
    d_out = empty_outputs(R, nch[1] * ce, dtype)
    plan.execute(to_device(ins, dtype), d_out)
    torch.cuda.synchronize()
    plan.status()
    want, _, _ = oracle.run(ops, R, nch, ce, dtype, ins)
    assert any(nan_mask(w, dtype).any() for w in want)
    assert_bitexact_but_nan(to_host(d_out, dtype), want, dtype)


def many_links_program(R):
    """Rank 0 hands a running sum to every other rank in turn and takes it
    back: copy to rank k, rank k adds its input, copy back to rank 0 --
    2 (R - 1) links, never two active at once, so packing puts all of rank
    0's on one threadblock."""
    ops = []
    for k in range(1, R):
        ops.append((0, 0, 0, 0, 1, 1, 0, 1) if k == 1 else (0, 0, 1, k - 1, k, 1, 0, 1))
        ops.append((1, k, 0, 0, k, 1, 0, 1))
        ops.append((0, k, 1, 0, 0, 1, k, 1))
    return ops


@pytest.mark.parametrize("fuse", [True, False])
@pytest.mark.parametrize("opts", [dict(), dict(protocol=1), dict(engine=1), dict(engine=1, protocol=1, cluster=2)])
def test_program_with_more_links_than_the_shared_link_table(ccl, fuse, opts):
    """A threadblock program on 24 links: the first ones come from the copy
    of the program's links in shared memory, the rest from the link array."""
    import torch
    import datagen
    import oracle
    from gpu_helpers import to_device, empty_outputs, to_host
    R, ce = 13, 4096
    nch = (R, R, R)
    ops = many_links_program(R)
    plan = ccl.Plan(ccl.Schedule.compile(ops, R, nch, fuse=fuse), ce, F32, tb_alloc=1, link_mode=0, channels=1,
                    slot_bytes=4096, **opts)
    st = plan.stats()
    assert st.nlinks == 2 * (R - 1) and st.nthreadblocks == R
    for rep in range(2):
        ins = datagen.rank_inputs(60 + rep, "normal", R, R * ce, F32)
        d_out = empty_outputs(R, R * ce, F32)
        plan.execute(to_device(ins, F32), d_out)
        torch.cuda.synchronize()
        plan.status()
        want, _, _ = oracle.run(np.array(ops, np.int32), R, nch, ce, F32, ins)
        assert_bitexact(to_host(d_out, F32), want)


@pytest.mark.parametrize("fuse", [True, "nochain"])
@pytest.mark.parametrize("opts", [dict(link_mode=0), dict(link_mode=1, tb_alloc=2), dict(link_mode=1, bulk=1),
                                  dict(engine=1), dict(protocol=1), dict(engine=1, protocol=1, cluster=4)])
@pytest.mark.parametrize("dtype", [F32, BF16])
def test_inplace_ring_allreduce_bitexact(ccl, fuse, opts, dtype):
    """In-place ring AllReduce (each rank's input is its output): the ring
    program reads a rank's input chunk before it writes that output chunk,
    so the result is the out-of-place oracle's, bit for bit."""
    import torch
    import datagen
    import oracle
    from gpu_helpers import oracle_program, to_device, to_host
    R = 8
    ce = 4096 if opts.get("protocol") else 3001
    flags = ccl.FLAG_NOCHAIN_COPIES if fuse == "nochain" else 0
    plan = ccl.Plan(ccl.Schedule.builtin(ccl.RING_ALLREDUCE, R, 0, flags), ce, dtype, channels=2, slot_bytes=8192,
                    **opts)
    ops, nch = oracle_program(0, R)
    ins = datagen.rank_inputs(17, DIST[dtype], R, R * ce, dtype)
    d = to_device(ins, dtype)
    plan.execute(d, d)
    torch.cuda.synchronize()
    plan.status()
    want, _, _ = oracle.run(ops, R, nch, ce, dtype, ins)
    assert_bitexact(to_host(d, dtype), want)


@pytest.mark.parametrize("cluster", [2, 4, 8])
def test_sequential_engine_on_clusters_bitexact(ccl, cluster):
    """Every threadblock program on a cluster of CTAs (the first waits and
    posts, each moves its share of a slot): ragged chunks, several slots per
    piece, FIFO and direct transport, every dtype."""
    cases = [(0, 8, 0, 4099, F32, True, 0), (0, 5, 0, 1000, BF16, "nochain", 1), (1, 8, 0, 3001, F16, False, 1),
             (2, 8, 0, 777, BF16, True, 0), (3, 4, 2, 2048, F32, "nochain", 1), (0, 8, 0, 3, I32, True, 0)]
    for kind, R, G, ce, dtype, fuse, lm in cases:
        got, want, plan = run_case(ccl, kind, R, G, ce, dtype, DIST[dtype], 31, fuse=fuse, link_mode=lm,
                                   engine=ccl.ENGINE_SEQUENTIAL, cluster=cluster, channels=2, slot_bytes=4096)
        assert plan.stats().cluster == cluster
        assert_bitexact(got, want)
