"""Host-side pins of the compiler, planner and tuner (no GPU).

* closed-form instruction mixes and schedule bytes of the built-in programs;
* fused instruction lists interpreted here (a plain reading of each fused
  kind's definition) and compared bit for bit with the oracle, for the
  built-ins and for random chunk programs, with fusion on and off;
* sub-pipeline constraints of RR and HPDS; threadblock packing; direct
  transport; deadlock rejection; argument validation;
* the tuner's coordinate descent on synthetic unimodal bandwidth surfaces.
"""
import math

import numpy as np
import pytest

import datagen
import oracle
from oracle import schedules as OS

ccl = pytest.importorskip("collective_communication_schedule_gb300")

F32, BF16, F16, I32 = 0, 1, 2, 3
KIND = {n: i for i, n in enumerate(ccl.KIND_NAMES)}
ORACLE_GEN = {0: ("ring_allreduce", lambda R, G: (R,)), 1: ("ring_allgather", lambda R, G: (R,)),
              2: ("ring_reducescatter", lambda R, G: (R,)), 3: ("hier_allreduce", lambda R, G: (G, R // G)),
              4: ("alltoall_two_phase", lambda R, G: (G, R // G)), 5: ("alltonext", lambda R, G: (G, R // G))}


# --------------------------------------------------------------- closed forms

@pytest.mark.parametrize("R", [2, 3, 8, 16])
def test_ring_allreduce_instruction_mix_and_bytes(R):
    s = ccl.Schedule.builtin(ccl.RING_ALLREDUCE, R)
    per_rank = {}
    for ins in s.instrs():
        per_rank.setdefault(ins["rank"], []).append(ccl.KIND_NAMES[ins["kind"]])
    for r in range(R):
        k = sorted(per_rank[r])
        want = sorted(["send"] + ["rrs"] * (R - 2) + ["rrcs"] + ["rcs"] * (R - 2) + ["recv"])
        assert k == want
    # R ranks x N (6 - 4/R) bytes, N = R chunks of one element-byte
    assert s.info().bytes_per_chunk_elem_x_esize == R * R * (6 * R - 4) // R


@pytest.mark.parametrize("R", [2, 4, 8])
def test_allgather_and_reducescatter_bytes(R):
    for kind in (ccl.RING_ALLGATHER, ccl.RING_REDUCESCATTER):
        s = ccl.Schedule.builtin(kind, R)
        assert s.info().bytes_per_chunk_elem_x_esize == R * (3 * R - 1)


def test_hierarchical_alltoall_alltonext_bytes():
    # hierarchical, G = 8, 2 groups: 6.125 x (16 chunks) per rank, 16 ranks
    assert ccl.Schedule.builtin(ccl.HIER_ALLREDUCE, 16, 8).info().bytes_per_chunk_elem_x_esize == 16 * 98
    # two-phase AllToAll, R = 32, G = 8: 216 blocks per rank
    assert ccl.Schedule.builtin(ccl.ALLTOALL_2PHASE, 32, 8).info().bytes_per_chunk_elem_x_esize == 32 * 216
    # AllToNext, 3 groups of 8: 21 direct pairs x 4 x 8 parts + 2 relayed pairs
    # x (two 2-hop parts of 6 + six 3-hop parts of 8, relays fused to recv-send)
    assert ccl.Schedule.builtin(ccl.ALLTONEXT, 24, 8).info().bytes_per_chunk_elem_x_esize == 21 * 32 + 2 * 60


def test_unfused_program_has_only_halves():
    s = ccl.Schedule.builtin(ccl.RING_ALLREDUCE, 8, 0, ccl.FLAG_NOFUSE)
    kinds = {ccl.KIND_NAMES[i["kind"]] for i in s.instrs()}
    assert kinds <= {"copy", "reduce", "send", "recv", "rrc"}
    # every transfer costs send 2n + receive 2n (or 3n when it reduces)
    fused = ccl.Schedule.builtin(ccl.RING_ALLREDUCE, 8).info().bytes_per_chunk_elem_x_esize
    assert s.info().bytes_per_chunk_elem_x_esize > fused


# ------------------------------------------- fused-instruction interpretation

def _add(a, b, dtype):
    if dtype == F32:
        return (a.astype(np.float32) + b.astype(np.float32)).astype(np.float32)
    if dtype == I32:
        return (a.astype(np.int64) + b.astype(np.int64)).astype(np.int32)
    if dtype == BF16:
        return oracle.add_bf16(a, b)
    return oracle.add_f16(a, b)


def interpret_fused(instrs, R, nchunks, ce, dtype, inputs):
    """Run fused instructions: every rank in position order, a receiving
    instruction once its transfer has been sent."""
    st = datagen.STORAGE[dtype]
    bufs = {}
    for r in range(R):
        bufs[(r, 0)] = np.asarray(inputs[r], st).copy()
        bufs[(r, 1)] = np.full(nchunks[1] * ce * datagen.ESIZE[dtype], 0xA5, np.uint8).view(st)
        bufs[(r, 2)] = np.full(max(nchunks[2], 0) * ce * datagen.ESIZE[dtype], 0xA5, np.uint8).view(st)

    def rng(rank, buf, off, cnt):
        return bufs[(rank, buf)][off * ce:(off + cnt) * ce]

    slots = {}
    by_rank = {}
    for i in instrs:
        by_rank.setdefault(i["rank"], []).append(i)
    for v in by_rank.values():
        v.sort(key=lambda x: x["position"])
    pc = {r: 0 for r in by_rank}
    remaining = len(instrs)
    while remaining:
        moved = False
        for r, lst in by_rank.items():
            while pc[r] < len(lst):
                ins = lst[pc[r]]
                if ins["xfer_in"] >= 0 and ins["xfer_in"] not in slots:
                    break
                k = ccl.KIND_NAMES[ins["kind"]]
                cnt = ins["count"]
                src = rng(ins["src_rank"], ins["src_buf"], ins["src_off"], cnt) if ins["src_rank"] >= 0 else None
                loc = rng(ins["loc_rank"], ins["loc_buf"], ins["loc_off"], cnt) if ins["loc_rank"] >= 0 else None
                inc = slots.pop(ins["xfer_in"]) if ins["xfer_in"] >= 0 else None
                if k in ("copy", "copy_send"):
                    val = src.copy()
                elif k == "reduce":
                    val = _add(loc, src, dtype)
                elif k == "send":
                    val = src.copy()
                elif k in ("recv", "rcs", "fwd"):
                    val = inc
                elif k in ("rrc", "rrs", "rrcs"):
                    val = _add(loc, inc, dtype)
                else:
                    raise AssertionError(k)
                if ins["dst_rank"] >= 0:
                    rng(ins["dst_rank"], ins["dst_buf"], ins["dst_off"], cnt)[:] = val
                if ins["xfer_out"] >= 0:
                    slots[ins["xfer_out"]] = val.copy()
                pc[r] += 1
                remaining -= 1
                moved = True
        assert moved, "fused program cannot make progress"
    return [bufs[(r, 1)] for r in range(R)]


@pytest.mark.parametrize("kind,R,G", [(0, 8, 0), (0, 3, 0), (1, 8, 0), (2, 8, 0), (2, 5, 0), (3, 16, 8), (3, 6, 3),
                                      (4, 8, 4), (4, 32, 8), (5, 24, 8), (5, 6, 2)])
@pytest.mark.parametrize("fuse", [True, False, "nochain"])
def test_fused_builtins_equal_oracle(kind, R, G, fuse):
    dtype, ce = BF16, 5
    flags = ccl.FLAG_NOCHAIN_COPIES if fuse == "nochain" else (0 if fuse else ccl.FLAG_NOFUSE)
    s = ccl.Schedule.builtin(kind, R, G, flags)
    name, args = ORACLE_GEN[kind]
    ops, nch = OS.BUILTINS[name](*args(R, G))
    assert tuple(s.info().nchunks) == tuple(nch)
    ins = datagen.rank_inputs(7, "normal", R, nch[0] * ce, dtype)
    got = interpret_fused(s.instrs(), R, nch, ce, dtype, ins)
    want, _, _ = oracle.run(ops, R, nch, ce, dtype, ins)
    for r in range(R):
        assert np.array_equal(got[r].view(np.uint8), want[r].view(np.uint8)), f"rank {r}"


def test_nochain_keeps_copy_receives_apart():
    """Ring AllReduce: full fusion chains every all-gather hop into a
    receive-copy-send; without copy chaining each middle hop stays a receive
    plus a send, while the reduce-scatter half keeps its fused reduce forms.
    Under direct transport the copy hops then become plain copies."""
    for R in (3, 8):
        nochain = ccl.Schedule.builtin(ccl.RING_ALLREDUCE, R, 0, ccl.FLAG_NOCHAIN_COPIES)
        per_rank = {}
        for ins in nochain.instrs():
            per_rank.setdefault(ins["rank"], []).append(ccl.KIND_NAMES[ins["kind"]])
        for r in range(R):
            want = ["send"] + ["rrs"] * (R - 2) + ["rrcs"] + ["recv", "send"] * (R - 2) + ["recv"]
            assert sorted(per_rank[r]) == sorted(want)
        # same bytes in FIFO mode: (R-2) chunks per rank move 2 bytes (recv)
        # + 2 (send) instead of 3 (rcs) and one more read of the output
        full = ccl.Schedule.builtin(ccl.RING_ALLREDUCE, R)
        nf = full.info().bytes_per_chunk_elem_x_esize
        nn = nochain.info().bytes_per_chunk_elem_x_esize
        assert nn == nf + R * (R - 2)
        # direct transport: a middle hop is one copy into the next rank's
        # output (2 bytes per element byte) instead of a receive-copy-send
        # (3), and the recv-reduce-copy-send that completes a chunk writes
        # the next rank's output itself, so that rank's receive (2) goes
        # (copy chains not folded)
        ce, es = 64, 4
        st_full = full.check(ce, F32, link_mode=ccl.LINK_DIRECT, fold=1)
        st_nochain = nochain.check(ce, F32, link_mode=ccl.LINK_DIRECT, fold=1)
        assert st_nochain.schedule_bytes == st_full.schedule_bytes - R * (R - 2) * ce * es - 2 * R * ce * es


def test_fusion_keeps_the_order_of_dependent_sends_on_a_link():
    """Rank 0 receives a reduction (op 0) and later sends two ranges of its
    result to rank 1 (ops 1 and 2); rank 1 takes op 1 before op 2 (op 2
    reduces into the range op 1 wrote).  Chaining op 2's send into the
    receive of op 0 would put it on the link ahead of op 1's send, which
    must follow op 0; the compiler leaves that send where it is, and the
    program plans in every fusion mode with the oracle's result."""
    ops = [(1, 1, 0, 0, 0, 1, 0, 3), (0, 0, 1, 0, 1, 2, 2, 1), (1, 0, 1, 0, 1, 2, 0, 3)]
    nch = (3, 3, 3)
    want, _, _ = oracle.run(np.array(ops, np.int32), 2, nch, 4, I32,
                            datagen.rank_inputs(1, "int", 2, 12, I32))
    for fuse in (ccl.FUSE_FULL, ccl.FUSE_NOCHAIN, ccl.FUSE_NONE):
        s = ccl.Schedule.compile(ops, 2, nch, fuse=fuse)
        s.check(64, F32)
        got = interpret_fused(s.instrs(), 2, nch, 4, I32, datagen.rank_inputs(1, "int", 2, 12, I32))
        for r in range(2):
            assert np.array_equal(got[r], want[r])


def test_send_is_not_chained_past_a_dependent_round_trip():
    """Rank 0 receives out[0] (op 0), sends it to rank 2 (op 2), which sends
    it back into rank 0's scratch (op 3); op 4 sends that scratch on to rank
    1 and op 5 reduces rank 0's out[0] into the same range of rank 1.  Op
    4's send depends on op 0 only through the round trip over rank 2; moving
    op 5's send up into op 0's receive would put it ahead of op 4's on the
    link 0 -> 1, although rank 1 takes op 4 first.  The compiler keeps op 4's
    send ahead and the program plans in every fusion mode with the oracle's
    result."""
    ops = [(0, 1, 0, 0, 0, 1, 0, 1), (0, 0, 1, 0, 0, 2, 1, 1), (0, 0, 2, 1, 2, 1, 0, 1),
           (0, 2, 1, 0, 0, 2, 0, 1), (0, 0, 2, 0, 1, 1, 1, 1), (1, 0, 1, 0, 1, 1, 1, 1)]
    nch, R = (3, 3, 3), 3
    ins = datagen.rank_inputs(4, "int", R, 12, I32)
    want, _, _ = oracle.run(np.array(ops, np.int32), R, nch, 4, I32, ins)
    for fuse in (ccl.FUSE_FULL, ccl.FUSE_NOCHAIN, ccl.FUSE_NONE):
        s = ccl.Schedule.compile(ops, R, nch, fuse=fuse)
        ins0 = [i for i in s.instrs() if i["rank"] == 0]
        pos_of = {i["xfer_out"]: i["position"] for i in ins0 if i["xfer_out"] >= 0}
        # transfers are numbered by their operation: op 4 -> 3, op 5 -> 4
        assert pos_of[3] < pos_of[4]
        for link_mode in (ccl.LINK_FIFO, ccl.LINK_DIRECT):
            st = s.check(64, F32, link_mode=link_mode)
            assert st.fuse == fuse
        got = interpret_fused(s.instrs(), R, nch, 4, I32, ins)
        for r in range(R):
            assert np.array_equal(got[r], want[r])


# Random programs (seeded fuzzing of the compiler) that the fused modes once
# failed to plan although their unfused form planned: cycles of the
# timeline through a fused receive-...-send or a copy-send whose send half
# waits on the receiver side for a dependent of its buffer effect (first
# three), and fused programs whose moved sends keep more transfers in flight
# on a link than 4 FIFO slots hold (last two: planned from a less fused form).
FUZZED = [
    (5, 2, [(1, 3, 1, 0, 1, 2, 0, 2), (0, 0, 1, 0, 4, 1, 0, 1), (0, 0, 2, 0, 3, 1, 0, 2), (0, 1, 1, 1, 2, 1, 1, 1),
            (1, 2, 2, 0, 4, 1, 1, 1), (0, 1, 0, 1, 0, 2, 0, 1), (0, 4, 1, 0, 0, 2, 0, 1), (1, 4, 1, 0, 4, 2, 0, 2),
            (0, 3, 1, 1, 0, 2, 0, 1), (1, 3, 1, 1, 2, 2, 0, 1), (1, 0, 2, 0, 3, 1, 0, 2), (1, 3, 2, 0, 4, 2, 1, 1),
            (0, 2, 0, 0, 4, 2, 0, 2), (0, 4, 1, 1, 3, 2, 0, 1), (0, 3, 2, 0, 2, 2, 1, 1)]),
    (2, 2, [(1, 0, 0, 1, 0, 1, 1, 1), (0, 1, 2, 0, 1, 1, 0, 1), (1, 0, 0, 0, 1, 1, 1, 1), (0, 1, 1, 0, 0, 2, 0, 1),
            (0, 1, 1, 0, 1, 2, 0, 1), (0, 1, 0, 1, 0, 2, 1, 1), (0, 0, 2, 0, 1, 1, 0, 2), (0, 0, 2, 0, 1, 1, 0, 2),
            (1, 0, 0, 0, 0, 1, 0, 2), (1, 0, 0, 0, 0, 2, 0, 2), (0, 0, 2, 1, 0, 1, 0, 1), (0, 0, 0, 0, 1, 1, 0, 2),
            (1, 1, 1, 0, 1, 2, 0, 2), (1, 0, 2, 0, 1, 2, 0, 2), (1, 1, 1, 0, 0, 2, 0, 2), (1, 1, 0, 0, 0, 2, 0, 2),
            (0, 1, 1, 0, 1, 2, 0, 1), (0, 0, 0, 1, 0, 2, 1, 1), (0, 1, 0, 1, 0, 2, 1, 1)]),
    (4, 3, [(0, 1, 0, 0, 1, 2, 0, 3), (0, 0, 2, 0, 3, 1, 0, 3), (0, 3, 2, 1, 2, 1, 2, 1), (0, 3, 1, 0, 1, 1, 0, 3),
            (1, 2, 1, 1, 1, 1, 0, 2), (1, 1, 0, 0, 0, 1, 0, 3), (0, 3, 1, 0, 3, 2, 0, 3), (0, 1, 2, 0, 1, 1, 0, 2),
            (0, 0, 2, 0, 1, 1, 0, 2), (0, 1, 2, 0, 0, 2, 0, 3), (0, 0, 2, 1, 2, 2, 1, 1), (0, 2, 0, 0, 0, 2, 0, 3),
            (1, 0, 1, 0, 1, 2, 0, 2), (1, 3, 2, 1, 2, 2, 1, 1), (0, 0, 1, 1, 2, 2, 2, 1), (1, 3, 1, 0, 1, 2, 1, 2),
            (0, 1, 2, 0, 3, 1, 0, 3), (1, 1, 2, 0, 3, 2, 0, 3), (1, 2, 0, 0, 2, 1, 0, 2), (1, 0, 1, 0, 3, 2, 0, 2),
            (1, 1, 1, 0, 3, 1, 0, 3), (0, 3, 1, 2, 0, 1, 0, 1), (0, 2, 1, 1, 0, 2, 0, 2), (1, 3, 0, 1, 1, 2, 1, 1),
            (1, 1, 0, 0, 0, 1, 1, 2), (0, 0, 2, 0, 0, 1, 1, 1), (0, 1, 0, 1, 2, 1, 1, 2), (0, 1, 0, 2, 3, 1, 0, 1),
            (0, 0, 2, 0, 2, 2, 0, 3)]),
    (2, 1, [(0, 1, 2, 0, 1, 1, 0, 1), (1, 0, 2, 0, 1, 1, 0, 1), (0, 0, 1, 0, 1, 1, 0, 1), (1, 0, 1, 0, 1, 1, 0, 1),
            (1, 1, 2, 0, 0, 1, 0, 1), (0, 1, 0, 0, 1, 2, 0, 1), (1, 1, 2, 0, 0, 1, 0, 1), (1, 0, 2, 0, 1, 2, 0, 1),
            (1, 0, 0, 0, 0, 2, 0, 1), (1, 1, 0, 0, 0, 1, 0, 1), (1, 1, 1, 0, 0, 2, 0, 1), (1, 1, 0, 0, 1, 2, 0, 1),
            (0, 0, 0, 0, 0, 1, 0, 1), (0, 1, 0, 0, 0, 2, 0, 1), (1, 0, 2, 0, 1, 2, 0, 1), (1, 1, 0, 0, 1, 1, 0, 1),
            (0, 0, 1, 0, 0, 2, 0, 1)]),
    (2, 1, [(1, 1, 1, 0, 0, 1, 0, 1), (0, 0, 1, 0, 1, 1, 0, 1), (0, 1, 2, 0, 0, 2, 0, 1), (1, 0, 1, 0, 1, 2, 0, 1),
            (0, 1, 2, 0, 1, 1, 0, 1), (0, 1, 0, 0, 1, 2, 0, 1), (1, 1, 0, 0, 0, 2, 0, 1), (0, 1, 0, 0, 1, 2, 0, 1),
            (1, 1, 2, 0, 0, 1, 0, 1), (0, 0, 1, 0, 0, 2, 0, 1), (0, 0, 0, 0, 0, 1, 0, 1), (1, 0, 2, 0, 1, 1, 0, 1),
            (1, 1, 2, 0, 0, 1, 0, 1), (1, 1, 2, 0, 0, 2, 0, 1), (1, 1, 1, 0, 0, 2, 0, 1), (1, 1, 1, 0, 0, 1, 0, 1),
            (0, 1, 0, 0, 0, 1, 0, 1), (1, 0, 2, 0, 1, 1, 0, 1), (1, 1, 1, 0, 1, 2, 0, 1), (0, 0, 0, 0, 1, 2, 0, 1),
            (1, 1, 2, 0, 0, 1, 0, 1)]),
]


@pytest.mark.parametrize("case", range(len(FUZZED)))
@pytest.mark.parametrize("fuse", [ccl.FUSE_FULL, ccl.FUSE_NOCHAIN])
def test_fuzzed_programs_plan_in_fused_modes(case, fuse):
    R, C, ops = FUZZED[case]
    nch = (C, C, C)
    s = ccl.Schedule.compile(ops, R, nch, fuse=fuse)
    for link_mode in (ccl.LINK_FIFO, ccl.LINK_DIRECT):
        st = s.check(64, F32, link_mode=link_mode)
        assert st.fuse in (fuse, ccl.FUSE_NOCHAIN, ccl.FUSE_NONE)
        if case < 3:
            assert st.fuse == fuse      # planned as compiled (split timeline)
    ins = datagen.rank_inputs(case, "int", R, C * 3, I32)
    got = interpret_fused(s.instrs(), R, nch, 3, I32, ins)
    want, _, _ = oracle.run(np.array(ops, np.int32), R, nch, 3, I32, ins)
    for r in range(R):
        assert np.array_equal(got[r], want[r])


def random_program(seed, R=3, C=4, nops=40):
    rng = np.random.default_rng(seed)
    ops = []
    while len(ops) < nops:
        op = int(rng.integers(0, 2))
        sr, dr = int(rng.integers(0, R)), int(rng.integers(0, R))
        sb = int(rng.choice([0, 1, 2]))
        db = int(rng.choice([1, 2]))          # never write inputs
        cnt = int(rng.integers(1, 3))
        so, do = int(rng.integers(0, C - cnt + 1)), int(rng.integers(0, C - cnt + 1))
        if sr == dr and sb == db and so < do + cnt and do < so + cnt:
            continue
        ops.append((op, sr, sb, so, dr, db, do, cnt))
    return ops, (C, C, C)


@pytest.mark.parametrize("seed", range(12))
@pytest.mark.parametrize("fuse", [True, False, ccl.FUSE_NOCHAIN])
def test_random_programs_fused_equal_oracle(seed, fuse):
    ops, nch = random_program(seed)
    R, ce = 3, 3
    s = ccl.Schedule.compile(ops, R, nch, fuse=fuse)
    ins = datagen.rank_inputs(seed, "int", R, nch[0] * ce, I32)
    # scratch starts as the sentinel on both sides; reads of it are part of
    # the program, so both must start from the same bytes
    got = interpret_fused(s.instrs(), R, nch, ce, I32, ins)
    want, _, _ = oracle.run(np.array(ops), R, nch, ce, I32, ins)
    for r in range(R):
        assert np.array_equal(got[r], want[r])
    ins = datagen.rank_inputs(seed, "normal", R, nch[0] * ce, F16)
    got = interpret_fused(s.instrs(), R, nch, ce, F16, ins)
    want, _, _ = oracle.run(np.array(ops), R, nch, ce, F16, ins)
    for r in range(R):
        assert np.array_equal(got[r], want[r])


def chain_program(seed, R=4, C=4, nops=30):
    """A seeded random program rich in chains: most ops read a range that
    one of the last few ops wrote (a copy or reduction passed on) and write
    another rank, the rest read an input.  Reads of scratch (and the
    destination of a reduction into scratch) only touch chunks an earlier op
    wrote, so the result does not depend on scratch's initial bytes;
    outputs start as the same sentinel on both sides."""
    rng = np.random.default_rng(seed)
    ops, written, recent = [], set(), []
    while len(ops) < nops:
        op = int(rng.random() < 0.4)
        if recent and rng.random() < 0.7:
            sr, sb, so, cnt = recent[-1 - int(rng.integers(0, min(4, len(recent))))]
        else:
            cnt = int(rng.integers(1, 3))
            sr, sb, so = int(rng.integers(0, R)), 0, int(rng.integers(0, C - cnt + 1))
        dr = (sr + int(rng.integers(1, R))) % R if rng.random() < 0.9 else sr
        db = int(rng.choice([1, 2]))
        do = int(rng.integers(0, C - cnt + 1))
        if sb == 2 and any((sr, 2, c) not in written for c in range(so, so + cnt)):
            continue
        if op == 1 and db == 2 and any((dr, 2, c) not in written for c in range(do, do + cnt)):
            continue
        if sr == dr and sb == db and so < do + cnt and do < so + cnt:
            continue
        ops.append((op, sr, sb, so, dr, db, do, cnt))
        written |= {(dr, db, c) for c in range(do, do + cnt)}
        recent.append((dr, db, do, cnt))
    return ops, (C, C, C)


@pytest.mark.parametrize("seed", range(40))
@pytest.mark.parametrize("fuse", [ccl.FUSE_FULL, ccl.FUSE_NOCHAIN, ccl.FUSE_NONE])
def test_chain_programs_plan_with_every_fold(seed, fuse):
    """Random chain-rich programs plan on direct transport under every fold
    mask, and each fold bit only ever saves schedule bytes: where a fold
    would make the timeline cyclic or the threadblocks deadlock, the planner
    gives up that kind of fold alone (three hops -> two, then reduction
    chains, ...) and keeps the rest.  Compared within one fusion form (a
    fold can let a fused form plan that otherwise falls back to a less
    fused one)."""
    ops, nch = chain_program(seed)
    s = ccl.Schedule.compile(ops, 4, nch, fuse=fuse)
    st = [s.check(3001, F32, link_mode=ccl.LINK_DIRECT, slot_bytes=4096, fold=f) for f in range(16)]
    for f in range(16):
        for g in (0, f & ~2, f & ~4, f & ~8):
            if st[f].fuse == st[g].fuse:
                assert st[f].schedule_bytes <= st[g].schedule_bytes, (f, g)


@pytest.mark.parametrize("bad", [
    [(0, 0, 0, 0, 0, 0, 0, 1)],            # overlapping source and destination
    [(0, 0, 0, 3, 1, 1, 0, 2)],            # source range outside the buffer
    [(0, 5, 0, 0, 1, 1, 0, 1)],            # rank out of range
    [(0, 0, 0, 0, 1, 1, 0, 0)],            # empty count
    [(9, 0, 0, 0, 1, 1, 0, 1)],            # unknown opcode
    [(0, 0, 4, 0, 1, 1, 0, 1)],            # unknown buffer kind
])
def test_invalid_programs_are_rejected(bad):
    with pytest.raises(ccl.CclError) as e:
        ccl.Schedule.compile(bad, 2, (4, 4, 0))
    assert e.value.code == 1


# ------------------------------------------------------------------ planner

@pytest.mark.parametrize("kind,R,G", [(0, 8, 0), (3, 16, 8), (4, 32, 8), (5, 24, 8), (1, 8, 0)])
@pytest.mark.parametrize("sched", [ccl.SCHED_RR, ccl.SCHED_HPDS])
def test_subpipelines_respect_links_and_dependencies(kind, R, G, sched):
    s = ccl.Schedule.builtin(kind, R, G)
    sp, nsub = s.timeline(sched)
    instrs = s.instrs()
    # transfers: (sender, receiver) of each transfer id
    ends = {}
    for i in instrs:
        if i["xfer_out"] >= 0:
            ends.setdefault(i["xfer_out"], {})["snd"] = i
        if i["xfer_in"] >= 0:
            ends.setdefault(i["xfer_in"], {})["rcv"] = i
    seen = {}
    for x, e in ends.items():
        link = (e["snd"]["rank"], e["rcv"]["rank"])
        assert (sp[x], link) not in seen, "two transfers on one link in one sub-pipeline"
        seen[(sp[x], link)] = x
        # a forwarded transfer comes after the one it forwards
        if e["snd"]["xfer_in"] >= 0:
            assert sp[x] > sp[e["snd"]["xfer_in"]]
    assert 0 <= min(sp) and max(sp) < nsub


def test_hpds_prioritises_least_scheduled_chunks():
    """Chunk 0 fans out from rank 0 on three links while chunk 1 takes one
    link; both then want link 1->2.  Round-robin keeps program order (chunk
    0 first); HPDS serves the chunk with fewer scheduled tasks (chunk 1)."""
    ops = [(0, 0, 0, 0, 1, 2, 0, 1), (0, 0, 0, 0, 2, 2, 0, 1), (0, 0, 0, 0, 3, 2, 0, 1),
           (0, 3, 0, 1, 1, 2, 1, 1),
           (0, 1, 2, 0, 2, 1, 0, 1), (0, 1, 2, 1, 2, 1, 1, 1)]
    s = ccl.Schedule.compile(ops, 4, (2, 2, 2))
    assert s.timeline(ccl.SCHED_RR) == ([0, 0, 0, 0, 1, 2], 3)
    assert s.timeline(ccl.SCHED_HPDS) == ([0, 0, 0, 0, 2, 1], 3)
    # the ring keeps its 2 (R - 1) steps under both
    r = ccl.Schedule.builtin(ccl.RING_ALLREDUCE, 8)
    assert r.timeline(ccl.SCHED_HPDS)[1] == r.timeline(ccl.SCHED_RR)[1] == 2 * (8 - 1)


@pytest.mark.parametrize("kind,R,G", [(0, 8, 0), (3, 16, 8), (4, 32, 8), (5, 24, 8)])
def test_state_based_packing_never_adds_threadblocks(kind, R, G):
    s = ccl.Schedule.builtin(kind, R, G)
    a = s.check(1024, F32, tb_alloc=ccl.TB_CONNECTION, link_mode=ccl.LINK_FIFO, channel_scaling=0)
    b = s.check(1024, F32, tb_alloc=ccl.TB_PACKED, link_mode=ccl.LINK_FIFO, channel_scaling=0)
    assert b.nthreadblocks <= a.nthreadblocks
    assert b.nthreadblocks_connection == a.nthreadblocks


def test_packing_merges_idle_inter_group_threadblocks():
    s = ccl.Schedule.builtin(ccl.HIER_ALLREDUCE, 16, 8)
    a = s.check(1024, F32, tb_alloc=ccl.TB_CONNECTION, microbatches=4, channel_scaling=0)
    b = s.check(1024, F32, tb_alloc=ccl.TB_PACKED, microbatches=4, channel_scaling=0)
    assert b.nthreadblocks == a.nthreadblocks // 2


def test_direct_transport_removes_fifos_from_alltoall():
    s = ccl.Schedule.builtin(ccl.ALLTOALL_2PHASE, 32, 8)
    fifo = s.check(1024, F16, link_mode=ccl.LINK_FIFO)
    direct = s.check(1024, F16, link_mode=ccl.LINK_DIRECT)
    assert direct.nlinks == 0 and fifo.nlinks > 0
    # per rank (G = 8, 4 groups): 7 peers x 4 blocks in the intra-group
    # phase, 3 peers x 8 blocks in the inter-group phase, 4 blocks copied
    # locally.  A FIFO transfer costs 4 bytes per element byte (staging
    # write + read), a direct one 2, like a copy.
    blk = 1024 * 2
    sent, copied = 32 * (7 * 4 + 3 * 8), 32 * 4
    assert fifo.schedule_bytes == blk * (4 * sent + 2 * copied)
    assert direct.schedule_bytes == blk * 2 * (sent + copied)


def test_channel_scaling_gives_small_instructions_fewer_threadblocks():
    s = ccl.Schedule.builtin(ccl.ALLTONEXT, 24, 8)
    flat = s.check(4096, F32, channels=8, channel_scaling=0)
    scaled = s.check(4096, F32, channels=8, channel_scaling=1)
    assert scaled.nthreadblocks < flat.nthreadblocks
    assert scaled.schedule_bytes == flat.schedule_bytes


def test_task_order_ring_with_big_pieces_plans_unfused():
    """Each fused ring step (receive, reduce, send on) must move a whole
    piece while its neighbour does the same: with a piece larger than the
    FIFO no fused step can finish, so the planner plans the program from its
    unfused compilation (sends and receives in steps of their own), which
    can; with micro-batches the fused form plans as compiled."""
    s = ccl.Schedule.builtin(ccl.RING_ALLREDUCE, 4)
    kw = dict(mb_order=ccl.MB_TASK, microbatches=1, slot_bytes=4096, fifo_slots=2)
    st = s.check(65536, F32, **kw)
    assert st.fuse == ccl.FUSE_NONE
    unfused = ccl.Schedule.builtin(ccl.RING_ALLREDUCE, 4, 0, ccl.FLAG_NOFUSE).check(65536, F32, **kw)
    assert st.schedule_bytes == unfused.schedule_bytes
    st = s.check(65536, F32, mb_order=ccl.MB_AUTO, slot_bytes=4096, fifo_slots=2)
    assert st.microbatches > 1 and st.fuse == ccl.FUSE_FULL


def test_plan_options_are_validated():
    s = ccl.Schedule.builtin(ccl.RING_ALLREDUCE, 4)
    for kw in (dict(channels=300), dict(nthreads=100), dict(slot_bytes=24), dict(fifo_slots=1),
               dict(tile_bytes=70000), dict(link_mode=5), dict(scheduler=7)):
        with pytest.raises(ccl.CclError) as e:
            s.check(1024, F32, **kw)
        assert e.value.code == 1, kw
    with pytest.raises(ccl.CclError):
        s.check(0, F32)


def test_channels_split_in_16_byte_units_and_keep_bytes():
    s = ccl.Schedule.builtin(ccl.RING_ALLREDUCE, 8)
    base = s.check(1000, BF16, channels=1)
    for p in (2, 3, 7):
        st = s.check(1000, BF16, channels=p, channel_scaling=0)
        assert st.schedule_bytes == base.schedule_bytes
        assert st.nthreadblocks == 8 * p


# -------------------------------------------------------------------- tuner

def _surface(peak):
    c0, t0, s0 = peak

    def f(o):
        return math.exp(-(math.log2(o.channels) - math.log2(c0)) ** 2 - (math.log2(o.nthreads) - math.log2(t0)) ** 2
                        - (math.log2(o.slot_bytes) - math.log2(s0)) ** 2)
    return f


@pytest.mark.parametrize("peak", [(12, 256, 1 << 18), (1, 1024, 1 << 14), (48, 128, 1 << 22), (4, 512, 1 << 17)])
def test_coordinate_descent_reaches_the_peak_of_unimodal_surfaces(peak):
    best, bw, n = ccl.tune_search(_surface(peak))
    assert (best.channels, best.nthreads, best.slot_bytes) == peak
    assert bw == pytest.approx(1.0)
    # sixteen subspaces (policy x protocol x transport x engine), each
    # probing far fewer points than its 324-point grid
    assert n <= 16 * 24


def test_coordinate_descent_treats_infeasible_points_as_zero():
    f = _surface((24, 512, 1 << 17))

    def g(o):
        return 0.0 if o.channels > 16 else f(o)   # too many threadblocks
    best, bw, n = ccl.tune_search(g)
    assert best.channels == 16 and bw > 0


def test_coordinate_descent_plateau_stops_early():
    # sixteen subspaces (policy x protocol x transport x engine): on a flat
    # surface each tries one step up and one down per coordinate (at most 6
    # probes; 8 on the sequential engine, which also has the CTAs per
    # program; 4 more with direct transport, one flip of each fold bit),
    # plus the start
    seen = set()

    def flat(o):
        seen.add((o.tb_alloc, o.protocol, o.link_mode, o.engine))
        return 1.0
    best, bw, n = ccl.tune_search(flat)
    assert bw == 1.0 and n <= 1 + 8 * 6 + 8 * 8 + 8 * 4
    assert len(seen) == 16


def test_microbatch_window_is_used_when_the_fifo_holds_it():
    s = ccl.Schedule.builtin(ccl.HIER_ALLREDUCE, 16, 8)
    kw = dict(channels=2, microbatches=8, tb_alloc=ccl.TB_PACKED, slot_bytes=65536, mb_order=ccl.MB_ALGO)
    assert s.check(65536, F32, fifo_slots=4, mb_window=1, **kw).mb_window == 1
    # auto: min(m, fifo_slots / (2 x slots per piece)); here a piece is one
    # slot (65536 elements / 2 channels / 8 micro-batches x 4 bytes = 16 KiB)
    assert s.check(65536, F32, fifo_slots=4, mb_window=0, **kw).mb_window == 2
    assert s.check(65536, F32, fifo_slots=9, mb_window=0, **kw).mb_window == 4
    assert s.check(65536, F32, fifo_slots=32, mb_window=0, **kw).mb_window == 8
    # pieces of two slots: five slots hold no double-buffered window of 2
    r = ccl.Schedule.builtin(ccl.RING_ALLREDUCE, 8)
    big = dict(channels=24, microbatches=6, slot_bytes=131072, mb_order=ccl.MB_ALGO)
    assert r.check(32 << 20 >> 2, F32, fifo_slots=5, mb_window=0, **big).mb_window == 1
    assert r.check(32 << 20 >> 2, F32, fifo_slots=8, mb_window=0, **big).mb_window == 2
    # same steps and bytes in another order
    a = s.check(65536, F32, fifo_slots=9, mb_window=1, **kw)
    b = s.check(65536, F32, fifo_slots=9, mb_window=8, **kw)
    assert (a.nsteps, a.schedule_bytes) == (b.nsteps, b.schedule_bytes)


def test_microbatch_window_larger_than_the_fifo_plans_unfused():
    """A fused ring step that must send a whole window before its neighbour
    reads any of it needs window + 1 slots per link: with fewer the fused
    form cannot finish and the program is planned unfused (its receives and
    sends in steps of their own), with enough slots it is planned fused."""
    s = ccl.Schedule.builtin(ccl.RING_ALLREDUCE, 4)
    kw = dict(microbatches=8, mb_window=8, slot_bytes=32768, mb_order=ccl.MB_ALGO)
    st = s.check(65536, F32, fifo_slots=4, **kw)
    assert st.fuse == ccl.FUSE_NONE and st.mb_window == 8
    st = s.check(65536, F32, fifo_slots=9, **kw)
    assert st.mb_window == 8 and st.fuse == ccl.FUSE_FULL


def test_ll_protocol_doubles_fifo_bytes_and_needs_16_byte_chunks():
    s = ccl.Schedule.builtin(ccl.RING_ALLREDUCE, 8)
    simple = s.check(4096, BF16, protocol=ccl.PROTO_SIMPLE, slot_bytes=16384)
    ll = s.check(4096, BF16, protocol=ccl.PROTO_LL, slot_bytes=16384)
    assert ll.protocol == ccl.PROTO_LL and simple.protocol == ccl.PROTO_SIMPLE
    assert ll.fifo_bytes == 2 * simple.fifo_bytes
    assert ll.schedule_bytes == simple.schedule_bytes
    with pytest.raises(ccl.CclError) as e:
        s.check(4093, BF16, protocol=ccl.PROTO_LL)      # 8186-byte chunks
    assert e.value.code == 5
    with pytest.raises(ccl.CclError) as e:
        s.check(4096, BF16, protocol=7)
    assert e.value.code == 1


def test_degenerate_sizes_and_programs():
    """An empty program plans to no threadblock (executing it launches
    nothing); a zero-element chunk is rejected; a one-element chunk plans
    (the element path carries it)."""
    empty = ccl.Schedule.compile([], 2, (1, 1, 0))
    st = empty.check(16, F32)
    assert (st.nthreadblocks, st.nsteps, st.schedule_bytes) == (0, 0, 0)
    s = ccl.Schedule.builtin(ccl.RING_ALLREDUCE, 8)
    with pytest.raises(ccl.CclError) as e:
        s.check(0, F32)
    assert e.value.code == 1
    one = s.check(1, BF16)
    assert one.schedule_bytes == 8 * 8 * (6 * 8 - 4) // 8 * 2   # R N (6 - 4/R), N = 8 chunks of 2 bytes


def test_unknown_plan_option_is_an_error():
    s = ccl.Schedule.builtin(ccl.RING_ALLREDUCE, 8)
    with pytest.raises(TypeError):
        s.check(4096, F32, channel=4)        # misspelt "channels"


def test_engine_option_is_validated():
    s = ccl.Schedule.builtin(ccl.RING_ALLREDUCE, 8)
    assert s.check(4096, F32).engine == ccl.ENGINE_PIPELINED
    st = s.check(4096, F32, engine=ccl.ENGINE_SEQUENTIAL, bulk=1)
    assert st.engine == ccl.ENGINE_SEQUENTIAL and st.schedule_bytes == s.check(4096, F32).schedule_bytes
    with pytest.raises(ccl.CclError) as e:
        s.check(4096, F32, engine=2)
    assert e.value.code == 1
    # LL slots on the sequential engine, also on clusters
    ll = s.check(4096, F32, engine=ccl.ENGINE_SEQUENTIAL, protocol=ccl.PROTO_LL, cluster=4)
    assert (ll.engine, ll.protocol, ll.cluster) == (ccl.ENGINE_SEQUENTIAL, ccl.PROTO_LL, 4)


def test_coordinate_descent_visits_both_protocols():
    seen = set()

    def f(o):
        seen.add(o.protocol)
        return (2.0 if o.protocol == ccl.PROTO_LL else 1.0) * _surface((4, 256, 1 << 16))(o)
    best, bw, n = ccl.tune_search(f)
    assert seen == {ccl.PROTO_SIMPLE, ccl.PROTO_LL}
    assert best.protocol == ccl.PROTO_LL and bw == pytest.approx(2.0)
    assert (best.channels, best.nthreads, best.slot_bytes) == (4, 256, 1 << 16)


def test_coordinate_descent_picks_the_faster_engine():
    def f(o):
        return (1.5 if o.engine == ccl.ENGINE_SEQUENTIAL else 1.0) * _surface((2, 512, 1 << 15))(o)
    best, bw, n = ccl.tune_search(f)
    assert best.engine == ccl.ENGINE_SEQUENTIAL and best.protocol == ccl.PROTO_SIMPLE
    assert bw == pytest.approx(1.5)


def test_balanced_allocation_merges_link_free_threadblocks():
    """Direct copies need no FIFO: a rank's copy threadblocks are binned into
    at most budget / (ranks x channels) threadblocks; bytes and steps keep."""
    counts = datagen.alltoallv_counts(3, 32, 512)
    s = ccl.Schedule.alltoallv(counts)
    kw = dict(link_mode=ccl.LINK_DIRECT, channels=4, channel_scaling=0)
    packed = s.check(1024, BF16, tb_alloc=ccl.TB_PACKED, **kw)
    bal = s.check(1024, BF16, tb_alloc=ccl.TB_BALANCED, tb_budget=256, **kw)
    assert packed.nthreadblocks > 900
    assert bal.nthreadblocks == 256          # 2 per rank x 4 channels x 32 ranks
    assert (bal.schedule_bytes, bal.nsteps) == (packed.schedule_bytes, packed.nsteps)
    assert s.check(1024, BF16, tb_alloc=ccl.TB_BALANCED, tb_budget=512, **kw).nthreadblocks == 512
    # threadblocks with FIFO links are left as packed
    h = ccl.Schedule.builtin(ccl.HIER_ALLREDUCE, 16, 8)
    a = h.check(65536, F32, tb_alloc=ccl.TB_PACKED, microbatches=4)
    b = h.check(65536, F32, tb_alloc=ccl.TB_BALANCED, microbatches=4, tb_budget=16)
    assert a.nthreadblocks == b.nthreadblocks
    with pytest.raises(ccl.CclError):
        s.check(1024, BF16, tb_alloc=3)


def test_coordinate_descent_visits_both_transports():
    seen = set()

    def f(o):
        seen.add((o.link_mode, o.tb_alloc, o.protocol))
        return (1.5 if o.link_mode == ccl.LINK_DIRECT else 1.0) * _surface((8, 512, 1 << 17))(o)
    best, bw, n = ccl.tune_search(f)
    assert {m for m, _, _ in seen} == {ccl.LINK_FIFO, ccl.LINK_DIRECT}
    assert len(seen) == 8
    assert best.link_mode == ccl.LINK_DIRECT and bw == pytest.approx(1.5)


def test_cluster_option_is_validated_and_reported():
    s = ccl.Schedule.builtin(ccl.RING_ALLREDUCE, 8)
    st = s.check(4096, F32, engine=ccl.ENGINE_SEQUENTIAL, cluster=4)
    assert st.cluster == 4 and st.nthreadblocks == 8
    assert s.check(4096, F32).cluster == 1
    for bad in (3, 16, -1):
        with pytest.raises(ccl.CclError) as e:
            s.check(4096, F32, engine=ccl.ENGINE_SEQUENTIAL, cluster=bad)
        assert e.value.code == 1
    with pytest.raises(ccl.CclError) as e:
        s.check(4096, F32, cluster=2)          # pipelined engine
    assert e.value.code == 5


def test_coordinate_descent_tries_clusters_on_the_sequential_engine():
    seen = set()

    def probe(o):
        seen.add((o.engine, o.cluster))
        return 1.0 + (o.cluster if o.engine == ccl.ENGINE_SEQUENTIAL else 0) + 0.001 * o.channels
    best, bw, n = ccl.tune_search(probe)
    assert best.engine == ccl.ENGINE_SEQUENTIAL and best.cluster == 8
    assert all(c in (0, 1) for e, c in seen if e == ccl.ENGINE_PIPELINED)


def test_direct_transport_folds_a_copy_send_and_its_receive():
    """The ring AllGather with copy receives left unchained starts on every
    rank with a copy-send (own block into the own output, and on to the
    next rank). Direct transport folds its receive in: one read written to
    both outputs (3 bytes per element byte) instead of a FIFO hop (3 + 2),
    the other hops plain copies (2): 15 units per rank, no FIFO left. The
    oracle's own count agrees."""
    from oracle import bytes as OB
    from oracle import schedules as OS
    R, ce = 8, 1024
    s = ccl.Schedule.builtin(ccl.RING_ALLGATHER, R, 0, ccl.FLAG_NOCHAIN_COPIES)
    fifo = s.check(ce, F32, link_mode=ccl.LINK_FIFO)
    direct = s.check(ce, F32, link_mode=ccl.LINK_DIRECT, fold=1)
    assert direct.nlinks == 0 and fifo.nlinks == R
    assert direct.schedule_bytes == R * 15 * ce * 4
    assert fifo.schedule_bytes == R * (3 + 7 * 2 + 6 * 2) * ce * 4   # copy-send, 7 receives, 6 sends
    ops, nch = OS.ring_allgather(R)
    assert OB.schedule_bytes(ops, R, nch, ce, F32, fuse="nochain", direct=True, fold=1) == direct.schedule_bytes


def test_fold_option():
    """fold = 0 keeps the copy-send's FIFO hop (and its bytes); values
    outside 0..15 are refused; the library default folds receives."""
    assert ccl.default_opts().fold & 1
    R, ce = 8, 1024
    s = ccl.Schedule.builtin(ccl.RING_ALLGATHER, R, 0, ccl.FLAG_NOCHAIN_COPIES)
    kept = s.check(ce, F32, link_mode=ccl.LINK_DIRECT, fold=0)
    assert kept.nlinks == R and kept.schedule_bytes == R * (3 + 2 + 6 * 2) * ce * 4
    for bad in (-1, 16):
        with pytest.raises(ccl.CclError) as e:
            s.check(ce, F32, link_mode=ccl.LINK_DIRECT, fold=bad)
        assert e.value.code == 1


def test_tuner_keeps_the_starting_fold():
    """The search starts from the caller's options, folds included (not
    reset to the library default): the first probe and every FIFO probe
    carry the caller's fold setting."""
    seen = []

    def probe(o):
        seen.append((o.link_mode, o.fold))
        return 1.0 + 0.001 * o.channels
    start = ccl.default_opts()
    start.fold, start.link_mode = 1, ccl.LINK_FIFO
    ccl.tune_search(probe, start)
    assert seen[0] == (ccl.LINK_FIFO, 1)
    assert {f for m, f in seen if m == ccl.LINK_FIFO} == {1}


def test_coordinate_descent_chooses_the_folds_with_direct_transport():
    """With direct transport the folds are a coordinate (from the caller's
    3 down to 2 here, where the surface peaks); FIFO subspaces keep the
    caller's folds."""
    seen = set()

    def probe(o):
        seen.add((o.link_mode, o.fold))
        return 1.0 + (0.5 if o.link_mode == ccl.LINK_DIRECT and o.fold == 2 else 0) + 0.001 * o.channels
    best, bw, n = ccl.tune_search(probe)
    assert best.link_mode == ccl.LINK_DIRECT and best.fold == 2
    assert {f for m, f in seen if m == ccl.LINK_FIFO} == {ccl.default_opts().fold}
    assert {f for m, f in seen if m == ccl.LINK_DIRECT} >= {2, 3}


def test_direct_transport_folds_copy_chains():
    """fold bit 1: the ring AllGather's chain of 6 direct copies after the
    folded copy-send becomes 3 two-destination copies (3 bytes per element
    byte each instead of 2 + 2), and every threadblock program 4 steps
    instead of 7; the plan's steps and bytes say so, with or without the
    receive fold (bit 0)."""
    R, ce = 8, 1024
    s = ccl.Schedule.builtin(ccl.RING_ALLGATHER, R, 0, ccl.FLAG_NOCHAIN_COPIES)
    units = {0: 3 + 2 + 6 * 2, 1: 3 + 6 * 2, 2: 3 + 2 + 3 * 3, 3: 3 + 3 * 3}
    for fold, u in units.items():
        st = s.check(ce, F32, link_mode=ccl.LINK_DIRECT, fold=fold, microbatches=1)
        assert st.schedule_bytes == R * u * ce * 4, fold
    p1 = s.check(ce, F32, link_mode=ccl.LINK_DIRECT, fold=1, microbatches=1)
    p3 = s.check(ce, F32, link_mode=ccl.LINK_DIRECT, fold=3, microbatches=1)
    assert p1.nsteps == R * 7 and p3.nsteps == R * 4
    # FIFO transport: nothing to fold
    assert s.check(ce, F32, link_mode=ccl.LINK_FIFO, fold=3).schedule_bytes == \
        s.check(ce, F32, link_mode=ccl.LINK_FIFO, fold=0).schedule_bytes


def test_copy_chains_fold_three_hops_per_step():
    """fold bit 3: the ring AllGather's chain of 6 direct copies after the
    folded copy-send becomes 2 three-destination copies: 3 steps per
    program instead of 4 (7 unfolded), 3 + 2 * 4 bytes per element byte of
    a chunk instead of 3 + 3 * 3."""
    R, ce = 8, 1024
    s = ccl.Schedule.builtin(ccl.RING_ALLGATHER, R, 0, ccl.FLAG_NOCHAIN_COPIES)
    p3 = s.check(ce, F32, link_mode=ccl.LINK_DIRECT, fold=3, microbatches=1)
    p11 = s.check(ce, F32, link_mode=ccl.LINK_DIRECT, fold=11, microbatches=1)
    assert p3.nsteps == R * 4 and p11.nsteps == R * 3
    assert p3.schedule_bytes == R * 12 * ce * 4 and p11.schedule_bytes == R * 11 * ce * 4


def test_direct_transport_folds_reduction_chains():
    """fold bit 2: the ReduceScatter's 8-hop chains (send, 6 rrs, rrc) become
    4 steps (send + rrs, rrs + rrs twice, rrs + rrc), run two ranks apart:
    every threadblock program takes 4 steps instead of 8, links go from a
    rank to the rank two ahead, and 15 instead of 23 bytes per element byte
    of a chunk move.  With the LL protocol nothing folds (its slot path
    takes no third operand); FIFO transport folds nothing either."""
    R, ce = 8, 1024
    s = ccl.Schedule.builtin(ccl.RING_REDUCESCATTER, R)
    plain = s.check(ce, F32, link_mode=ccl.LINK_DIRECT, fold=3, microbatches=1)
    folded = s.check(ce, F32, link_mode=ccl.LINK_DIRECT, fold=7, microbatches=1)
    assert plain.schedule_bytes == R * 23 * ce * 4 and folded.schedule_bytes == R * 15 * ce * 4
    assert plain.nsteps == R * 8 and folded.nsteps == R * 4
    assert folded.nthreadblocks == plain.nthreadblocks == R
    ll = s.check(ce, F32, link_mode=ccl.LINK_DIRECT, fold=7, protocol=ccl.PROTO_LL)
    assert ll.schedule_bytes == plain.schedule_bytes
    fifo = s.check(ce, F32, link_mode=ccl.LINK_FIFO, fold=7)
    assert fifo.schedule_bytes == plain.schedule_bytes


def test_reduce_chain_fold_keeps_the_ring_allreduce_on_one_threadblock_per_rank():
    """With every fold on, the ring AllReduce's reduce-scatter pairs run two
    ranks apart and the step that completes a chunk joins the last pair and
    writes the next rank's output itself: still one threadblock per rank and
    channel."""
    R = 8
    s = ccl.Schedule.builtin(ccl.RING_ALLREDUCE, R, 0, ccl.FLAG_NOCHAIN_COPIES)
    for ch in (1, 4):
        st = s.check(1024, F32, link_mode=ccl.LINK_DIRECT, fold=7, channels=ch, tb_alloc=ccl.TB_BALANCED,
                     tb_budget=R * ch)
        assert st.nthreadblocks == R * ch


def test_copy_chain_fold_keeps_dependencies():
    """A folded pair runs at the first copy's time, so everything the second
    copy waited for must be able to come first: a program where a rank
    overwrites the range it forwards between receiving and sending it keeps
    the two copies apart (the oracle agrees on the bytes)."""
    from oracle import bytes as OB
    IN_, OUT_ = 0, 1
    ops = [(0, 0, IN_, 0, 1, OUT_, 0, 1),     # rank 0 -> rank 1
           (0, 1, IN_, 1, 1, OUT_, 0, 1),     # rank 1 overwrites it locally
           (0, 1, OUT_, 0, 2, OUT_, 0, 1)]    # and forwards the new value
    s = ccl.Schedule.compile(ops, 3, (2, 2, 0), fuse=False)
    st = s.check(64, F32, link_mode=ccl.LINK_DIRECT, fold=3)
    assert st.schedule_bytes == OB.schedule_bytes(ops, 3, (2, 2, 0), 64, F32, "none", True, 3)
    assert st.schedule_bytes == (2 + 2 + 2) * 64 * 4
