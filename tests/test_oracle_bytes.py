"""The oracle's byte accounting (``oracle.bytes``), pinned to closed forms
derived by hand from the collective programs and the fused-instruction costs
(copy 2, send 2, recv 2, reduce / rrc / rcs / rrs / copy-send 3, rrcs 4,
recv-send 2 bytes per element byte; with direct transport a plain receive
is written by its sender), then compared with the product's own count for
every benchmark row."""
import numpy as np
import pytest

from oracle import bytes as OB
from oracle import schedules as OS

F32, BF16, F16, I32 = 0, 1, 2, 3


@pytest.mark.parametrize("R", [2, 3, 5, 8])
def test_ring_allreduce_closed_forms(R):
    """Per rank, n = chunk bytes.  Full fusion: send 2 + (R-2) rrs 3 +
    rrcs 4 + (R-2) rcs 3 + recv 2 = 6R - 4.  Copy receives unchained: the
    all-gather is R-1 receives and R-2 sends of 2: 3R + 4R - 6 = 7R - 6.
    Direct transport: the R-2 send/receive pairs between plain ends become
    copies of 2, and a plain receive fed by the rrcs that completes a chunk
    is written by the rrcs itself (its 2 go): unchained 3R + 2 + 2(R-2) - 2
    = 5R - 4; fully fused only at R = 2, where the rrcs feeds the last
    receive directly.  Unfused: R local copies 2, R-1 reduce transfers
    2 + 3, R-1 copy transfers 2 + 2 = 11R - 9."""
    ops, nch = OS.ring_allreduce(R)
    ce, es = 1000, 4
    n = ce * es
    full_direct = 6 * R - 4 - (2 if R == 2 else 0)
    assert OB.schedule_bytes(ops, R, nch, ce, F32, "full", direct=False) == R * (6 * R - 4) * n
    assert OB.schedule_bytes(ops, R, nch, ce, F32, "full", direct=True) == R * full_direct * n
    assert OB.schedule_bytes(ops, R, nch, ce, F32, "nochain", direct=False) == R * (7 * R - 6) * n
    assert OB.schedule_bytes(ops, R, nch, ce, F32, "nochain", direct=True) == R * (5 * R - 4) * n
    assert OB.schedule_bytes(ops, R, nch, ce, F32, "none", direct=False) == R * (11 * R - 9) * n
    # per rank N(6 - 4/R) with N = R n bytes per rank (FIFO transport)
    assert OB.schedule_bytes(ops, R, nch, ce, F32, direct=False) * R == R * R * n * (6 * R - 4)


@pytest.mark.parametrize("R", [2, 4, 8])
def test_allgather_and_reducescatter_closed_forms(R):
    """Per rank, n = S / R: AllGather copy-send 3 + (R-2) rcs 3 + recv 2;
    ReduceScatter send 2 + (R-2) rrs 3 + rrc 3; both 3R - 1.  AllGather
    unfused with direct copies: the local copy and R-1 hops of 2 = 2R."""
    for prog in (OS.ring_allgather, OS.ring_reducescatter):
        ops, nch = prog(R)
        assert OB.schedule_bytes(ops, R, nch, 512, BF16, "full", direct=False) == R * (3 * R - 1) * 1024
    ops, nch = OS.ring_allgather(R)
    assert OB.schedule_bytes(ops, R, nch, 512, BF16, "none", direct=True) == R * 2 * R * 1024


def test_hierarchical_allreduce_closed_form():
    """G = 8, 2 groups, M = 16 n per rank, slices of 2 chunks.  Intra
    reduce-scatter: send 2x2 + 6 rrs 3x2 + rrc 3x2 = 46 n.  The inter-group
    step works on single chunks, which partly overlap the slices, so nothing
    fuses across it: send 2 + rrcs 4 (the reduced chunk is sent back) +
    recv 2 = 8 n.  Intra all-gather: send 2x2 + 6 rcs 3x2 + recv 2x2 = 44 n.
    98 n = 6.125 M."""
    ops, nch = OS.hier_allreduce(8, 2)
    n = 4096 * 4
    assert OB.schedule_bytes(ops, 16, nch, 4096, F32, "full", direct=False) == 16 * 98 * n


def test_two_phase_alltoall_closed_form():
    """R = 32 = 4 x 8, one chunk per block: per rank the own block (local
    copy 2), 7 in-group blocks (transfers 4), 24 blocks to aggregators -- 3
    of them the rank itself (local copies 2), 21 transfers 4 -- and 24
    blocks of phase 2 (transfers 4): 2 + 28 + 6 + 84 + 96 = 216 blocks.
    With direct transport every transfer is a copy of 2: 2 (sent + copied)
    = 2 * (7 + 21 + 24 + 1 + 3) = 112."""
    ops, nch = OS.alltoall_two_phase(8, 4)
    n = 1024 * 2
    assert OB.schedule_bytes(ops, 32, nch, 1024, F16, "full", direct=False) == 32 * 216 * n
    assert OB.schedule_bytes(ops, 32, nch, 1024, F16, "full", direct=True) == 32 * 112 * n


def test_alltonext_closed_forms():
    """R = 24 = 3 x 8, 8 parts of n per rank.  21 in-group pairs of 8 parts:
    transfers of 4 (FIFO) or copies of 2 (direct, unfused).  The 2 pairs
    that leave a group: parts 0 and 7 take 2 hops, parts 1..6 take 3; fused
    through FIFOs a part costs send 2 + a recv-send 2 per relay + recv 2
    (6 and 8), unfused with direct copies 2 per hop (4 and 6)."""
    ops, nch = OS.alltonext(8, 3)
    n = 1000 * 4
    assert OB.schedule_bytes(ops, 24, nch, 1000, F32, "full", direct=False) == (21 * 8 * 4 + 2 * (2 * 6 + 6 * 8)) * n
    assert OB.schedule_bytes(ops, 24, nch, 1000, F32, "none", direct=True) == (21 * 8 * 2 + 2 * (2 * 4 + 6 * 6)) * n


@pytest.mark.parametrize("R", [2, 3, 4, 7, 8])
def test_copy_chain_folds_closed_forms(R):
    """Direct transport with copy chains folded (fold bit 1): a copy that
    sends on exactly what another direct copy delivered is written by that
    copy's pass, one read written twice (3) instead of 2 + 2; a chain of k
    hops from its head becomes floor(k/2) such pairs and, for odd k, one
    plain copy.  Ring AllGather, copy receives unchained: the copy-send 3
    (its receive folded by bit 0, else a FIFO receive 2 more), then a chain
    of R - 2 copies.  Ring AllReduce likewise: reduce-scatter 3R (send 2,
    R - 2 rrs 3, rrcs 4; its receive folded by bit 0, else 2 more) and a
    chain of R - 2 all-gather copies."""
    chain = 3 * ((R - 2) // 2) + 2 * ((R - 2) % 2)
    n = 100 * 2
    ops, nch = OS.ring_allgather(R)
    for fold, first in ((2, 3 + 2), (3, 3)):
        assert OB.schedule_bytes(ops, R, nch, 100, BF16, "nochain", True, fold) == R * (first + chain) * n
    ops, nch = OS.ring_allreduce(R)
    for fold, rs in ((2, 3 * R + 2), (3, 3 * R)):
        assert OB.schedule_bytes(ops, R, nch, 100, BF16, "nochain", True, fold) == R * (rs + chain) * n


@pytest.mark.parametrize("R", [2, 3, 4, 5, 8, 9])
def test_copy_chain_folds_three_hops_per_step(R):
    """fold bit 3: a chain of k direct copies groups into floor(k/3) steps of
    one read written three times (4 instead of 2 + 2 + 2) and, for k mod 3
    = 2, a pair (3) or, for k mod 3 = 1, a single copy (2).  Ring AllGather,
    copy receives unchained, with the copy-send's receive folded (3): a
    chain of R - 2 copies."""
    k = R - 2
    chain = 4 * (k // 3) + {0: 0, 1: 2, 2: 3}[k % 3]
    ops, nch = OS.ring_allgather(R)
    n = 100 * 2
    assert OB.schedule_bytes(ops, R, nch, 100, BF16, "nochain", True, 11) == R * (3 + chain) * n
    assert OB.schedule_bytes(ops, R, nch, 100, BF16, "nochain", True, 15) == R * (3 + chain) * n


def test_copy_chain_folds_of_the_hierarchical_allreduce_and_alltonext():
    """Hierarchical AllReduce (G = 8, 2 groups, copy receives unchained,
    direct): intra reduce-scatter 46 n as above, the inter-group step send 2
    + rrcs 4 + its receive 2 (folded by bit 0: 6), the intra all-gather of
    2-chunk slices 7 copies of 4 n -- with chains folded three pairs of 6 n
    and one copy of 4 n, 22 n.  AllToNext unfused, direct: a part relayed
    once costs 3 instead of 4, one relayed twice 3 + 2 instead of 6."""
    ops, nch = OS.hier_allreduce(8, 2)
    n = 64 * 4
    for fold, per_rank in ((0, 46 + 8 + 28), (1, 46 + 6 + 28), (2, 46 + 8 + 22), (3, 46 + 6 + 22)):
        assert OB.schedule_bytes(ops, 16, nch, 64, F32, "nochain", True, fold) == 16 * per_rank * n
    ops, nch = OS.alltonext(8, 3)
    n = 1000 * 4
    assert OB.schedule_bytes(ops, 24, nch, 1000, F32, "none", True, 2) == (21 * 8 * 2 + 2 * (2 * 3 + 6 * 5)) * n


def test_planted_mistake_in_the_chain_fold_is_caught():
    """Folding a copy chain without the head rule (every hop into its
    predecessor, so the 7-hop all-gather of the ring AllGather at R = 8
    would count 3 + 6 * 1 extra writes instead of pairs) breaks the pin."""
    ops, nch = OS.ring_allgather(8)
    good = OB.schedule_bytes(ops, 8, nch, 10, F32, "nochain", True, 3)
    saved = OB._chain_folds
    try:
        OB._chain_folds = lambda halves, depth=2: 2 * saved(halves, depth)
        assert OB.schedule_bytes(ops, 8, nch, 10, F32, "nochain", True, 3) != good
    finally:
        OB._chain_folds = saved


@pytest.mark.parametrize("R", [2, 3, 5, 8])
def test_reduce_chain_folds_closed_forms(R):
    """Direct transport with reduction chains folded (fold bit 2): a send or
    recv-reduce-send and the receive-reduce its slot feeds become one step
    that reads the second rank's local operand itself; the slot between them
    (written 1, read 1) goes.  A chain of k hops pairs up from its head,
    floor(k/2) pairs.  ReduceScatter (R hops per chunk): 3R - 1 - 2
    floor(R/2).  Ring AllReduce, copy receives unchained, all folds (7):
    the reduce-scatter 3R - 2 floor(R/2); the receive its last step feeds
    is folded into that step (bit 0), paired or not; then the all-gather's
    R - 2 copies fold in pairs (3 per pair, 2 for an odd one out)."""
    n = 64 * 4
    ops, nch = OS.ring_reducescatter(R)
    assert OB.schedule_bytes(ops, R, nch, 64, F32, "full", True, 4) == R * (3 * R - 1 - 2 * (R // 2)) * n
    ops, nch = OS.ring_allreduce(R)
    ag = 3 * ((R - 2) // 2) + 2 * ((R - 2) % 2)
    want = 3 * R - 2 * (R // 2) + ag
    assert OB.schedule_bytes(ops, R, nch, 64, F32, "nochain", True, 7) == R * want * n


def test_reduce_chain_folds_of_the_hierarchical_allreduce():
    """G = 8, 2 groups, copy receives unchained, direct.  The in-group
    reduce-scatter's 8 hops of 2-chunk slices (46 n) fold into 4 pairs (16 n
    less: 30 n); the inter-group send and the recv-reduce-copy-send it feeds
    become one step (4 n instead of 6 n), whose receive keeps its FIFO (2
    n) unless receives fold as well (bit 0): 6 n or 4 n; the in-group
    all-gather 28 n, or 22 n with copy chains folded."""
    ops, nch = OS.hier_allreduce(8, 2)
    n = 64 * 4
    for fold, per_rank in ((4, 30 + 6 + 28), (5, 30 + 4 + 28), (6, 30 + 6 + 22), (7, 30 + 4 + 22)):
        assert OB.schedule_bytes(ops, 16, nch, 64, F32, "nochain", True, fold) == 16 * per_rank * n


def test_planted_mistake_in_the_reduce_chain_fold_is_caught():
    """Counting every reduction hop as folded into its predecessor (no head
    rule) breaks the ReduceScatter pin."""
    ops, nch = OS.ring_reducescatter(8)
    good = OB.schedule_bytes(ops, 8, nch, 10, F32, "full", True, 4)
    saved = OB._reduce_chain_folds
    try:
        def every_hop(halves):
            s, taken = saved(halves)
            return 2 * s, taken
        OB._reduce_chain_folds = every_hop
        assert OB.schedule_bytes(ops, 8, nch, 10, F32, "full", True, 4) != good
    finally:
        OB._reduce_chain_folds = saved


def test_min_bytes_closed_forms():
    """Every input chunk a program reads, read once, and every output chunk
    it writes, written once: AllReduce R (R + R) chunks, AllGather R (1 +
    R), AllToNext without wrap 23 senders and 23 receivers of 8 chunks."""
    ops, nch = OS.ring_allreduce(8)
    assert OB.min_bytes(ops, 8, nch, 100, F32) == 2 * 8 * 8 * 100 * 4
    ops, nch = OS.ring_allgather(8)
    assert OB.min_bytes(ops, 8, nch, 100, BF16) == (8 * 1 + 8 * 8) * 100 * 2
    ops, nch = OS.alltonext(8, 3)          # rank 23 sends nothing, rank 0 receives nothing
    assert OB.min_bytes(ops, 24, nch, 100, F32) == 2 * 23 * 8 * 100 * 4


def test_planted_mistake_in_a_factor_is_caught():
    """A wrong cost for one fused kind (a receive-reduce-copy-send counted as
    3 instead of 4) breaks the ring closed form."""
    ops, nch = OS.ring_allreduce(8)
    saved = OB.FACTOR["rrcs"]
    try:
        OB.FACTOR["rrcs"] = 3
        assert OB.schedule_bytes(ops, 8, nch, 10, F32, "full", direct=False) != 8 * (6 * 8 - 4) * 40
    finally:
        OB.FACTOR["rrcs"] = saved


# ------------------------------------------------- against the product count

ccl = pytest.importorskip("collective_communication_schedule_gb300")

KIND_PROGRAM = {0: lambda R, G: OS.ring_allreduce(R), 1: lambda R, G: OS.ring_allgather(R),
                2: lambda R, G: OS.ring_reducescatter(R), 3: lambda R, G: OS.hier_allreduce(G, R // G),
                4: lambda R, G: OS.alltoall_two_phase(G, R // G), 5: lambda R, G: OS.alltonext(G, R // G)}


def _fuse_name(flags):
    return "none" if flags & ccl.FLAG_NOFUSE else ("nochain" if flags & ccl.FLAG_NOCHAIN_COPIES else "full")


def test_oracle_count_equals_the_product_count_for_every_benchmark_row():
    import bench

    class A:
        only, scale = "", 1.0
    assert bench.DEFAULT_LINK_MODE == ccl.default_opts().link_mode
    assert bench.DEFAULT_FOLD == ccl.default_opts().fold
    for name, kind, R, G, dt, cb, dist, seed, opts in bench.selected_suite(A):
        sched, popts = bench.schedule_and_opts(ccl, kind, R, G, opts)
        ce = cb // bench.ESIZE[dt]
        st = sched.check(ce, dt, **popts)
        # the count the CPU baseline and the reference arm use
        assert bench.oracle_bytes(kind, R, G, dt, ce, opts) == (st.schedule_bytes, st.min_bytes), name
        fl = {"nochain": ccl.FLAG_NOCHAIN_COPIES, False: ccl.FLAG_NOFUSE}.get(opts.get("fuse", True), 0)
        ops, nch = KIND_PROGRAM[kind](R, G)
        direct = popts.get("link_mode", ccl.default_opts().link_mode) == ccl.LINK_DIRECT
        fold = int(popts.get("fold", ccl.default_opts().fold))
        assert OB.schedule_bytes(ops, R, nch, ce, dt, _fuse_name(fl), direct, fold) == st.schedule_bytes, name


@pytest.mark.parametrize("kind,R,G", [(0, 8, 0), (0, 3, 0), (1, 8, 0), (2, 5, 0), (3, 16, 8), (3, 4, 2),
                                      (4, 32, 8), (4, 8, 4), (5, 24, 8), (5, 6, 3)])
@pytest.mark.parametrize("flags", [0, 2, 4])
@pytest.mark.parametrize("link_mode,fold", [(0, 1), (1, 1), (1, 0), (1, 2), (1, 3), (1, 4), (1, 5), (1, 6), (1, 7),
                                            (1, 10), (1, 15)])
def test_oracle_count_equals_the_product_count_for_builtins(kind, R, G, flags, link_mode, fold):
    ops, nch = KIND_PROGRAM[kind](R, G)
    st = ccl.Schedule.builtin(kind, R, G, flags).check(333, F32, link_mode=link_mode, fold=fold)
    assert OB.schedule_bytes(ops, R, nch, 333, F32, _fuse_name(flags), link_mode == 1, fold) == \
        st.schedule_bytes


def test_oracle_fused_kinds_equal_the_compiled_kinds():
    """Instruction by instruction: the fused kinds the oracle derives for the
    benchmark collectives are the kinds the compiler emits."""
    for kind, R, G in [(0, 8, 0), (1, 8, 0), (2, 8, 0), (3, 16, 8), (4, 32, 8), (5, 24, 8)]:
        ops, _ = KIND_PROGRAM[kind](R, G)
        for flags in (0, 2, 4):
            mine = sorted(k for k, *_ in OB.fused_instructions(ops, R, _fuse_name(flags)))
            theirs = sorted(ccl.KIND_NAMES[i["kind"]] for i in ccl.Schedule.builtin(kind, R, G, flags).instrs())
            assert mine == theirs, (kind, flags)
