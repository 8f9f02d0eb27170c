"""Schedule bytes of a chunk program, counted by fused-instruction semantics.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).  Nothing here is
shared with ``collective_communication_schedule_gb300``; the benchmark's CPU
baseline and reference arm take their byte counts from here.

The MSCCLang report (§III.1, "instruction generation" and "instruction
fusion") lowers every cross-rank copy or reduce into a send on the source
rank and a receive (or receive-reduce) on the destination rank, and fuses a
receive with the send that forwards its value into one compound instruction
(recv-copy-send, recv-reduce-send, recv-reduce-copy-send, ...) so that the
forwarded value is not read back from memory.  The bytes an instruction moves
(§8(d) accounting, per element byte of its range) are its buffer and FIFO
slot reads plus writes:

    copy 2   reduce 3   send 2   recv 2   recv-reduce-copy 3
    recv-copy-send 3   recv-send 2   recv-reduce-send 3
    recv-reduce-copy-send 4   copy-send 3

Fusion (reading c-12: only exact chunk ranges fuse; a partial overlap never
does), applied per rank in program order until nothing changes:

* a local copy whose value is next used only as the local operand of a
  reduce is folded into that reduce (the reduce reads the copy's source);
* a send of a value a local copy just made reads the copy's source instead
  (the copy disappears when nothing else needs its value), or the two
  become one copy-send;
* a received (or received-and-reduced) value that is sent on is sent from
  the receiving instruction (recv-copy-send / recv-reduce-copy-send); its
  buffer write is dropped when nothing else reads the value and it does not
  survive in an input or output buffer (recv-send / recv-reduce-send).  In
  "nochain" mode only received-and-reduced values are chained this way.

Direct transport (the plan option): a plain send whose transfer ends in a
plain receive is one copy into the receiver's buffer (2 bytes per element
byte instead of 2 + 2), and with copy chains folded a copy that sends on
exactly what another one delivered is written by that one's pass too (3
instead of 2 + 2); with reduction chains folded, two consecutive steps of a
reduction chain are one step that reads the second rank's local operand
itself (the slot between them, 2, goes).  Channels and micro-batches split
ranges without changing these totals.
"""
from __future__ import annotations

import numpy as np

COPY, REDUCE = 0, 1
IN, OUT, SCR = 0, 1, 2
ESIZE = {0: 4, 1: 2, 2: 2, 3: 4}

FACTOR = {"copy": 2, "reduce": 3, "send": 2, "recv": 2, "rrc": 3, "rcs": 3, "fwd": 2, "rrs": 3, "rrcs": 4,
          "copy_send": 3}


class _Half:
    """One instruction on one rank: what it reads (src, loc), writes (dst),
    receives and sends.  Ranges are (rank, buf, off, count) tuples."""

    def __init__(self, rank, pos, count, src=None, loc=None, dst=None, recv=None, send=None, recv_reduce=False,
                 local_reduce=False):
        self.rank, self.pos, self.count = rank, pos, count
        self.src, self.loc, self.dst = src, loc, dst
        self.recv, self.send = recv, send
        self.recv_reduce, self.local_reduce = recv_reduce, local_reduce
        self.alive = True

    def kind(self):
        if self.recv is None and self.send is None:
            return "reduce" if self.local_reduce else "copy"
        if self.recv is None:
            return "copy_send" if self.dst else "send"
        if self.send is None:
            return "rrc" if self.recv_reduce else "recv"
        if self.recv_reduce:
            return "rrcs" if self.dst else "rrs"
        return "rcs" if self.dst else "fwd"


def _overlap(a, b):
    return a is not None and b is not None and a[0] == b[0] and a[1] == b[1] and \
        a[2] < b[2] + b[3] and b[2] < a[2] + a[3]


def _lower(ops):
    halves = []
    for pos, (op, sr, sb, so, dr, db, do, cnt) in enumerate(np.asarray(ops).reshape(-1, 8).tolist()):
        src, dst = (sr, sb, so, cnt), (dr, db, do, cnt)
        if sr == dr:
            halves.append(_Half(sr, pos, cnt, src=src, dst=dst, loc=dst if op == REDUCE else None,
                                local_reduce=op == REDUCE))
        else:
            halves.append(_Half(sr, pos, cnt, src=src, send=pos))
            halves.append(_Half(dr, pos, cnt, dst=dst, loc=dst if op == REDUCE else None, recv=pos,
                                recv_reduce=op == REDUCE))
    return halves


def _readers(rank_halves, w):
    """Exact readers of the value half ``w`` writes, up to its overwrite;
    whether another access to it is partial, and whether it survives."""
    D = w.dst
    readers, partial, overwritten = [], False, False
    after = False
    for x in rank_halves:
        if x is w:
            after = True
            continue
        if not after or not x.alive:
            continue
        reads = [r for r in (x.src, x.loc) if _overlap(r, D)]
        if any(r != D for r in reads):
            partial = True
        if any(r == D for r in reads):
            readers.append(x)
        if _overlap(x.dst, D):
            if x.dst == D:
                overwritten = True
            else:
                partial = True
            break
    survives = partial or (not overwritten and D[1] != SCR)
    return readers, partial, survives


def _unchanged(rank_halves, A, p0, p1):
    return not any(x.alive and p0 < x.pos <= p1 and _overlap(x.dst, A) for x in rank_halves)


def _pure_copy(h):
    return h.recv is None and h.send is None and not h.local_reduce and h.src is not None and h.dst is not None


def _plain_send(h):
    return h.send is not None and h.recv is None and not h.local_reduce and h.dst is None and h.src is not None


def fused_instructions(ops, nranks, fuse="full"):
    """The fused instruction kinds of ``ops`` as (kind, rank, count, sent,
    received) tuples; ``fuse``: "full", "nochain" or "none"."""
    return [(h.kind(), h.rank, h.count, h.send, h.recv) for h in _fused_halves(ops, nranks, fuse)]


def _fused_halves(ops, nranks, fuse):
    halves = _lower(ops)
    if fuse != "none":
        changed = True
        while changed:
            changed = False
            for r in range(nranks):
                mine = sorted((h for h in halves if h.alive and h.rank == r), key=lambda h: h.pos)
                for w in mine:
                    if not w.alive or w.dst is None:
                        continue
                    readers, partial, survives = _readers(mine, w)
                    # a local copy folded into the reduce that uses it
                    if _pure_copy(w) and not partial and len(readers) == 1:
                        x = readers[0]
                        if x.loc == w.dst and x.src != w.dst and _unchanged(mine, w.src, w.pos, x.pos):
                            x.loc = w.src
                            if not survives:
                                w.alive = False
                            changed = True
                            break
                    # a send of a copied value
                    if _pure_copy(w):
                        done = False
                        for x in readers:
                            if not _plain_send(x) or x.src != w.dst or not _unchanged(mine, w.src, w.pos, x.pos):
                                continue
                            if len(readers) == 1 and not survives:
                                x.src = w.src
                                w.alive = False
                            else:
                                w.send, x.alive = x.send, False
                            done = True
                            break
                        if done:
                            changed = True
                            break
                    # a received value sent on
                    if w.recv is not None and w.send is None and (fuse == "full" or w.recv_reduce):
                        done = False
                        for x in readers:
                            if not _plain_send(x) or x.src != w.dst:
                                continue
                            w.send, x.alive = x.send, False
                            if len(readers) == 1 and not survives:
                                w.dst = None
                            done = True
                            break
                        if done:
                            changed = True
                            break
                if changed:
                    break
    return [h for h in halves if h.alive]


def _chain_folds(halves, depth=2):
    """Element chunks saved by folding copy chains under direct transport.

    A direct copy is a plain send whose transfer ends in a plain receive.
    When a later direct copy sends on, unchanged, exactly the range an
    earlier one received, the earlier copy's pass writes both destinations:
    one read written twice (3) instead of 2 + 2; with ``depth`` 3 the copy
    that forwards that second destination joins too (one read written three
    times, 4 instead of 2 + 2 + 2).  A step holds at most ``depth``
    destinations and each copy it takes over saves 1; the transfers are
    visited in program order, so a chain groups up from its head.  A copy
    taken over must not write over the step's other ranges."""
    sends = {h.send: h for h in halves if h.send is not None}
    recvs = {h.recv: h for h in halves if h.recv is not None}
    direct = sorted(t for t, h in sends.items() if h.kind() == "send" and recvs[t].kind() == "recv")
    by_rank = {}
    for h in sorted(halves, key=lambda h: h.pos):
        by_rank.setdefault(h.rank, []).append(h)
    gone, saved = set(), 0
    for t1 in direct:
        if t1 in gone:
            continue
        s1, last = sends[t1], recvs[t1]
        ranges = [s1.src, last.dst]
        for _ in range(depth - 1):
            found = None
            for t2 in direct:
                if t2 <= t1 or t2 in gone:
                    continue
                s2, r2 = sends[t2], recvs[t2]
                if s2.rank != last.rank or s2.src != last.dst or s2.count != last.count:
                    continue
                if any(_overlap(r2.dst, r) for r in ranges):
                    continue
                if not _unchanged(by_rank[last.rank], last.dst, last.pos, s2.pos):
                    continue
                found = t2
                break
            if found is None:
                break
            gone.add(found)
            saved += last.count
            last = recvs[found]
            ranges.append(last.dst)
    return saved


def _reduce_chain_folds(halves):
    """Element chunks saved by folding reduction chains under direct
    transport, and the receive-reduce halves taken into a pair.

    A send or recv-reduce-send whose transfer ends in a receive-reduce
    (recv-reduce-send, -copy or -copy-send) becomes one step with it: the
    first rank's pass reads the second rank's local operand itself and adds
    it after its own sum, so the slot between them -- written once, read
    once, 2 per element byte -- goes.  A step that has taken one over takes
    no other, and one taken over is gone; transfers are visited in program
    order, so each chain pairs up from its head."""
    sends = {h.send: h for h in halves if h.send is not None}
    recvs = {h.recv: h for h in halves if h.recv is not None}
    taken, merged, saved = set(), set(), 0
    for t in sorted(sends):
        x = sends[t]
        if id(x) in taken or id(x) in merged or x.kind() not in ("send", "rrs"):
            continue
        y = recvs.get(t)
        if y is None or id(y) in taken or id(y) in merged or y.kind() not in ("rrs", "rrc", "rrcs"):
            continue
        if y.count != x.count:
            continue
        taken.add(id(y))
        merged.add(id(x))
        saved += 2 * x.count
    return saved, taken


def schedule_bytes(ops, nranks, nchunks, chunk_elems, dtype, fuse="full", direct=True, fold=1):
    """Bytes one execution reads and writes (buffers and FIFO slots) when
    ``ops`` runs as fused instructions; ``direct``: a plain receive whose
    sender is a plain send, a copy-send or a recv-reduce-copy-send takes no
    FIFO: the sender writes the receiver's buffer itself (send 2 + receive
    2 -> one copy of 2; copy-send 3 + receive 2 -> one read written twice,
    3; recv-reduce-copy-send 4 + receive 2 -> 4).  ``fold`` bit 0 (True)
    takes the last two without their FIFO (cleared: they keep it); bit 1
    also folds copy chains two hops per step (``_chain_folds``), bit 3
    three; bit 2 reduction chains
    (``_reduce_chain_folds``; the receive fed by a recv-reduce-copy-send
    taken into a pair is folded into the pair's step the same way)."""
    halves = _fused_halves(ops, nranks, fuse)
    units = sum(FACTOR[h.kind()] * h.count for h in halves)
    if direct:
        if int(fold) & 4:
            units -= _reduce_chain_folds(halves)[0]
        sender = {h.send: h for h in halves if h.send is not None}
        for h in halves:
            if h.kind() != "recv":
                continue
            s = sender[h.recv]
            # (a recv-reduce-copy-send taken into a reduction pair still
            # writes the receiver's buffer itself)
            if s.kind() == "send" or (int(fold) & 1 and s.kind() in ("copy_send", "rrcs")):
                units -= 2 * h.count
        if int(fold) & 10:
            units -= _chain_folds(halves, 3 if int(fold) & 8 else 2)
    return units * int(chunk_elems) * ESIZE[dtype]


def min_bytes(ops, nranks, nchunks, chunk_elems, dtype):
    """Each input chunk a program reads read once, each output chunk it
    writes written once."""
    read, written = set(), set()
    for op, sr, sb, so, dr, db, do, cnt in np.asarray(ops).reshape(-1, 8).tolist():
        if sb == IN:
            read.update((sr, so + k) for k in range(cnt))
        if db == OUT:
            written.update((dr, do + k) for k in range(cnt))
    return (len(read) + len(written)) * int(chunk_elems) * ESIZE[dtype]
