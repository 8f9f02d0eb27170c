"""Exhaustive interleaving explorer for tiny chunk programs.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).  Pure Python, meant
for R <= 4 ranks and a handful of chunks.

Model (MSCCLang report, §III.1: the compiler lowers a copy/reduce between two
ranks into a send on the source and a receive (or receive-reduce) on the
destination; §I "goals": the system must rule out deadlock and data races).
Every rank runs its own part of the program in program order:

* an operation local to rank r is one step of rank r;
* an operation from rank a to rank b is a *send* step of a, which pushes the
  source values into the link FIFO (a -> b), and a *receive* step of b, which
  pops them and copies or reduces them into the destination.

A link FIFO holds at most ``K`` messages; a send blocks while it is full, a
receive while it is empty.  The explorer visits every reachable state
(memoised) and reports the set of distinct final outputs and the number of
stuck states (deadlocks).

Values are symbolic: an input element is a leaf, a reduce forms the
unordered pair of its operands (addition commutes bit for bit, but not
associates), so two runs give the same symbolic result exactly when every
floating-point sum is formed in the same association order.
"""
from __future__ import annotations

import sys

COPY, REDUCE = 0, 1
IN, OUT, SCR = 0, 1, 2


class _Interner:
    def __init__(self):
        self.ids = {}
        self.exprs = []

    def get(self, e):
        i = self.ids.get(e)
        if i is None:
            i = len(self.exprs)
            self.ids[e] = i
            self.exprs.append(e)
        return i

    def add(self, a, b):
        return self.get(("+", min(a, b), max(a, b)))

    def render(self, i):
        e = self.exprs[i]
        if e[0] == "+":
            return f"({self.render(e[1])}+{self.render(e[2])})"
        return f"{e[0]}{e[1]}.{e[2]}" + (f".{e[3]}" if len(e) > 3 else "")


def _rank_programs(ops, nranks):
    progs = [[] for _ in range(nranks)]
    for i, o in enumerate(ops):
        op, sr, sb, so, dr, db, do, cnt = (int(v) for v in o)
        if sr == dr:
            progs[sr].append(("local", i))
        else:
            progs[sr].append(("send", i))
            progs[dr].append(("recv", i))
    return progs


def explore(ops, nranks, nchunks, K=1, progs=None, max_states=2_000_000):
    """Returns dict(outputs=set_of_output_tuples, deadlocks=int, states=int,
    interner=_Interner).

    ``progs`` optionally replaces the program-order lowering with explicit
    per-rank step lists of ``("local"|"send"|"recv", op_index)``; with the
    program-order lowering a deadlock cannot occur (executing the operations
    one by one in program order is always one available interleaving), so
    explicit step lists are how a reordered lowering is checked."""
    ops = [tuple(int(v) for v in o) for o in ops]
    if progs is None:
        progs = _rank_programs(ops, nranks)
    it = _Interner()
    # buffers: per (rank, kind) a tuple of element ids (1 element per chunk)
    bufs0 = []
    for r in range(nranks):
        for kind in (IN, OUT, SCR):
            if kind == IN:
                bufs0.append(tuple(it.get(("x", r, k)) for k in range(nchunks[kind])))
            else:
                bufs0.append(tuple(it.get(("s", r, k, kind)) for k in range(nchunks[kind])))
    links = {}
    for o in ops:
        if o[1] != o[4]:
            links.setdefault((o[1], o[4]), len(links))
    nl = len(links)

    def bi(r, kind):
        return 3 * r + kind

    start = (tuple([0] * nranks), tuple(() for _ in range(nl)), tuple(bufs0))
    seen = set()
    outputs = set()
    deadlocks = 0
    stack = [start]
    sys.setrecursionlimit(10000)
    while stack:
        st = stack.pop()
        if st in seen:
            continue
        seen.add(st)
        if len(seen) > max_states:
            raise RuntimeError("state space too large for the explorer")
        pcs, fifos, bufs = st
        if all(pcs[r] == len(progs[r]) for r in range(nranks)):
            outputs.add(tuple(bufs[bi(r, OUT)] for r in range(nranks)))
            continue
        moved = False
        for r in range(nranks):
            if pcs[r] == len(progs[r]):
                continue
            kind, oi = progs[r][pcs[r]]
            op, sr, sb, so, dr, db, do, cnt = ops[oi]
            nb = None
            nf = None
            if kind == "local":
                src = bufs[bi(sr, sb)][so:so + cnt]
                dst = list(bufs[bi(dr, db)])
                for k in range(cnt):
                    dst[do + k] = src[k] if op == COPY else it.add(dst[do + k], src[k])
                nb = list(bufs)
                nb[bi(dr, db)] = tuple(dst)
            elif kind == "send":
                li = links[(sr, dr)]
                if len(fifos[li]) >= K:
                    continue
                msg = (oi, bufs[bi(sr, sb)][so:so + cnt])
                nf = list(fifos)
                nf[li] = fifos[li] + (msg,)
            else:
                li = links[(sr, dr)]
                if not fifos[li]:
                    continue
                (moi, vals), rest = fifos[li][0], fifos[li][1:]
                if moi != oi:
                    raise AssertionError(f"link {sr}->{dr}: received op {moi}, expected {oi}")
                dst = list(bufs[bi(dr, db)])
                for k in range(cnt):
                    dst[do + k] = vals[k] if op == COPY else it.add(dst[do + k], vals[k])
                nb = list(bufs)
                nb[bi(dr, db)] = tuple(dst)
                nf = list(fifos)
                nf[li] = rest
            npcs = list(pcs)
            npcs[r] += 1
            stack.append((tuple(npcs), tuple(nf) if nf is not None else fifos,
                          tuple(nb) if nb is not None else bufs))
            moved = True
        if not moved:
            deadlocks += 1
    return {"outputs": outputs, "deadlocks": deadlocks, "states": len(seen), "interner": it}
