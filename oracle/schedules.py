"""The oracle's own generators of collective chunk programs.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Each generator returns ``(ops, nchunks)`` where ``ops`` is an ``(n, 8)`` int32
array of ``[op, src_rank, src_buf, src_off, dst_rank, dst_buf, dst_off, count]``
rows (chunk units, program order) and ``nchunks = (in, out, scratch)`` chunks
per rank.  The programs are written the way a chunk-oriented DSL program is
written (MSCCLang report, §III.1): ``copy`` moves a chunk range, ``reduce``
adds a source range into a destination range, and the order of the list is
the program order from which dependencies are traced.

Readings (the pages name these algorithms but do not spell them out):

* ring (MSCCLang report, §II "test cases: ring AllReduce", §IV.1): rank r
  sends to r+1 mod R.  In the reduce-scatter phase chunk c starts at rank
  c+1 and ends at rank c, so the sum for chunk c is the left fold
  in[c+1] + in[c+2] + ... + in[c] (indices mod R), one rounding per hop.
  The all-gather phase then circulates chunk c starting at rank c.
* hierarchical AllReduce (MSCCLang report, §IV.2; HetCCL summary,
  "hierarchical algorithms and pipelined execution"): intra-group ring
  reduce-scatter, then for every slice a ring AllReduce across groups among
  the ranks holding that slice (same local index), then intra-group ring
  all-gather.
* two-phase AllToAll (MSCCLang report, §IV.3): blocks for another group are
  first gathered on the in-group aggregator whose local index equals the
  destination's local index, then sent to the destination as one batch.
* AllToNext (MSCCLang report, §II and §IV.4): rank r sends its buffer to
  r+1; a transfer that leaves a group is split into G parts, part j relayed
  through local rank j of the source group and local rank j of the
  destination group, so that every link of the two groups carries a share.
  No wrap-around unless ``wrap`` is set.
* hierarchical AllGather (HetCCL summary, "hierarchical algorithm design
  and pipelined execution": an in-cluster step, a cross-cluster step, a
  final in-cluster step, the cross-cluster transfers overlapping the
  in-cluster work): groups of G ranks stand for the clusters.  (1) ring
  AllGather of a group's own blocks inside the group; (2) rank (g, i)
  copies its block to local rank i of every other group -- it reads only
  the input, so it runs beside (1); (3) inside group h every block received
  in (2) circulates the group ring starting from the rank that received it.
  Every block crosses into each other group exactly once.
* uneven AllToAll (per-pair sizes, the token exchange of a mixture-of-
  experts layer; a variant of the AllToAll of the MSCCLang report, §IV.3):
  rank s lays out its blocks by destination, rank d receives them ordered by
  source; every pair is one direct copy.
"""
from __future__ import annotations

import numpy as np

COPY, REDUCE = 0, 1
IN, OUT, SCR = 0, 1, 2


def _arr(ops):
    if not ops:
        return np.zeros((0, 8), np.int32)
    return np.asarray(ops, dtype=np.int32).reshape(-1, 8)


def ring_allreduce(R: int):
    """out[r] = sum_k in[k]; chunk c folded from rank c+1 around to rank c."""
    ops = []
    for r in range(R):
        for c in range(R):
            ops.append((COPY, r, IN, c, r, OUT, c, 1))
    for s in range(R - 1):                       # reduce-scatter steps
        for c in range(R):
            src, dst = (c + 1 + s) % R, (c + 2 + s) % R
            ops.append((REDUCE, src, OUT, c, dst, OUT, c, 1))
    for s in range(R - 1):                       # all-gather steps
        for c in range(R):
            src, dst = (c + s) % R, (c + s + 1) % R
            ops.append((COPY, src, OUT, c, dst, OUT, c, 1))
    return _arr(ops), (R, R, 0)


def ring_allgather(R: int):
    """out[r] = concat_s in[s] (input = 1 chunk, output = R chunks)."""
    ops = [(COPY, r, IN, 0, r, OUT, r, 1) for r in range(R)]
    for s in range(R - 1):
        for c in range(R):
            src, dst = (c + s) % R, (c + s + 1) % R
            ops.append((COPY, src, OUT, c, dst, OUT, c, 1))
    return _arr(ops), (1, R, 0)


def ring_reducescatter(R: int):
    """out[r] = chunk r of sum_k in[k] (input = R chunks, output = 1 chunk).

    The running partial of chunk c sits in scratch chunk c of the rank that
    holds it, and in the output of rank c at the last hop."""
    if R == 1:
        return _arr([(COPY, 0, IN, 0, 0, OUT, 0, 1)]), (1, 1, 0)
    ops = []
    for s in range(R - 1):
        for c in range(R):
            src, dst = (c + 1 + s) % R, (c + 2 + s) % R
            sbuf, soff = (IN, c) if s == 0 else (SCR, c)
            dbuf, doff = (OUT, 0) if s == R - 2 else (SCR, c)
            ops.append((COPY, dst, IN, c, dst, dbuf, doff, 1))
            ops.append((REDUCE, src, sbuf, soff, dst, dbuf, doff, 1))
    return _arr(ops), (R, 1, R)


def hier_allreduce(G: int, ng: int):
    """R = G*ng ranks; buffer = G slices of ng chunks (slice i = chunks
    [i*ng, (i+1)*ng)).  Intra ring RS leaves slice i on local rank i; ring
    AllReduce of slice i across the ng ranks g*G+i; intra ring AG."""
    R = G * ng
    C = G * ng
    ops = []
    for r in range(R):
        for i in range(G):
            ops.append((COPY, r, IN, i * ng, r, OUT, i * ng, ng))
    for s in range(G - 1):                      # intra-group reduce-scatter
        for g in range(ng):
            for i in range(G):
                src, dst = g * G + (i + 1 + s) % G, g * G + (i + 2 + s) % G
                ops.append((REDUCE, src, OUT, i * ng, dst, OUT, i * ng, ng))
    for s in range(ng - 1):                     # inter-group ring RS per slice
        for i in range(G):
            for k in range(ng):
                src, dst = ((k + 1 + s) % ng) * G + i, ((k + 2 + s) % ng) * G + i
                ops.append((REDUCE, src, OUT, i * ng + k, dst, OUT, i * ng + k, 1))
    for s in range(ng - 1):                     # inter-group ring AG per slice
        for i in range(G):
            for k in range(ng):
                src, dst = ((k + s) % ng) * G + i, ((k + s + 1) % ng) * G + i
                ops.append((COPY, src, OUT, i * ng + k, dst, OUT, i * ng + k, 1))
    for s in range(G - 1):                      # intra-group all-gather
        for g in range(ng):
            for i in range(G):
                src, dst = g * G + (i + s) % G, g * G + (i + s + 1) % G
                ops.append((COPY, src, OUT, i * ng, dst, OUT, i * ng, ng))
    return _arr(ops), (C, C, 0)


def alltoall_two_phase(G: int, ng: int):
    """out[d] block s = in[s] block d, R = G*ng, one chunk per block.

    Phase 1: a block for another group h goes to aggregator p = g*G + d%G
    (same group g as the source), scratch slot h'*G + s%G with
    h' = (h - g - 1) mod ng; blocks for the own group go straight to out.
    Phase 2: p sends its G slots for group h as one batch to h*G + p%G."""
    R = G * ng
    ops = []
    for s in range(R):
        g = s // G
        for d in range(R):
            h = d // G
            if h == g:
                ops.append((COPY, s, IN, d, d, OUT, s, 1))
            else:
                p = g * G + d % G
                hp = (h - g - 1) % ng
                ops.append((COPY, s, IN, d, p, SCR, hp * G + s % G, 1))
    for p in range(R):
        g, l = p // G, p % G
        for h in range(ng):
            if h == g:
                continue
            hp = (h - g - 1) % ng
            ops.append((COPY, p, SCR, hp * G, h * G + l, OUT, g * G, G))
    return _arr(ops), (R, R, (ng - 1) * G)


def alltonext(G: int, ng: int, wrap: bool = False):
    """out[r+1] = in[r]; buffers have G chunks (parts).  A pair that leaves
    group g for group h is split into G parts; part j goes
    r -> g*G+j -> h*G+j -> r+1 (repeated ranks dropped).  The first relay
    stages part j in scratch chunk 0, the second in scratch chunk 1."""
    R = G * ng
    ops = []
    last = R if wrap else R - 1
    for r in range(last):
        dst = (r + 1) % R
        g, h = r // G, dst // G
        if g == h:
            ops.append((COPY, r, IN, 0, dst, OUT, 0, G))
            continue
        for j in range(G):
            # a relay equal to the source (j = G-1) or to the destination
            # (j = 0) is skipped; the two relays are in different groups
            stops = [(r, IN, j)]
            if g * G + j != r:
                stops.append((g * G + j, SCR, 0))
            if h * G + j != dst:
                stops.append((h * G + j, SCR, 1))
            stops.append((dst, OUT, j))
            for a, b in zip(stops[:-1], stops[1:]):
                ops.append((COPY, a[0], a[1], a[2], b[0], b[1], b[2], 1))
    return _arr(ops), (G, G, 2)


def alltoallv(counts):
    """``counts[s][d]`` chunks from rank s to rank d.  Input of s: blocks for
    d = 0, 1, ... back to back; output of d: blocks from s = 0, 1, ... back
    to back; buffers as long as the longest rank's."""
    c = np.asarray(counts, dtype=np.int64)
    R = c.shape[0]
    ops = []
    # source-major program order (any order gives the same result: every
    # pair writes its own output range and reads only inputs)
    for s in range(R):
        for d in range(R):
            if c[s, d] == 0:
                continue
            src_off = int(c[s, :d].sum())
            dst_off = int(c[:s, d].sum())
            ops.append((COPY, s, IN, src_off, d, OUT, dst_off, int(c[s, d])))
    nin = int(c.sum(axis=1).max())
    nout = int(c.sum(axis=0).max())
    return _arr(ops), (nin, nout, 0)


def hier_allgather(G: int, ng: int):
    """out[r] = in[0] ++ in[1] ++ ... ++ in[R-1] over R = G * ng ranks, one
    chunk per rank in, R chunks out (block s at chunk s)."""
    R = G * ng
    ops = []
    rank = lambda g, i: g * G + i   # noqa: E731
    # (1) in-group ring AllGather of the group's own blocks
    for g in range(ng):
        for i in range(G):
            b = rank(g, i)
            ops.append((COPY, b, IN, 0, b, OUT, b, 1))
            for k in range(G - 1):
                ops.append((COPY, rank(g, (i + k) % G), OUT, b, rank(g, (i + k + 1) % G), OUT, b, 1))
    # (2) cross-group: same local index, every other group, from the input
    for g in range(ng):
        for i in range(G):
            b = rank(g, i)
            for h in range(ng):
                if h != g:
                    ops.append((COPY, b, IN, 0, rank(h, i), OUT, b, 1))
    # (3) in group h, the block of (g, i) circulates from rank (h, i)
    for h in range(ng):
        for g in range(ng):
            if g == h:
                continue
            for i in range(G):
                b = rank(g, i)
                for k in range(G - 1):
                    ops.append((COPY, rank(h, (i + k) % G), OUT, b, rank(h, (i + k + 1) % G), OUT, b, 1))
    return _arr(ops), (1, R, 0)


BUILTINS = {
    "ring_allreduce": ring_allreduce,
    "ring_allgather": ring_allgather,
    "ring_reducescatter": ring_reducescatter,
    "hier_allreduce": hier_allreduce,
    "alltoall_two_phase": alltoall_two_phase,
    "alltonext": alltonext,
    "hier_allgather": hier_allgather,
}
