"""Brute force over every interleaving of tiny programs (oracle explorer)."""
import pytest

from oracle import explore as E
from oracle import schedules as S

CASES = [
    ("ring_allreduce", (2,)), ("ring_allreduce", (3,)), ("ring_allreduce", (4,)),
    ("ring_allgather", (3,)), ("ring_allgather", (4,)),
    ("ring_reducescatter", (3,)), ("ring_reducescatter", (4,)),
    ("hier_allreduce", (2, 2)),
    ("alltoall_two_phase", (2, 2)),
    ("alltonext", (2, 2)), ("alltonext", (2, 2, True)), ("alltonext", (4, 1)),
]


@pytest.mark.parametrize("name,args", CASES)
@pytest.mark.parametrize("K", [1, 2])
def test_every_interleaving_gives_one_result_and_never_sticks(name, args, K):
    ops, ch = S.BUILTINS[name](*args)
    R = max(int(ops[:, 1].max()), int(ops[:, 4].max())) + 1
    res = E.explore(ops, R, ch, K=K)
    assert res["deadlocks"] == 0
    assert len(res["outputs"]) == 1


def _leaves(it, i, acc):
    e = it.exprs[i]
    if e[0] == "+":
        _leaves(it, e[1], acc)
        _leaves(it, e[2], acc)
    else:
        acc.append(e)
    return acc


@pytest.mark.parametrize("R", [2, 3, 4])
def test_allreduce_adds_each_rank_exactly_once(R):
    """Every output chunk is a sum with exactly one leaf per rank, of that
    chunk (reduced R-1 times)."""
    ops, ch = S.ring_allreduce(R)
    res = E.explore(ops, R, ch, K=1)
    (out,) = res["outputs"]
    it = res["interner"]
    for r in range(R):
        for c in range(R):
            leaves = sorted(_leaves(it, out[r][c], []))
            assert leaves == sorted(("x", k, c) for k in range(R))


def test_hier_allreduce_adds_each_rank_exactly_once():
    ops, ch = S.hier_allreduce(2, 2)
    res = E.explore(ops, 4, ch, K=1)
    (out,) = res["outputs"]
    it = res["interner"]
    for r in range(4):
        for c in range(ch[1]):
            assert sorted(_leaves(it, out[r][c], [])) == sorted(("x", k, c) for k in range(4))


def test_planted_deadlock_is_found():
    """Two ranks that each receive before sending wait for each other."""
    ops = [(0, 0, 0, 0, 1, 1, 0, 1), (0, 1, 0, 0, 0, 1, 0, 1)]
    progs = [[("recv", 1), ("send", 0)], [("recv", 0), ("send", 1)]]
    res = E.explore(ops, 2, (1, 1, 0), K=1, progs=progs)
    assert res["deadlocks"] > 0 and not res["outputs"]


def test_planted_capacity_deadlock_is_found():
    """Rank 0 sends two messages before reading the reply; rank 1 replies
    before reading the second message.  With one slot per link this sticks,
    with two it completes."""
    ops = [(0, 0, 0, 0, 1, 1, 0, 1), (0, 0, 0, 1, 1, 1, 1, 1), (0, 1, 0, 0, 0, 1, 0, 1),
           (0, 1, 0, 1, 0, 1, 1, 1)]
    progs = [[("send", 0), ("send", 1), ("recv", 2), ("recv", 3)],
             [("send", 2), ("send", 3), ("recv", 0), ("recv", 1)]]
    assert E.explore(ops, 2, (2, 2, 0), K=1, progs=progs)["deadlocks"] > 0
    res = E.explore(ops, 2, (2, 2, 0), K=2, progs=progs)
    assert res["deadlocks"] == 0 and len(res["outputs"]) == 1
