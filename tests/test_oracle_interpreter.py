"""Pins of the oracle interpreter and the oracle's schedule generators.

Independent references used here (none of them calls the oracle's rounding):
* closed-form collective definitions written with numpy indexing
  (AllGather = concatenation, AllToAll = block transpose, AllToNext = shift);
* exact integer sums (int32 / int64) for AllReduce and ReduceScatter;
* a fixed-order fold written separately below with library rounding
  (numpy float32 / float16 arithmetic, torch bf16 arithmetic);
* the float64 sum with the recursive-summation error bound;
* hand-worked fixtures in ``tests/golden``.
"""
import json
import os

import numpy as np
import pytest
import torch

import datagen
import oracle
from oracle import schedules as S

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
F32, BF16, F16, I32 = oracle.F32, oracle.BF16, oracle.F16, oracle.I32


# --------------------------------------------------------------------------
# library-rounded fixed-order folds (independent of the oracle's C code)

def lib_add(a, b, dtype):
    if dtype == F32:
        return (a.astype(np.float32) + b.astype(np.float32)).astype(np.float32)
    if dtype == F16:
        return (a.view(np.float16) + b.view(np.float16)).view(np.uint16)
    if dtype == BF16:
        ta = torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16)
        tb = torch.from_numpy(b.view(np.int16).copy()).view(torch.bfloat16)
        return (ta + tb).view(torch.int16).numpy().view(np.uint16)
    if dtype == I32:
        return (a.astype(np.int64) + b.astype(np.int64)).astype(np.int32)
    raise ValueError(dtype)


def fold(vals, order, dtype):
    acc = vals[order[0]].copy()
    for k in order[1:]:
        acc = lib_add(acc, vals[k], dtype)
    return acc


def ring_allreduce_closed(ins, R, dtype):
    """Chunk c: left fold over ranks c+1, c+2, ..., c (mod R)."""
    n = ins[0].size // R
    res = np.empty_like(ins[0])
    for c in range(R):
        order = [(c + 1 + k) % R for k in range(R)]
        res[c * n:(c + 1) * n] = fold([x[c * n:(c + 1) * n] for x in ins], order, dtype)
    return res


def hier_closed(ins, G, ng, dtype):
    """Slice i sub k: intra-group fold over local ranks i+1, ..., i, then
    inter-group fold over groups k+1, ..., k."""
    C = G * ng
    n = ins[0].size // C
    res = np.empty_like(ins[0])
    for i in range(G):
        for k in range(ng):
            c = i * ng + k
            chunk = [x[c * n:(c + 1) * n] for x in ins]
            partial = []
            for g in range(ng):
                order = [g * G + (i + 1 + t) % G for t in range(G)]
                partial.append(fold(chunk, order, dtype))
            res[c * n:(c + 1) * n] = fold(partial, [(k + 1 + t) % ng for t in range(ng)], dtype)
    return res


# --------------------------------------------------------------------------

@pytest.mark.parametrize("R", [1, 2, 3, 5, 8])
@pytest.mark.parametrize("dtype", [F32, BF16, F16, I32])
def test_allgather_is_concatenation(R, dtype):
    ops, ch = S.ring_allgather(R)
    n = 37
    ins = datagen.rank_inputs(1, "int" if dtype == I32 else "normal", R, n, dtype)
    outs, _, _ = oracle.run(ops, R, ch, n, dtype, ins)
    want = np.concatenate(ins)
    for r in range(R):
        assert np.array_equal(outs[r].view(np.uint8), want.view(np.uint8))


@pytest.mark.parametrize("G,ng", [(1, 1), (2, 2), (4, 2), (8, 4), (3, 3)])
@pytest.mark.parametrize("dtype", [F16, I32])
def test_alltoall_is_block_transpose(G, ng, dtype):
    R = G * ng
    ops, ch = S.alltoall_two_phase(G, ng)
    B = 5
    ins = datagen.rank_inputs(3, "int" if dtype == I32 else "uniform", R, R * B, dtype)
    outs, _, _ = oracle.run(ops, R, ch, B, dtype, ins)
    for d in range(R):
        for s in range(R):
            assert np.array_equal(outs[d][s * B:(s + 1) * B], ins[s][d * B:(d + 1) * B])


@pytest.mark.parametrize("G,ng,wrap", [(1, 1, False), (8, 3, False), (4, 2, True), (3, 4, False),
                                       (2, 1, True)])
def test_alltonext_is_shift(G, ng, wrap):
    R = G * ng
    ops, ch = S.alltonext(G, ng, wrap)
    n = 6
    ins = datagen.rank_inputs(4, "normal", R, G * n, F32)
    outs, _, _ = oracle.run(ops, R, ch, n, F32, ins, sentinel=0xA5)
    for r in range(R):
        src = r - 1
        if src < 0:
            if wrap:
                src = R - 1
            else:
                # rank 0 receives nothing: output keeps the sentinel
                assert np.all(outs[0].view(np.uint8) == 0xA5)
                continue
        assert np.array_equal(outs[r], ins[src])


@pytest.mark.parametrize("R", [1, 2, 3, 8])
def test_int32_allreduce_and_reducescatter_exact(R):
    n = 16
    ins = datagen.rank_inputs(0, "int", R, R * n, I32)
    total = np.sum(np.stack(ins).astype(np.int64), axis=0)
    ops, ch = S.ring_allreduce(R)
    outs, _, _ = oracle.run(ops, R, ch, n, I32, ins)
    for r in range(R):
        assert np.array_equal(outs[r].astype(np.int64), total)
    ops, ch = S.ring_reducescatter(R)
    outs, _, _ = oracle.run(ops, R, ch, n, I32, ins)
    for r in range(R):
        assert np.array_equal(outs[r].astype(np.int64), total[r * n:(r + 1) * n])


@pytest.mark.parametrize("G,ng", [(2, 2), (8, 2), (4, 3), (1, 4), (4, 1)])
def test_int32_hier_allreduce_exact(G, ng):
    R = G * ng
    n = 3
    ins = datagen.rank_inputs(2, "int", R, G * ng * n, I32)
    total = np.sum(np.stack(ins).astype(np.int64), axis=0)
    ops, ch = S.hier_allreduce(G, ng)
    outs, _, _ = oracle.run(ops, R, ch, n, I32, ins)
    for r in range(R):
        assert np.array_equal(outs[r].astype(np.int64), total)


@pytest.mark.parametrize("R", [2, 3, 5, 8])
@pytest.mark.parametrize("dtype", [F32, BF16, F16])
def test_ring_allreduce_equals_fixed_order_fold(R, dtype):
    n = 64
    ins = datagen.rank_inputs(0, "normal", R, R * n, dtype)
    ops, ch = S.ring_allreduce(R)
    outs, _, _ = oracle.run(ops, R, ch, n, dtype, ins)
    want = ring_allreduce_closed(ins, R, dtype)
    for r in range(R):
        assert np.array_equal(outs[r].view(np.uint8), want.view(np.uint8))


@pytest.mark.parametrize("R", [2, 4, 8])
@pytest.mark.parametrize("dtype", [F32, BF16])
def test_ring_reducescatter_equals_fold_slice(R, dtype):
    n = 33
    ins = datagen.rank_inputs(1, "normal", R, R * n, dtype)
    ops, ch = S.ring_reducescatter(R)
    outs, _, _ = oracle.run(ops, R, ch, n, dtype, ins)
    want = ring_allreduce_closed(ins, R, dtype)
    for r in range(R):
        assert np.array_equal(outs[r].view(np.uint8), want[r * n:(r + 1) * n].view(np.uint8))


@pytest.mark.parametrize("G,ng", [(2, 2), (4, 2), (8, 2), (3, 3)])
@pytest.mark.parametrize("dtype", [F32, BF16, F16])
def test_hier_allreduce_equals_grouped_fold(G, ng, dtype):
    R = G * ng
    n = 8
    ins = datagen.rank_inputs(2, "normal", R, G * ng * n, dtype)
    ops, ch = S.hier_allreduce(G, ng)
    outs, _, _ = oracle.run(ops, R, ch, n, dtype, ins)
    want = hier_closed(ins, G, ng, dtype)
    for r in range(R):
        assert np.array_equal(outs[r].view(np.uint8), want.view(np.uint8))


def _gamma(h, u):
    return h * u / (1 - h * u)


@pytest.mark.parametrize("dtype,u,rel", [(F32, 2.0 ** -24, 1e-5), (BF16, 2.0 ** -8, 1e-2),
                                         (F16, 2.0 ** -11, 1e-2)])
def test_allreduce_within_float64_bounds(dtype, u, rel):
    R, n = 8, 4096
    ins = datagen.rank_inputs(0, "uniform", R, R * n, dtype)
    ops, ch = S.ring_allreduce(R)
    outs, _, _ = oracle.run(ops, R, ch, n, dtype, ins)
    x64 = np.stack([datagen.to_f64(a, dtype) for a in ins])
    y64 = x64.sum(axis=0)
    y = datagen.to_f64(outs[0], dtype)
    assert np.linalg.norm(y - y64) / np.linalg.norm(y64) <= rel
    # elementwise recursive-summation bound: R-1 rounded additions
    bound = _gamma(R - 1, u) * np.abs(x64).sum(axis=0)
    assert np.all(np.abs(y - y64) <= bound + 1e-300)


@pytest.mark.parametrize("dtype", [BF16, F16, F32])
def test_small_integers_exact_in_every_order(dtype):
    """Small integers sum exactly in any order, so the float path must equal
    the integer closed form."""
    R, n = 8, 128
    ins = datagen.rank_inputs(9, "smallint", R, R * n, dtype)
    total = np.stack([datagen.to_f64(a, dtype) for a in ins]).sum(axis=0)
    for gen, args in [(S.ring_allreduce, (R,)), (S.hier_allreduce, (4, 2))]:
        ops, ch = gen(*args)
        outs, _, _ = oracle.run(ops, R, ch, n, dtype, ins)
        for r in range(R):
            assert np.array_equal(datagen.to_f64(outs[r], dtype), total)


def test_trivial_rank_counts():
    x = datagen.rank_inputs(5, "normal", 1, 40, BF16)
    for gen in (S.ring_allreduce, S.ring_allgather, S.ring_reducescatter):
        ops, ch = gen(1)
        outs, _, _ = oracle.run(ops, 1, ch, 40 // ch[0], BF16, x)
        assert np.array_equal(outs[0], x[0])
    # R = 2: one rounding, equal to the torch bf16 sum
    ins = datagen.rank_inputs(5, "normal", 2, 64, BF16)
    ops, ch = S.ring_allreduce(2)
    outs, _, _ = oracle.run(ops, 2, ch, 32, BF16, ins)
    t = [torch.from_numpy(a.view(np.int16)).view(torch.bfloat16) for a in ins]
    want = (t[0] + t[1]).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(outs[0], want) and np.array_equal(outs[1], want)


def test_golden_ring_order():
    g = json.load(open(os.path.join(GOLDEN, "ring_allreduce_bf16_order.json")))
    R = g["R"]
    ins = [np.asarray(v, np.uint16) for v in g["inputs_bf16_bits"]]
    ops, ch = S.ring_allreduce(R)
    outs, _, _ = oracle.run(ops, R, ch, 1, BF16, ins)
    for r in range(R):
        assert outs[r].tolist() == g["expected_out_bf16_bits"][r]
    ops, ch = S.ring_reducescatter(R)
    outs, _, _ = oracle.run(ops, R, ch, 1, BF16, ins)
    for r in range(R):
        assert outs[r].tolist() == [g["expected_out_bf16_bits"][r][r]]


def test_golden_hier_grouping():
    g = json.load(open(os.path.join(GOLDEN, "hier_allreduce_bf16_grouping.json")))
    G, ng, ce = g["G"], g["ng"], g["chunk_elems"]
    R = G * ng
    ins = [np.full(G * ng * ce, v, np.uint16) for v in g["rank_value_bf16_bits"]]
    ops, ch = S.hier_allreduce(G, ng)
    outs, _, _ = oracle.run(ops, R, ch, ce, BF16, ins)
    for r in range(R):
        assert np.all(outs[r] == g["expected_value_bf16_bits"])


def test_golden_alltoall_labels():
    g = json.load(open(os.path.join(GOLDEN, "alltoall_two_phase_blocks.json")))
    G, ng = g["G"], g["ng"]
    R = G * ng
    ins = [np.asarray(v, np.int32) for v in g["inputs_i32"]]
    ops, ch = S.alltoall_two_phase(G, ng)
    outs, _, _ = oracle.run(ops, R, ch, 1, I32, ins)
    for r in range(R):
        assert outs[r].tolist() == g["expected_out_i32"][r]


def test_sampled_run_equals_full_columns():
    R, n = 8, 100
    ins = datagen.rank_inputs(0, "normal", R, R * n, BF16)
    ops, ch = S.ring_allreduce(R)
    full, _, _ = oracle.run(ops, R, ch, n, BF16, ins)
    offs = np.array([0, 3, 17, 99])
    samp = oracle.run_sampled(ops, R, ch, n, BF16, ins, offs)
    for r in range(R):
        assert np.array_equal(samp[r], full[r].reshape(R, n)[:, offs])


def test_interpreter_rejects_bad_ops():
    ins = [np.zeros(4, np.float32)]
    with pytest.raises(oracle.OracleError):   # overlapping source and destination
        oracle.run(np.array([[0, 0, 1, 0, 0, 1, 1, 2]]), 1, (4, 4, 0), 1, F32, ins)
    with pytest.raises(oracle.OracleError):   # out of range
        oracle.run(np.array([[0, 0, 0, 3, 0, 1, 0, 2]]), 1, (4, 4, 0), 1, F32, ins)
    with pytest.raises(oracle.OracleError):   # bad rank
        oracle.run(np.array([[0, 1, 0, 0, 0, 1, 0, 1]]), 1, (4, 4, 0), 1, F32, ins)
    with pytest.raises(oracle.OracleError):   # bad opcode
        oracle.run(np.array([[7, 0, 0, 0, 0, 1, 0, 1]]), 1, (4, 4, 0), 1, F32, ins)


def test_planted_order_mistake_is_caught_by_the_fold():
    """A reversed ring (chunk c folded from rank c-1 downwards) must not equal
    the closed form: guards the fold itself against being order-blind."""
    R, n = 5, 64
    ins = datagen.rank_inputs(0, "normal", R, R * n, BF16)
    ops, ch = S.ring_allreduce(R)
    ops = ops.copy()
    # rewrite the reduce-scatter hops to run the other way round
    rs = ops[:, 0] == 1
    ops[rs, 1] = (R - ops[rs, 1]) % R
    ops[rs, 4] = (R - ops[rs, 4]) % R
    outs, _, _ = oracle.run(ops, R, ch, n, BF16, ins)
    want = ring_allreduce_closed(ins, R, BF16)
    assert not np.array_equal(outs[0], want)
