"""Pins of the oracle's rounding primitives against library routines and exact
arithmetic.

The oracle's reading: a reduce of two bf16 (f16) values widens both to
binary32, adds, and rounds the binary32 sum to bf16 (f16) to nearest even.
These tests check (a) the conversions against numpy / torch, over a cover of
every rounding decision, and (b) the composed add against the correctly
rounded sum (exact rational arithmetic on samples, and exact float64 sums for
f16 over a quarter-billion pairs).
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle


def _torch_bf16(x32):
    return torch.from_numpy(np.ascontiguousarray(x32, np.float32)).to(torch.bfloat16) \
        .view(torch.int16).numpy().view(np.uint16)


def _bf16_cover():
    """Every upper half (sign, exponent, 7 kept bits) combined with the lower
    halves that decide round-to-nearest-even: 0, 1, just below / at / just
    above half, the maximum, and a few random ones."""
    rng = np.random.default_rng(12345)
    upper = np.arange(1 << 16, dtype=np.uint32) << 16
    lows = [0, 1, 0x7FFF, 0x8000, 0x8001, 0xFFFF] + list(rng.integers(0, 1 << 16, 10))
    u = (upper[:, None] | np.asarray(lows, np.uint32)[None, :]).reshape(-1)
    return u.view(np.float32)


def test_f32_to_bf16_matches_torch_on_full_cover():
    x = _bf16_cover()
    ours = oracle.f32_to_bf16(x)
    ref = _torch_bf16(x)
    nan = np.isnan(x)
    assert np.array_equal(ours[~nan], ref[~nan])
    # NaN stays NaN (payload is not pinned)
    assert np.all((ours[nan] & 0x7F80) == 0x7F80) and np.all((ours[nan] & 0x7F) != 0)


def _f16_cover():
    """For every binary32 exponent and sign: all kept-bit patterns that a
    binary16 result can hold at that exponent, times the dropped-bit patterns
    0, 1, half-1, half, half+1, all-ones and random ones."""
    rng = np.random.default_rng(777)
    vals = []
    for e in range(256):
        E = e - 127
        shift = 13 if E >= -14 else 13 + (-14 - E)
        shift = min(shift, 24)
        kept_bits = 23 - shift if shift <= 23 else 0
        kept = np.arange(1 << max(kept_bits, 0), dtype=np.uint32) << shift if shift <= 23 \
            else np.zeros(1, np.uint32)
        half = 1 << (shift - 1)
        lows = {0, 1, half - 1, half, half + 1, (1 << shift) - 1}
        lows |= set(int(v) for v in rng.integers(0, 1 << shift, 4))
        lows = np.asarray(sorted(v & 0x7FFFFF for v in lows), np.uint32)
        m = (kept[:, None] | lows[None, :]).reshape(-1) & 0x7FFFFF
        for s in (0, 1):
            vals.append((np.uint32(s << 31) | np.uint32(e << 23) | m).astype(np.uint32))
    return np.concatenate(vals).view(np.float32)


def test_f32_to_f16_matches_numpy_on_full_cover():
    x = _f16_cover()
    assert x.size > 1_000_000
    ours = oracle.f32_to_f16(x)
    with np.errstate(over="ignore", invalid="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    nan = np.isnan(x)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.all((ours[nan] & 0x7C00) == 0x7C00) and np.all((ours[nan] & 0x3FF) != 0)


def test_f16_to_f32_exhaustive():
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ours = oracle.f16_to_f32(h)
    ref = h.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(ours[~nan].view(np.uint32), ref[~nan].view(np.uint32))
    assert np.all(np.isnan(ours[nan]))


def test_bf16_to_f32_is_exact_widening():
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    w = oracle.bf16_to_f32(h)
    t = torch.from_numpy(h.view(np.int16)).view(torch.bfloat16).float().numpy()
    nan = np.isnan(t)
    assert np.array_equal(w[~nan].view(np.uint32), t[~nan].view(np.uint32))


def _finite_bf16(n=None):
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    return h[(h & 0x7F80) != 0x7F80]


def test_bf16_add_matches_torch_on_pair_sweep():
    """All finite b against a stride-7 sample of a (~9400 values): 600M pairs
    would be slow, this is ~1/7 of the 2^32 pairs and covers every exponent
    combination."""
    b_all = _finite_bf16()
    a_sample = b_all[::7]
    tb = torch.from_numpy(b_all.view(np.int16)).view(torch.bfloat16)
    rows = 256
    for i in range(0, a_sample.size, rows):
        a = np.repeat(a_sample[i:i + rows], b_all.size)
        b = np.tile(b_all, min(rows, a_sample.size - i))
        ours = oracle.add_bf16(a, b)
        ta = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
        ref = (ta + torch.from_numpy(b.view(np.int16)).view(torch.bfloat16)) \
            .view(torch.int16).numpy().view(np.uint16)
        fin = (ref & 0x7F80) != 0x7F80
        assert np.array_equal(ours[fin], ref[fin])
        # overflow cases: both infinite with the same sign
        assert np.array_equal(ours[~fin & ((ref & 0x7F) == 0)], ref[~fin & ((ref & 0x7F) == 0)])
    del tb


def _exact_round(q: Fraction, pbits: int, emin: int, emax: int) -> Fraction:
    """Correctly rounded (nearest, ties to even) value of rational q in a
    binary format with pbits significant bits, minimum normal exponent emin
    and maximum exponent emax; returns None for overflow."""
    if q == 0:
        return Fraction(0)
    sign = -1 if q < 0 else 1
    a = abs(q)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    e = max(e, emin)
    ulp = Fraction(2) ** (e - pbits + 1)
    k = a / ulp
    fl = k.numerator // k.denominator
    rem = k - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    r = fl * ulp
    if r >= Fraction(2) ** (emax + 1):
        return None
    return sign * r


def _bf16_val(h):
    return Fraction(float(oracle.bf16_to_f32(np.array([h], np.uint16))[0]))


def test_bf16_add_is_correctly_rounded_exact_rationals():
    rng = np.random.default_rng(2024)
    fin = _finite_bf16()
    a = rng.choice(fin, 6000)
    b = rng.choice(fin, 6000)
    # ties on purpose: b = a * 2^-8 style pairs (half-ulp addends)
    a2 = rng.choice(fin[(fin & 0x7F80) > 0x0400], 2000)
    b2 = ((a2 & 0x8000) | np.clip(((a2 & 0x7F80).astype(np.int32) - (8 << 7)), 0x80, 0x7F00)).astype(np.uint16)
    a = np.concatenate([a, a2])
    b = np.concatenate([b, b2])
    ours = oracle.add_bf16(a, b)
    for x, y, z in zip(a, b, ours):
        exact = _bf16_val(int(x)) + _bf16_val(int(y))
        want = _exact_round(exact, 8, -126, 127)
        if want is None:
            assert (z & 0x7FFF) == 0x7F80
            continue
        got = _bf16_val(int(z))
        assert got == want, (hex(x), hex(y), hex(z))


def test_f16_add_is_correctly_rounded_pair_sweep():
    """float64 holds every sum of two binary16 values exactly (their bits span
    at most 40 positions), and numpy rounds float64 to float16 directly, so
    ``(a64 + b64).astype(float16)`` is the correctly rounded sum."""
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    fin = h[(h & 0x7C00) != 0x7C00]
    a_sample = fin[::13]
    b64 = fin.view(np.float16).astype(np.float64)
    rows = 256
    for i in range(0, a_sample.size, rows):
        aa = a_sample[i:i + rows]
        a = np.repeat(aa, fin.size)
        b = np.tile(fin, aa.size)
        ours = oracle.add_f16(a, b)
        with np.errstate(over="ignore"):
            ref = (np.repeat(aa.view(np.float16).astype(np.float64), fin.size)
                   + np.tile(b64, aa.size)).astype(np.float16).view(np.uint16)
        # -0 vs +0: x + (-x) is +0 under round-to-nearest in both
        assert np.array_equal(ours, ref)


def test_i32_add_wraps():
    lib = oracle.lib()
    lib.oracle_add_i32.restype = __import__("ctypes").c_int32
    assert lib.oracle_add_i32(2**31 - 1, 1) == -2**31
    assert lib.oracle_add_i32(-5, 3) == -2


def _special_values(dtype):
    """Zeros, ones, the largest finite value, the smallest subnormal, both
    infinities and NaNs of either sign and two payloads, as storage bits."""
    if dtype == "f32":
        b = [0x00000000, 0x80000000, 0x3F800000, 0xBF800000, 0x7F7FFFFF, 0xFF7FFFFF, 0x00000001, 0x80000001,
             0x7F800000, 0xFF800000, 0x7FC00000, 0xFFC00000, 0x7F800001, 0x7FBFFFFF]
        return np.array(b, np.uint32)
    if dtype == "bf16":
        b = [0x0000, 0x8000, 0x3F80, 0xBF80, 0x7F7F, 0xFF7F, 0x0001, 0x8001, 0x7F80, 0xFF80, 0x7FC0, 0xFFC0,
             0x7F81, 0x7FBF]
    else:
        b = [0x0000, 0x8000, 0x3C00, 0xBC00, 0x7BFF, 0xFBFF, 0x0001, 0x8001, 0x7C00, 0xFC00, 0x7E00, 0xFE00,
             0x7C01, 0x7DFF]
    return np.array(b, np.uint16)


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_special_values_follow_ieee_through_a_reduction(dtype):
    """Reading for special values: IEEE 754 addition in the buffer type (for
    bf16 / f16: widened to f32, added, rounded to nearest even): a NaN
    operand gives NaN, an infinity plus a finite value keeps the infinity,
    opposite infinities give NaN, a sum past the largest finite value rounds
    to infinity.  A NaN's payload and sign are not pinned.  Every pair of
    special values goes through the oracle's interpreter (a reduce of rank
    1's input into rank 0's copy of its own) and is checked against numpy
    (f32, and f16 through an exact float64 sum) or torch (bf16)."""
    code = {"f32": 0, "bf16": 1, "f16": 2}[dtype]
    v = _special_values(dtype)
    a = np.repeat(v, v.size)
    b = np.tile(v, v.size)
    n = a.size
    # out[0] = in[0] + in[1], element by element
    ops = np.array([(0, 0, 0, 0, 0, 1, 0, 1), (1, 1, 0, 0, 0, 1, 0, 1)], np.int32)
    ins = [a.view(np.float32), b.view(np.float32)] if dtype == "f32" else [a, b]
    outs, _, _ = oracle.run(ops, 2, (1, 1, 0), n, code, ins)
    got = np.asarray(outs[0])
    got = got.view(np.uint32) if dtype == "f32" else got.view(np.uint16)
    if dtype == "f32":
        with np.errstate(over="ignore", invalid="ignore"):
            ref = (a.view(np.float32) + b.view(np.float32)).view(np.uint32)
        nan_ref = np.isnan(ref.view(np.float32))
        nan_got = np.isnan(got.view(np.float32))
    elif dtype == "bf16":
        ta = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
        tb = torch.from_numpy(b.view(np.int16)).view(torch.bfloat16)
        ref = (ta + tb).view(torch.int16).numpy().view(np.uint16)
        nan_ref = ((ref & 0x7F80) == 0x7F80) & ((ref & 0x7F) != 0)
        nan_got = ((got & 0x7F80) == 0x7F80) & ((got & 0x7F) != 0)
    else:
        with np.errstate(over="ignore", invalid="ignore"):
            ref = (a.view(np.float16).astype(np.float64) + b.view(np.float16).astype(np.float64)) \
                .astype(np.float16).view(np.uint16)
        nan_ref = np.isnan(ref.view(np.float16))
        nan_got = np.isnan(got.view(np.float16))
    assert np.array_equal(nan_got, nan_ref)
    assert nan_ref.any() and (~nan_ref).any()
    assert np.array_equal(got[~nan_ref], ref[~nan_ref])
